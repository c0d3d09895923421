// Causal multi-query attention on the 5th-generation tensor cores (bf16,
// head dim 128): forward, and the backward as a Q-major dQ pass plus a
// KV-major dK/dV pass (launch article, architecture list: multi-query
// attention -- the H query heads share one K/V head; causal for next-token
// prediction).
//
// Query rows of one sequence are packed as r = t * H + head, so a tile of
// packed rows meets a single K/V tile and every K/V byte brought on chip
// serves all H heads; key j is visible to packed row r iff j <= r / H.
//
// Every kernel is warp-specialised: warp 0 issues TMA, two single threads
// issue tcgen05.mma (one for the score products, one for the products that
// consume the softmax warps' output: an MMA issue holds its thread for about
// the MMA's run time, so a lone issuer's waits and commits would idle the
// tensor pipe), warp 2 owns the TMEM allocation, and the warps from 4 on are
// softmax warpgroups -- a thread owns one TMEM lane, i.e. one row of the
// score tile, and a slice of its columns (the slices of a row belong to the
// threads of the same lane in the other warpgroups): two warpgroups of 64
// columns in the backward passes (384 threads), four of 32 in the forward
// (640 threads, four warps per scheduler).  Row reductions need no shuffles.
// The probability-like operands (P in the forward, P^T and dS^T in the dK/dV
// pass, dS in the dQ pass) go from registers to tensor memory as bf16 pairs
// and feed the next MMA as its A operand; the streamed Q, K, V, dO tiles stay
// in 128B-swizzled shared memory as TMA delivers them.  A 64-wide [row][64
// dims] swizzled tile is both a K-major operand (rows = N) and an MN-major one
// (rows = K), so no operand is ever transposed.  All mbarrier waits are
// bounded; on timeout the CTA records DEV_TIMEOUT, stops, drains in-flight
// copies and MMAs, and frees TMEM.
#include <algorithm>

#include "nc_common.cuh"
#include "nc_internal.h"
#include "tc_common.cuh"

namespace nc {
namespace {

using namespace tc;

constexpr int HD = 128;
constexpr int NT = 384;  // backward passes: 4 control warps + 2 softmax warpgroups
constexpr int NSW = 8;   // their softmax warps (4..11); warp w reads TMEM lanes 32 (w % 4) ..
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int SITE_ATTN = 300;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// (x - d) * p on both halves of a packed fp32 pair: one instruction each for
// the subtract and the multiply instead of two.
__device__ __forceinline__ void sub_mul2(float& r0, float& r1, float x0, float x1, float d0,
                                         float d1, float p0, float p1) {
  asm("{\n\t.reg .b64 x, d, p, r;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 d, {%4, %5};\n\tmov.b64 p, {%6, %7};\n\t"
      "sub.rn.f32x2 r, x, d;\n\tmul.rn.f32x2 r, r, p;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1), "f"(d0), "f"(d1), "f"(p0), "f"(p1));
}

// 2^x on the special-function unit (approximate, flushes denormals; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// D (+)= A B^T with the A operand (M rows = TMEM lanes, 16 K values packed
// two bf16 per 32-bit column) read from tensor memory at a_tmem.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Store 32 fp32 values as bf16 to global (64 contiguous bytes).
__device__ __forceinline__ void store_bf16_32(bf16* dst, const float (&v)[32], float scale) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 q;
    q.x = pack2(v[i * 8 + 0] * scale, v[i * 8 + 1] * scale);
    q.y = pack2(v[i * 8 + 2] * scale, v[i * 8 + 3] * scale);
    q.z = pack2(v[i * 8 + 4] * scale, v[i * 8 + 5] * scale);
    q.w = pack2(v[i * 8 + 6] * scale, v[i * 8 + 7] * scale);
    reinterpret_cast<uint4*>(dst)[i] = q;
  }
}

// 32 bf16 pairs of this thread's row into its TMEM lane (32 columns).
__device__ __forceinline__ void pairs_to_tmem(uint32_t taddr, const uint32_t (&p)[32]) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(p[j]);
  tmem_st_32cols(taddr, v);
}

struct CtaSync {
  volatile int* abort_flag;
  int* err;
  long long timeout_ns;
  __device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity) const {
    return mbar_wait_bounded(bar, parity, abort_flag, err, SITE_ATTN, timeout_ns);
  }
  // The same wait with one outcome for the whole warp (called by all 32
  // lanes): a warp that goes on to a warp-collective tcgen05.ld/st must not
  // split when some lanes give up at the limit and others do not.
  __device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) const {
    return __all_sync(0xffffffffu, wait(bar, parity));
  }
};

// ======================================================================
// forward: persistent CTAs, one per SM, each walking a list of query-tile
// pairs (tile 0: packed rows r0 .. r0 + 127, tile 1: the next 128) of every
// sequence, heaviest pairs first and the order reversed every other round so
// that the CTAs get similar shares of key tiles; per pair one stream of
// 128-key tiles serves both query tiles.  The rings and barrier phases carry
// on from one pair to the next, so the next pair's loads and first score
// products overlap the current pair's output epilogue.
// ======================================================================
namespace fwd {
constexpr int BQ = 128, BKV = 128;
constexpr int NTF = 352;                    // 3 control warps + one softmax warpgroup per tile
constexpr int ATOM = 16384;                 // [128 rows][64] bf16
constexpr int Q_OFF = 0;                    // 2 tiles x 32 KB
constexpr int K_OFF = 2 * 32768;            // 2 stages x 32 KB
constexpr int V_OFF = K_OFF + 2 * 32768;    // 2 stages x 32 KB
constexpr int BAR_OFF = V_OFF + 2 * 32768;
constexpr int SMEM = BAR_OFF + 256 + 1024;
static_assert(SMEM <= 232448, "forward shared memory exceeds 227 KB");
}  // namespace fwd

// fma on both halves of a packed fp32 pair.
__device__ __forceinline__ void fma2(float& r0, float& r1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n\t.reg .b64 a, b, c, r;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 r, a, b, c;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// a += b on both halves of a packed fp32 pair.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b;\n\t"
      "mov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, b;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// 64 bf16 pairs of this thread's row into its TMEM lane (64 columns), one
// wait for both halves.
__device__ __forceinline__ void pairs64_to_tmem(uint32_t taddr, const uint32_t (&p)[64]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t* q = p + 32 * h;
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr + 32 * h),
        "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3]), "r"(q[4]), "r"(q[5]), "r"(q[6]), "r"(q[7]),
        "r"(q[8]), "r"(q[9]), "r"(q[10]), "r"(q[11]), "r"(q[12]), "r"(q[13]), "r"(q[14]),
        "r"(q[15]), "r"(q[16]), "r"(q[17]), "r"(q[18]), "r"(q[19]), "r"(q[20]), "r"(q[21]),
        "r"(q[22]), "r"(q[23]), "r"(q[24]), "r"(q[25]), "r"(q[26]), "r"(q[27]), "r"(q[28]),
        "r"(q[29]), "r"(q[30]), "r"(q[31])
        : "memory");
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Work item k of CTA c among G persistent CTAs: round k takes items k G ..
// k G + G - 1, forwards in even rounds and backwards in odd ones.
__device__ __forceinline__ long snake_item(int c, int k, int G, long n_items) {
  const long u = (long)k * G + ((k & 1) ? G - 1 - c : c);
  return u < n_items ? u : -1;
}

// Tensor memory (512 columns): S of tile x at columns 128 x, O of tile x at
// 256 + 128 x.  P(j) of a tile, bf16 pairs, overwrites the first 64 columns
// of its S once the softmax threads have read S(j); so the tile's next score
// product is issued only after the P V product that reads P(j) has
// completed.  While one tile's softmax runs, the tensor pipe works on the
// other tile's products.
__global__ void __launch_bounds__(fwd::NTF, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ o,
                       float* __restrict__ lse, int B, int T, int H, int* err,
                       long long timeout_ns) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* q_full = bars + 0;    // [2] by tile
  uint64_t* q_empty = bars + 2;   // [2] by tile: the pair's last score product is done
  uint64_t* k_full = bars + 4;    // [2] by stage
  uint64_t* k_empty = bars + 6;   // [2] by stage, one commit per tile
  uint64_t* v_full = bars + 8;    // [2]
  uint64_t* v_empty = bars + 10;  // [2]
  uint64_t* s_full = bars + 12;   // [2] by tile
  uint64_t* p_full = bars + 14;   // [2] by tile, one arrival per softmax warp
  uint64_t* pv_done = bars + 16;  // [2] by tile
  uint64_t* drain = bars + 18;    // [2] by tile (its MMA issuer)
  uint64_t* s0_read = bars + 20;  // [2] by tile 0's step parity: its softmax has S's row maxima
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 22);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long TH = (long)T * H;
  const int n_pairs = (int)((TH + 2 * BQ - 1) / (2 * BQ));
  const long n_items = (long)B * n_pairs;
  const int G = gridDim.x, cta = blockIdx.x;
  // Item u: sequence u % B (fastest, so concurrent CTAs share no K/V), pair
  // n_pairs - 1 - u / B (the heaviest first).
  auto item_b = [&](long u) { return (int)(u % B); };
  auto item_r0 = [&](long u) { return (long)(n_pairs - 1 - (int)(u / B)) * 2 * BQ; };
  // Key tiles query tile x of an item sees (up to its last row's token); the
  // K/V stream runs to tile 1's count, at most one more than tile 0's.
  auto key_tiles = [&](long u, int x) {
    const long last = min(item_r0(u) + (long)(x + 1) * BQ - 1, TH - 1);
    return (int)(last / H) / BKV + 1;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 2);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 2);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
      mbar_init(&drain[i], 1);
      mbar_init(&s0_read[i], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const CtaSync sync{abort_flag, err, timeout_ns};

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    int armed[6] = {-1, -1, -1, -1, -1, -1};  // q0, q1, k0, k1, v0, v1 parities for the drain
    long g = 0;  // key tiles streamed so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const long u = snake_item(cta, k, G, n_items);
      if (u < 0) break;
      const int b = item_b(u);
      const long r0 = item_r0(u);
      const int nkv = key_tiles(u, 1);
      for (int x = 0; x < 2 && ok; ++x) {
        // The previous pair's last score product of this tile has read Q.
        if (k > 0 && !sync.wait(&q_empty[x], (k - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&q_full[x], 2 * ATOM);
        const int y = (int)(r0 + x * BQ);  // rows past the sequence read as zero
        tma_load_3d(smem + Q_OFF + x * 32768, &tmQ, &q_full[x], 0, y, b);
        tma_load_3d(smem + Q_OFF + x * 32768 + ATOM, &tmQ, &q_full[x], 64, y, b);
        armed[x] = k & 1;
      }
      for (int j = 0; ok && j < nkv; ++j, ++g) {
        const int st = (int)(g & 1);
        const uint32_t ph = (uint32_t)(g >> 1) & 1u;
        if (!sync.wait(&k_empty[st], ph ^ 1u)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[st], 2 * ATOM);
        tma_load_3d(smem + K_OFF + st * 32768, &tmK, &k_full[st], 0, j * BKV, b);
        tma_load_3d(smem + K_OFF + st * 32768 + ATOM, &tmK, &k_full[st], 64, j * BKV, b);
        armed[2 + st] = (int)ph;
        if (!sync.wait(&v_empty[st], ph ^ 1u)) { ok = false; break; }
        mbar_arrive_expect_tx(&v_full[st], 2 * ATOM);
        tma_load_3d(smem + V_OFF + st * 32768, &tmV, &v_full[st], 0, j * BKV, b);
        tma_load_3d(smem + V_OFF + st * 32768 + ATOM, &tmV, &v_full[st], 64, j * BKV, b);
        armed[4 + st] = (int)ph;
      }
    }
    if (*abort_flag) {
      int none = 0;
      uint64_t* fb[6] = {&q_full[0], &q_full[1], &k_full[0], &k_full[1], &v_full[0], &v_full[1]};
      for (int i = 0; i < 6; ++i)
        if (armed[i] >= 0) mbar_wait_bounded(fb[i], (uint32_t)armed[i], &none, err, SITE_ATTN, timeout_ns / 8);
    }
  } else if ((warp == 1 || warp == 2) && lane == 0) {
    // ------------------------------------------------ MMA issuers
    // Warp 1 issues tile 0's products, warp 2 tile 1's: per key tile j,
    // S(j) = Q K(j)^T, then O += P(j) V(j) once the softmax warps have
    // written P(j).  An MMA issue holds its thread for about the MMA's run
    // time, so each issuer's waits overlap the other's MMAs; a commit tracks
    // the MMAs of its own thread.  Tile 1 runs half a step behind tile 0:
    // its S(j) is issued once tile 0's softmax warps have their S(j) row maxima,
    // so that it computes while they do and their softmax and tile 1's take
    // turns on the SM's schedulers instead of running at once.  Descriptors
    // are built once; a k-step or ring stage only moves the 14-bit
    // start-address field (shared memory < 256 KB: no carry).
    const int x = warp == 1 ? 0 : 1;
    constexpr uint32_t idS = idesc_bf16_mn(false, false, BQ, BKV);
    constexpr uint32_t idPV = idesc_bf16_mn(false, true, BQ, HD);
    constexpr uint64_t kStage = 32768 >> 4;
    auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * ATOM + (kk & 3) * 32) >> 4); };
    auto moff = [](int kk) { return (uint64_t)((kk * 2048) >> 4); };
    const uint64_t dQ = sdesc_sw128(smem_u32(smem + Q_OFF + x * 32768), 16, 1024);
    const uint64_t dK = sdesc_sw128(smem_u32(smem + K_OFF), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(smem + V_OFF), ATOM, 1024);  // MN-major
    const uint32_t s_t = tmem + x * BKV, o_t = tmem + 256 + x * HD;
    bool ok = true, issued = false;
    long g = 0, n = 0;  // key tiles streamed; this tile's (pair, key tile) steps
    long n0 = 0;        // tile 0's steps before the current pair (tile 1's issuer)
    for (int k = 0; ok; ++k) {
      const long u = snake_item(cta, k, G, n_items);
      if (u < 0) break;
      const int nkx = key_tiles(u, x), nkv = key_tiles(u, 1), nk0 = key_tiles(u, 0);
      if (!sync.wait(&q_full[x], k & 1)) { ok = false; break; }
      for (int j = 0; j < nkx; ++j, ++g, ++n) {
        const int st = (int)(g & 1);
        const uint32_t ph = (uint32_t)(g >> 1) & 1u;
        // S overwrites the previous step's P: wait for the product that reads it.
        if (!sync.wait(&k_full[st], ph) || (n > 0 && !sync.wait(&pv_done[x], (uint32_t)(n - 1) & 1u))) {
          ok = false;
          break;
        }
        // Tile 1: after tile 0's softmax has S(j)'s row maxima (tile 0 is at most
        // one step further on: its S(j + 2) needs the K stage that S(j) of
        // this tile releases, so the two alternating barriers cannot alias).
        if (x == 1 && j < nk0) {
          const long m = n0 + j;
          if (!sync.wait(&s0_read[m & 1], (uint32_t)(m >> 1) & 1u)) { ok = false; break; }
        }
        tc_fence_after();
        const uint64_t bk = dK + st * kStage;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16(s_t, dQ + koff(kk), bk + koff(kk), idS, kk > 0 ? 1u : 0u);
        umma_commit(&s_full[x]);
        umma_commit(&k_empty[st]);
        if (j == nkx - 1) umma_commit(&q_empty[x]);
        issued = true;
        // P(j) written (and O rescaled; the first step of a pair also
        // follows the softmax warps' read of the previous pair's O).
        if (!sync.wait(&p_full[x], (uint32_t)n & 1u) || !sync.wait(&v_full[st], ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t bv = dV + st * kStage;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          umma_bf16_tmem_a(o_t, s_t + kk * 8, bv + moff(kk), idPV, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[x]);
        umma_commit(&v_empty[st]);
      }
      // Key tiles past this tile's last row: release their stages unread (once
      // they have landed, so that the arrival counts toward their own phase).
      for (int j = nkx; ok && j < nkv; ++j, ++g) {
        const int st = (int)(g & 1);
        const uint32_t ph = (uint32_t)(g >> 1) & 1u;
        if (!sync.wait(&k_full[st], ph)) { ok = false; break; }
        mbar_arrive(&k_empty[st]);
        if (!sync.wait(&v_full[st], ph)) { ok = false; break; }
        mbar_arrive(&v_empty[st]);
      }
      n0 += nk0;
    }
    if ((!ok || *abort_flag) && issued) {
      int none = 0;
      umma_commit(&drain[x]);
      mbar_wait_bounded(&drain[x], 0, &none, err, SITE_ATTN, timeout_ns / 8);
    }
  } else if (warp >= 3) {
    // ------------------------------------------------ softmax / epilogue
    // Warps 3-6 serve tile 0, warps 7-10 tile 1; a warp reads TMEM lanes
    // 32 (warp % 4) .. + 31, so it owns the tile's rows 32 quarter ..
    // 32 quarter + 31 with quarter = warp % 4, one thread per row over all
    // 128 keys of a key tile: a row's maximum needs no exchange.
    const int x = (warp - 3) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_t = tmem + lane_off + x * BKV, o_t = tmem + lane_off + 256 + x * HD;
    const float sl2 = rsqrtf((float)HD) * kLog2e;
    bool ok = true;
    long n = 0;  // this tile's (pair, key tile) steps
    for (int k = 0; ok; ++k) {
      const long u = snake_item(cta, k, G, n_items);
      if (u < 0) break;
      const int b = item_b(u);
      const long rx0 = item_r0(u) + (long)x * BQ;
      const long r = rx0 + row;
      const bool valid = r < TH;
      const int nkx = key_tiles(u, x);
      const int tmax = (int)(min(r, TH - 1) / H);   // the last key this row sees
      const int t0 = (int)(min(rx0, TH - 1) / H);   // the tile's first row's token
      float m_run = -INFINITY, l_run = 0.f;  // in log2 units of the scaled scores
      for (int j = 0; j < nkx; ++j, ++n) {
        if (!sync.wait_warp(&s_full[x], (uint32_t)n & 1u)) { ok = false; break; }
        tc_fence_after();
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32cols_nowait(s_t + c * 32, raw[c]);
        tmem_ld_wait();
        float s[BKV];
#pragma unroll
        for (int i = 0; i < BKV; ++i) s[i] = __uint_as_float(raw[i >> 5][i & 31]);
        // Keys past a row's token occur only in tiles reaching beyond t0.
        if (j * BKV + BKV - 1 > t0) {
          const int lim = tmax - j * BKV;
#pragma unroll
          for (int i = 0; i < BKV; ++i)
            if (i > lim) s[i] = -INFINITY;
        }
        float m8[8];  // eight partial maxima: a short dependency chain
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
        for (int i = 8; i < BKV; ++i) m8[i & 7] = fmaxf(m8[i & 7], s[i]);
        float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        // Tile 1's S(j) may start now (it writes other columns): issued here,
        // its product lands about when this warpgroup's exponentials end
        // (measured against releasing it right after the load, or after P is
        // stored: 2 % faster, and 5 % faster).
        if (x == 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&s0_read[n & 1]);
        }
        mx *= sl2;
        float alpha = 1.f;
        if (mx > m_run + 8.f) {  // rescale only when the maximum grows by more than 2^8
          alpha = ex2(m_run - mx);  // 0 on the first tile
          l_run *= alpha;
          m_run = mx;
        }
        const float nm = -m_run;
        float ls0 = 0.f, ls1 = 0.f;
        uint32_t pk[BKV / 2];
#pragma unroll
        for (int i = 0; i < BKV; i += 2) {
          float e0, e1;
          fma2(e0, e1, s[i], s[i + 1], sl2, sl2, nm, nm);
          const float p0 = ex2(e0), p1 = ex2(e1);
          add2(ls0, ls1, p0, p1);
          pk[i / 2] = pack2(p0, p1);
        }
        l_run += ls0 + ls1;
        pairs64_to_tmem(s_t, pk);
        // O holds the products through P(j - 1) V(j - 1): S(j) was issued
        // after that product completed, and s_full tracks both.  The TMEM
        // load and store are warp-collective, so the whole warp takes the
        // branch when any row rescales (the others multiply by 1).
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < HD; c += 32) {
            float v[32];
            tmem_ld_32cols(o_t + c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st_32cols(o_t + c, v);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
      }
      if (!ok) break;
      // The pair's last P V product done: O is final.  The next pair's first
      // P V product (which overwrites O) follows this warp's next p_full
      // arrival, after these loads.
      if (!sync.wait_warp(&pv_done[x], (uint32_t)(n - 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      const float inv = 1.f / l_run;
      bf16* orow = o + ((long)b * TH + r) * HD;
#pragma unroll 1
      for (int c = 0; c < HD; c += 32) {
        float v[32];
        tmem_ld_32cols(o_t + c, v);
        if (valid) store_bf16_32(orow + c, v, inv);
      }
      if (valid) lse[(long)b * TH + r] = (m_run + log2f(l_run)) * kLn2;
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================
// backward, dQ pass: persistent CTAs, one per SM, each walking a list of
// 128-row query tiles (heaviest first, the order reversed every other round
// so that every CTA gets a similar share of key tiles).  Per query tile the
// CTA streams the key tiles it sees; Q and dO of the tile stay in shared
// memory as the A operands of S = Q K^T and dP = dO V^T while K and V stream
// through rings of their own (K, read by the S and dQ products, three stages;
// V, read only by dP and so released earlier, two), so the loads of the next
// key tiles are in flight while the current ones are used; dQ accumulates in
// tensor memory.  One counter g runs over every (query tile, key tile) pair
// of the CTA, so the rings, buffers and barrier phases carry on across query
// tiles: the score products of the next pair (the next query tile's first
// one included) are issued while the dQ product of the current one waits for
// dS, and the softmax warps drain a finished dQ while the tensor pipe already
// computes the next tile's scores.
// The next tile's Q and dO are prefetched into L2 while the current tile
// runs and loaded once the last S/dP of the current tile are done.  Every
// MMA is N = 128 wide (narrower ones run at ~60% of the tensor rate).
// ======================================================================
// delta[r] = sum_d O[r][d] dO[r][d] in fp32 for every packed row r (the
// softmax-gradient row term of the attention backward): 16 threads per row,
// one 16-byte slice each, then a 16-lane shuffle sum.
__global__ void __launch_bounds__(256)
    attn_delta_kernel(const bf16* __restrict__ o, const bf16* __restrict__ dout,
                      float* __restrict__ delta, long rows) {
  const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
  const int part = threadIdx.x & 15;
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = reinterpret_cast<const uint4*>(o + row * HD)[part];
    const uint4 d = reinterpret_cast<const uint4*>(dout + row * HD)[part];
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 fa = __bfloat1622float2(a2[k]), fd = __bfloat1622float2(d2[k]);
      acc = fmaf(fa.x, fd.x, acc);
      acc = fmaf(fa.y, fd.y, acc);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) delta[row] = acc;
}

namespace bdq {
constexpr int BQ = 128, BKV = 128;
constexpr int ATOM = 16384;                  // [128 rows][64] bf16
constexpr int KS = 3;                        // K ring stages (32 KB each): K is read by S and dQ
constexpr int VS = 2;                        // V ring stages (32 KB each): V only by dP
constexpr int K_OFF = 0;                     // KS x 32 KB ([128 keys][128 dims] = 2 atoms)
constexpr int V_OFF = K_OFF + KS * 32768;    // VS x 32 KB
constexpr int Q_OFF = V_OFF + VS * 32768;    // 32 KB, the current tile's 128 rows
constexpr int DO_OFF = Q_OFF + 32768;        // 32 KB
constexpr int BAR_OFF = DO_OFF + 32768;
constexpr int SMEM = BAR_OFF + 256 + 1024;
constexpr int kPrefetchAhead = 4;            // key tiles prefetched into L2 ahead of their load
static_assert(SMEM <= 232448, "dQ pass shared memory exceeds 227 KB");
}  // namespace bdq


__global__ void __launch_bounds__(NT, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmDO, const float* __restrict__ lse,
                          const float* __restrict__ delta, bf16* __restrict__ dq, long ldq, int B,
                          int T, int H, int* err, long long timeout_ns) {
  using namespace bdq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* k_full = bars + 0;              // [KS]
  uint64_t* k_empty = bars + KS;            // [KS]: the dQ product read it
  uint64_t* v_full = bars + 2 * KS;         // [VS]
  uint64_t* v_empty = bars + 2 * KS + VS;   // [VS]: the dP product read it
  uint64_t* s_full = bars + 2 * (KS + VS);      // S of the pair ready
  uint64_t* s_free = s_full + 1;            // S copied out, one arrival per softmax warp
  uint64_t* ds_full = s_full + 2;           // [2] by dS buffer, one arrival per softmax warp
  uint64_t* dq_done = s_full + 4;           // [2] by dS buffer: the dQ MMA that read it is done
  uint64_t* drain = s_full + 6;             // [2], one per MMA issuer
  uint64_t* qd_full = s_full + 8;           // the tile's Q and dO staged (TMA)
  uint64_t* qd_free = s_full + 9;           // the tile's last S / dP products are done
  uint64_t* dq_full = s_full + 10;          // the tile's last dQ product is done
  uint64_t* dp_full = s_full + 11;          // dP of the pair ready
  uint64_t* dp_free = s_full + 12;          // dP copied out, one arrival per softmax warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long TH = (long)T * H;
  const int n_qt = (int)((TH + BQ - 1) / BQ);
  const long n_tiles = (long)B * n_qt;
  const int G = gridDim.x, c = blockIdx.x;
  // tile u -> sequence b, first packed row r0, key tiles nkv
  auto tile_b = [&](long u) { return (int)(u % B); };
  auto tile_r0 = [&](long u) { return (long)(n_qt - 1 - (int)(u / B)) * BQ; };
  auto tile_nkv = [&](long u) {
    const long r0 = tile_r0(u);
    return (int)(min(r0 + BQ - 1, TH - 1) / H) / BKV + 1;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < KS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, NSW);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, NSW);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ds_full[i], NSW);
      mbar_init(&dq_done[i], 1);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(qd_full, 1);
    mbar_init(qd_free, 1);
    mbar_init(dq_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const CtaSync sync{abort_flag, err, timeout_ns};
  // TMEM columns: S at 0, dP at 128, dQ at 256, dS at 384 and 448 (bf16 pairs,
  // by the parity of the pair counter g).

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer (Q, dO per tile; K, V rings)
    int armed_qd = -1;
    int armed_k[KS], armed_v[VS];
    for (int i = 0; i < KS; ++i) armed_k[i] = -1;
    for (int i = 0; i < VS; ++i) armed_v[i] = -1;
    long g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const long u = snake_item(c, k, G, n_tiles);
      if (u < 0) break;
      const int b = tile_b(u);
      const int r0 = (int)tile_r0(u);
      if (k > 0 && !sync.wait(qd_free, (k - 1) & 1)) break;
      mbar_arrive_expect_tx(qd_full, 4 * ATOM);
      tma_load_3d(smem + Q_OFF, &tmQ, qd_full, 0, r0, b);
      tma_load_3d(smem + Q_OFF + ATOM, &tmQ, qd_full, 64, r0, b);
      tma_load_3d(smem + DO_OFF, &tmDO, qd_full, 0, r0, b);
      tma_load_3d(smem + DO_OFF + ATOM, &tmDO, qd_full, 64, r0, b);
      armed_qd = k & 1;
      const long un = snake_item(c, k + 1, G, n_tiles);
      if (un >= 0) {  // the next tile's rows into L2 while this one runs
        const int bn = tile_b(un), rn = (int)tile_r0(un);
        tma_prefetch_l2_3d(&tmQ, 0, rn, bn);
        tma_prefetch_l2_3d(&tmQ, 64, rn, bn);
        tma_prefetch_l2_3d(&tmDO, 0, rn, bn);
        tma_prefetch_l2_3d(&tmDO, 64, rn, bn);
      }
      const int nkv = tile_nkv(u);
      for (int j = 0; j < nkv; ++j, ++g) {
        if (j + kPrefetchAhead < nkv) {  // key tiles a few pairs ahead into L2
          tma_prefetch_l2_3d(&tmK, 0, (j + kPrefetchAhead) * BKV, b);
          tma_prefetch_l2_3d(&tmK, 64, (j + kPrefetchAhead) * BKV, b);
          tma_prefetch_l2_3d(&tmV, 0, (j + kPrefetchAhead) * BKV, b);
          tma_prefetch_l2_3d(&tmV, 64, (j + kPrefetchAhead) * BKV, b);
        }
        const int ks = (int)(g % KS), vs = (int)(g % VS);
        const uint32_t kph = (uint32_t)(g / KS) & 1u, vph = (uint32_t)(g / VS) & 1u;
        if (!sync.wait(&v_empty[vs], vph ^ 1u)) { ok = false; break; }
        mbar_arrive_expect_tx(&v_full[vs], 2 * ATOM);
        tma_load_3d(smem + V_OFF + vs * 32768, &tmV, &v_full[vs], 0, j * BKV, b);
        tma_load_3d(smem + V_OFF + vs * 32768 + ATOM, &tmV, &v_full[vs], 64, j * BKV, b);
        armed_v[vs] = (int)vph;
        if (!sync.wait(&k_empty[ks], kph ^ 1u)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[ks], 2 * ATOM);
        tma_load_3d(smem + K_OFF + ks * 32768, &tmK, &k_full[ks], 0, j * BKV, b);
        tma_load_3d(smem + K_OFF + ks * 32768 + ATOM, &tmK, &k_full[ks], 64, j * BKV, b);
        armed_k[ks] = (int)kph;
      }
    }
    if (*abort_flag) {
      int none = 0;
      if (armed_qd >= 0)
        mbar_wait_bounded(qd_full, (uint32_t)armed_qd, &none, err, SITE_ATTN, timeout_ns / 8);
      for (int i = 0; i < KS; ++i)
        if (armed_k[i] >= 0)
          mbar_wait_bounded(&k_full[i], (uint32_t)armed_k[i], &none, err, SITE_ATTN,
                            timeout_ns / 8);
      for (int i = 0; i < VS; ++i)
        if (armed_v[i] >= 0)
          mbar_wait_bounded(&v_full[i], (uint32_t)armed_v[i], &none, err, SITE_ATTN,
                            timeout_ns / 8);
    }
  } else if ((warp == 1 || warp == 3) && lane == 0) {
    // ------------------------------------------------ MMA issuers
    // Two threads issue the MMAs: warp 1 the S = Q K^T and dP = dO V^T
    // products of every pair, warp 3 the dQ += dS K products.  An MMA issue
    // holds its thread for about the MMA's run time, so with one issuer every
    // barrier wait and commit between two MMA groups left the tensor pipe
    // idle; with two, one stream's bookkeeping overlaps the other's MMAs.  A
    // commit tracks the MMAs of its own thread, which is exactly what each
    // release needs (K of pair g is last read by dQ(g), which follows S(g)
    // through the softmax warps' dS).  Descriptors are built once; a k-step or
    // ring stage only moves the start-address field.
    constexpr uint32_t idS = idesc_bf16_mn(false, false, BQ, BKV);
    constexpr uint32_t idQ = idesc_bf16_mn(false, true, BQ, HD);
    constexpr uint64_t kStage = 32768 >> 4;
    auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * ATOM + (kk & 3) * 32) >> 4); };
    auto moff = [](int kk) { return (uint64_t)((kk * 2048) >> 4); };
    bool ok = true, issued = false;
    long g = 0;
    if (warp == 1) {
      const uint64_t dKk = sdesc_sw128(smem_u32(smem + K_OFF), 16, 1024);    // K-major
      const uint64_t dVk = sdesc_sw128(smem_u32(smem + V_OFF), 16, 1024);
      const uint64_t dQk = sdesc_sw128(smem_u32(smem + Q_OFF), 16, 1024);
      const uint64_t dOk = sdesc_sw128(smem_u32(smem + DO_OFF), 16, 1024);
      for (int k = 0; ok; ++k) {
        const long u = snake_item(c, k, G, n_tiles);
        if (u < 0) break;
        const int nkv = tile_nkv(u);
        if (!sync.wait(qd_full, (uint32_t)k & 1u)) { ok = false; break; }
        for (int j = 0; j < nkv; ++j, ++g) {
          // S(g), then dP(g), each into its TMEM buffer once pair g - 1's copy
          // of it is out: the softmax warps start on S(g) while dP(g) runs.
          const int ks = (int)(g % KS), vs = (int)(g % VS);
          if (!sync.wait(&k_full[ks], (uint32_t)(g / KS) & 1u) ||
              (g > 0 && !sync.wait(s_free, (uint32_t)(g - 1) & 1u))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bk = dKk + ks * kStage, bv = dVk + vs * kStage;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16(tmem + 0, dQk + koff(kk), bk + koff(kk), idS, kk > 0 ? 1u : 0u);
          umma_commit(s_full);
          if (!sync.wait(&v_full[vs], (uint32_t)(g / VS) & 1u) ||
              (g > 0 && !sync.wait(dp_free, (uint32_t)(g - 1) & 1u))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16(tmem + 128, dOk + koff(kk), bv + koff(kk), idS, kk > 0 ? 1u : 0u);
          umma_commit(dp_full);
          umma_commit(&v_empty[vs]);
          if (j == nkv - 1) umma_commit(qd_free);  // the tile's Q, dO are read for the last time
          issued = true;
        }
      }
    } else {
      const uint64_t dKm = sdesc_sw128(smem_u32(smem + K_OFF), ATOM, 1024);  // MN-major
      for (int k = 0; ok; ++k) {
        const long u = snake_item(c, k, G, n_tiles);
        if (u < 0) break;
        const int nkv = tile_nkv(u);
        for (int j = 0; j < nkv; ++j, ++g) {
          // dQ (+)= dS(g) K(g), dS(g) read from tensor memory
          const int ks = (int)(g % KS), db = (int)(g & 1);
          if (!sync.wait(&ds_full[db], (uint32_t)(g >> 1) & 1u)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bk = dKm + ks * kStage;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            umma_bf16_tmem_a(tmem + 256, tmem + 384 + db * 64 + kk * 8, bk + moff(kk), idQ,
                             (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&dq_done[db]);
          umma_commit(&k_empty[ks]);
          if (j == nkv - 1) umma_commit(dq_full);
          issued = true;
        }
      }
    }
    if ((!ok || *abort_flag) && issued) {
      int none = 0;
      umma_commit(&drain[warp == 1 ? 0 : 1]);
      mbar_wait_bounded(&drain[warp == 1 ? 0 : 1], 0, &none, err, SITE_ATTN, timeout_ns / 8);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax warps
    // Warp 4 + 4 half + quarter owns packed rows 32 quarter .. 32 quarter + 31
    // (its TMEM lanes) and key columns 64 half .. 64 half + 63 of each tile.
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = rsqrtf((float)HD) * kLog2e;
    bool ok = true;
    long g = 0;
    // this row's lse and delta, one tile ahead
    auto row_data = [&](long u, float& l2, float& d) {
      const long r = tile_r0(u) + row;
      const bool v = r < TH;
      const long grow = (long)tile_b(u) * TH + r;
      d = v ? delta[grow] : 0.f;
      l2 = v ? lse[grow] * kLog2e : 0.f;
    };
    long u = snake_item(c, 0, G, n_tiles);
    float lse2 = 0.f, dl = 0.f;
    if (u >= 0) row_data(u, lse2, dl);
    for (int k = 0; ok && u >= 0; ++k) {
      const int b = tile_b(u);
      const long r0 = tile_r0(u);
      const long r = r0 + row;
      const bool valid = r < TH;
      const int t = (int)(r / H);
      const int nkv = tile_nkv(u);
      const long un = snake_item(c, k + 1, G, n_tiles);
      float lse2_n = 0.f, dl_n = 0.f;
      if (un >= 0) row_data(un, lse2_n, dl_n);
      // Rows of this tile hold tokens t0 .. ; a key tile needs the mask only
      // where it reaches past t0 (or the tile has rows past the sequence).
      const int t0 = (int)(r0 / H);
      const bool rows_ragged = r0 + BQ > TH;
      for (int j = 0; j < nkv; ++j, ++g) {
        if (!sync.wait_warp(s_full, (uint32_t)g & 1u)) { ok = false; break; }
        tc_fence_after();
        float s[64], dp[64];
        {
          uint32_t r0_[32], r1_[32];
          tmem_ld_32cols_nowait(tmem + lane_off + half * 64, r0_);
          tmem_ld_32cols_nowait(tmem + lane_off + half * 64 + 32, r1_);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(r0_[i]);
            s[32 + i] = __uint_as_float(r1_[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        const int key0 = j * BKV + half * 64;
        const bool need_mask = rows_ragged || key0 + 63 > t0;
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = ex2(fmaf(s[i], sl2, -lse2));
        if (need_mask) {  // key key0 + i is visible to token t; padding rows see nothing
          const int lim = valid ? t - key0 : -1;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i > lim) s[i] = 0.f;
        }
        if (!sync.wait_warp(dp_full, (uint32_t)g & 1u)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t r2_[32], r3_[32];
          tmem_ld_32cols_nowait(tmem + lane_off + 128 + half * 64, r2_);
          tmem_ld_32cols_nowait(tmem + lane_off + 128 + half * 64 + 32, r3_);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            dp[i] = __uint_as_float(r2_[i]);
            dp[32 + i] = __uint_as_float(r3_[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dp_free);
#pragma unroll
        for (int i = 0; i < 64; i += 2)
          sub_mul2(s[i], s[i + 1], dp[i], dp[i + 1], dl, dl, s[i], s[i + 1]);
        const int db = (int)(g & 1);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack2(s[2 * i], s[2 * i + 1]);
        if (g > 1) {  // the dQ MMA of pair g - 2 has read this dS buffer
          if (!sync.wait_warp(&dq_done[db], (uint32_t)((g >> 1) - 1) & 1u)) { ok = false; break; }
          tc_fence_after();
        }
        pairs_to_tmem(tmem + lane_off + 384 + db * 64 + half * 32, pk);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ds_full[db]);
      }
      if (!ok) break;
      // dQ MMAs complete in issue order: the tile's last one done means all are.
      if (!sync.wait_warp(dq_full, (uint32_t)k & 1u)) { ok = false; break; }
      tc_fence_after();
      const float scale = rsqrtf((float)HD);
      bf16* qrow = dq + ((long)b * T + t) * ldq + (long)(r % H) * HD;
#pragma unroll 1
      for (int cc = 2 * half; cc < 2 * half + 2; ++cc) {
        float v[32];
        tmem_ld_32cols(tmem + lane_off + 256 + cc * 32, v);
        if (valid) store_bf16_32(qrow + cc * 32, v, scale);
      }
      tc_fence_before();
      u = un;
      lse2 = lse2_n;
      dl = dl_n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================
// backward, dK/dV pass: 128 keys per CTA against 128-row query tiles over
// every packed row that can see them (all heads: the MQA head sum).  K and
// V, the same for every query tile, sit in tensor memory as the A operands
// of S^T = K Q^T and dP^T = V dO^T; one 128-column score buffer holds S^T,
// is copied out, then holds dP^T.  dV += P^T dO and dK += dS^T Q accumulate
// in tensor memory; every MMA is N = 128 wide.
// ======================================================================
namespace bkv {
constexpr int BKV = 128, BQ = 128;
constexpr int ATOM = 16384;                   // [128 rows][64] bf16
constexpr int QS = 3;                         // Q ring stages (32 KB each)
constexpr int DS = 2;                         // dO ring stages (32 KB each)
constexpr int Q_OFF = 0;
constexpr int DO_OFF = Q_OFF + QS * 32768;
constexpr int K_OFF = DO_OFF + DS * 32768;    // 32 KB, the CTA's 128 keys
constexpr int V_OFF = K_OFF + 32768;          // 32 KB
constexpr int INFO_OFF = V_OFF + 32768;       // [2][128] x (lse2, delta)
constexpr int BAR_OFF = INFO_OFF + 2 * 128 * 8;
constexpr int USED = BAR_OFF + 256;
constexpr int SMEM = 232448;                  // the per-CTA maximum
constexpr int SLACK = SMEM - USED;            // room to align the base to 1024 bytes
constexpr int kGroup = 8;                     // sequences per launch group (L2 residency)
static_assert(SLACK >= 0, "dK/dV pass shared memory exceeds 227 KB");
}  // namespace bkv

// dK/dV pass: one CTA per 128-key tile, K and V resident in shared memory,
// query tiles (Q, dO) streamed through two TMA rings.  Per query tile i one
// MMA thread issues S^T(i) = K Q(i)^T and dP^T(i) = V dO(i)^T, another
// dV += P^T(i) dO(i) and dK += dS^T(i) Q(i), so the gradient products of
// one tile run while the score products of the next wait for the softmax
// warps.  S^T and dP^T share one 128-column score buffer; the softmax warps
// write P^T and dS^T as bf16 into tensor memory, where the dV and dK
// products read them as their A operand.  Shared-memory traffic per query tile is then the
// TMA fills (64 KB) and the B operands plus K, V (192 KB): below the tensor
// pipe's time for the four 128 x 128 x 128 products.
__global__ void __launch_bounds__(NT, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmDO,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const float* __restrict__ lse,
                            const float* __restrict__ delta, bf16* __restrict__ dk, long ldk,
                            bf16* __restrict__ dv, long ldv, int T, int H, int* err,
                            long long timeout_ns) {
  using namespace bkv;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > (uint32_t)SLACK) {  // uniform: no barrier or tensor memory touched yet
    if (threadIdx.x == 0) raise_error(err, DEV_CUDA, SITE_ATTN, (int)pad);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* kv_full = bars + 0;      // K, V tiles landed (TMA)
  uint64_t* q_full = bars + 1;       // [QS]
  uint64_t* q_empty = bars + 4;      // [QS]
  uint64_t* do_full = bars + 7;      // [DS]
  uint64_t* do_empty = bars + 9;     // [DS]
  uint64_t* sc_full = bars + 11;     // score buffer holds S^T, then dP^T
  uint64_t* sc_free = bars + 12;     // copied out, one arrival per softmax warp
  uint64_t* p_full = bars + 13;      // P^T stored, one arrival per softmax warp
  uint64_t* ds_full = bars + 14;     // dS^T stored, one arrival per softmax warp
  uint64_t* pt_free = bars + 15;     // dV MMAs done reading P^T (and the earlier dV, dK ones)
  uint64_t* dst_free = bars + 16;    // dK MMAs done reading dS^T (and the earlier dV, dK ones)
  uint64_t* drain = bars + 17;       // [2], one per MMA issuer
  uint64_t* info_full = bars + 19;   // [2], 32 arrivals (warp 3)
  uint64_t* info_free = bars + 21;   // [2], one arrival per softmax warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 23);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* info_lse = reinterpret_cast<float*>(smem + INFO_OFF);  // [2][128]
  float* info_dl = info_lse + 2 * 128;                          // [2][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Launch order: sequences in groups of kGroup; inside a group the heaviest
  // key tiles (the earliest keys, which meet every later query row) first,
  // sequence fastest.  The Q and dO rows that a group streams stay resident
  // in L2 while its CTAs run, and heavy tiles still start first.
  const int NY = (T + BKV - 1) / BKV;
  const int g0 = (int)(blockIdx.x / (kGroup * NY)) * kGroup;  // first sequence of the group
  const int gsz = min(kGroup, (int)(gridDim.x / NY) - g0);
  const int r = (int)blockIdx.x - g0 * NY;
  const int b = g0 + r % gsz;
  const int j0 = (r / gsz) * BKV;
  const long TH = (long)T * H;
  const long rt0 = ((long)j0 * H) / BQ;
  const int n_rt = (int)((TH + BQ - 1) / BQ - rt0);

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < QS; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < DS; ++i) {
      mbar_init(&do_full[i], 1);
      mbar_init(&do_empty[i], 2);  // released by a commit of each MMA issuer
    }
    mbar_init(sc_full, 1);
    mbar_init(sc_free, NSW);
    mbar_init(p_full, NSW);
    mbar_init(ds_full, NSW);
    mbar_init(pt_free, 1);
    mbar_init(dst_free, 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&info_full[i], 32);
      mbar_init(&info_free[i], NSW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const CtaSync sync{abort_flag, err, timeout_ns};
  // TMEM columns: score at 0, dV at 128, dK at 256, P^T at 384, dS^T at 448
  // (bf16 pairs: query rows 2c, 2c + 1 in column c).

  if (warp == 3) {
    // ------------------------------------------------ per-row data of each query tile
    for (int i = 0; i < n_rt; ++i) {
      const int st = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      if (!sync.wait(&info_free[st], ph ^ 1u)) break;
      for (int c = lane; c < BQ; c += 32) {
        const long rr = (rt0 + i) * BQ + c;
        const bool v = rr < TH;
        info_lse[st * 128 + c] = v ? lse[(long)b * TH + rr] * kLog2e : 0.f;
        info_dl[st * 128 + c] = v ? delta[(long)b * TH + rr] : 0.f;
      }
      mbar_arrive(&info_full[st]);
    }
  }

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer (K, V; Q ring, dO ring)
    mbar_arrive_expect_tx(kv_full, 4 * ATOM);
    tma_load_3d(smem + K_OFF, &tmK, kv_full, 0, j0, b);
    tma_load_3d(smem + K_OFF + ATOM, &tmK, kv_full, 64, j0, b);
    tma_load_3d(smem + V_OFF, &tmV, kv_full, 0, j0, b);
    tma_load_3d(smem + V_OFF + ATOM, &tmV, kv_full, 64, j0, b);
    int armed_q[QS], armed_do[DS];
    for (int i = 0; i < QS; ++i) armed_q[i] = -1;
    for (int i = 0; i < DS; ++i) armed_do[i] = -1;
    for (int i = 0; i < n_rt; ++i) {
      const int rr = (int)((rt0 + i) * BQ);
      const int qs = i % QS, ds = i % DS;
      const uint32_t qph = (i / QS) & 1, dph = (i / DS) & 1;
      if (!sync.wait(&q_empty[qs], qph ^ 1u)) break;
      mbar_arrive_expect_tx(&q_full[qs], 2 * ATOM);
      tma_load_3d(smem + Q_OFF + qs * 32768, &tmQ, &q_full[qs], 0, rr, b);
      tma_load_3d(smem + Q_OFF + qs * 32768 + ATOM, &tmQ, &q_full[qs], 64, rr, b);
      armed_q[qs] = (int)qph;
      if (!sync.wait(&do_empty[ds], dph ^ 1u)) break;
      mbar_arrive_expect_tx(&do_full[ds], 2 * ATOM);
      tma_load_3d(smem + DO_OFF + ds * 32768, &tmDO, &do_full[ds], 0, rr, b);
      tma_load_3d(smem + DO_OFF + ds * 32768 + ATOM, &tmDO, &do_full[ds], 64, rr, b);
      armed_do[ds] = (int)dph;
    }
    if (*abort_flag) {
      int none = 0;
      mbar_wait_bounded(kv_full, 0, &none, err, SITE_ATTN, timeout_ns / 8);
      for (int i = 0; i < QS; ++i)
        if (armed_q[i] >= 0)
          mbar_wait_bounded(&q_full[i], (uint32_t)armed_q[i], &none, err, SITE_ATTN,
                            timeout_ns / 8);
      for (int i = 0; i < DS; ++i)
        if (armed_do[i] >= 0)
          mbar_wait_bounded(&do_full[i], (uint32_t)armed_do[i], &none, err, SITE_ATTN,
                            timeout_ns / 8);
    }
  } else if ((warp == 1 || warp == 2) && lane == 0) {
    // ------------------------------------------------ MMA issuers
    // Warp 1 issues the score products S^T(i) = K Q(i)^T and dP^T(i) =
    // V dO(i)^T, warp 2 (idle between the TMEM allocation and release) the
    // gradient products dV += P^T(i) dO(i) and dK += dS^T(i) Q(i).  An MMA
    // issue holds its thread for about the MMA's run time, so one stream's
    // waits and commits overlap the other stream's MMAs.  A commit tracks the
    // MMAs of its own thread: dO(i) is read by dP^T(i) (warp 1) and dV(i)
    // (warp 2), so its ring slot is released by a commit from each; Q(i) is
    // last read by dK(i), which follows S^T(i) through the softmax warps'
    // dS^T.  Each issuer waits for every shared-memory operand it reads that
    // its other waits do not already prove landed.  Descriptors are built once; a k-step
    // or ring stage only moves the 14-bit start-address field (shared memory
    // < 256 KB: no carry).
    constexpr uint32_t idS = idesc_bf16_mn(false, false, BKV, BQ);
    constexpr uint32_t idG = idesc_bf16_mn(false, true, BKV, HD);
    constexpr uint64_t kStage = 32768 >> 4;
    // start-field offsets of k-step kk: K-major across 64-wide atoms, MN-major by 16 rows
    auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * ATOM + (kk & 3) * 32) >> 4); };
    auto moff = [](int kk) { return (uint64_t)((kk * 2048) >> 4); };
    bool ok = sync.wait(kv_full, 0), issued = false;
    if (warp == 1) {
      const uint64_t dK = sdesc_sw128(smem_u32(smem + K_OFF), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(smem + V_OFF), 16, 1024);
      const uint64_t dQk = sdesc_sw128(smem_u32(smem + Q_OFF), 16, 1024);    // K-major
      const uint64_t dOk = sdesc_sw128(smem_u32(smem + DO_OFF), 16, 1024);
      for (int i = 0; ok && i < n_rt; ++i) {
        const int qs = i % QS, ds = i % DS;
        const uint32_t qph = (i / QS) & 1, dph = (i / DS) & 1;
        // S^T(i) once dP^T(i - 1) has been copied out of the score buffer
        if (!sync.wait(&q_full[qs], qph) || (i > 0 && !sync.wait(sc_free, 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t bq = dQk + qs * kStage;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16(tmem, dK + koff(kk), bq + koff(kk), idS, kk > 0 ? 1u : 0u);
        umma_commit(sc_full);
        issued = true;
        // dP^T(i) once S^T(i) has been copied out
        if (!sync.wait(&do_full[ds], dph) || !sync.wait(sc_free, 0)) { ok = false; break; }
        tc_fence_after();
        const uint64_t bo = dOk + ds * kStage;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16(tmem, dV + koff(kk), bo + koff(kk), idS, kk > 0 ? 1u : 0u);
        umma_commit(sc_full);
        umma_commit(&do_empty[ds]);
      }
    } else {
      const uint64_t dQm = sdesc_sw128(smem_u32(smem + Q_OFF), ATOM, 1024);  // MN-major
      const uint64_t dOm = sdesc_sw128(smem_u32(smem + DO_OFF), ATOM, 1024);
      for (int i = 0; ok && i < n_rt; ++i) {
        const int qs = i % QS, ds = i % DS;
        const uint32_t dph = (i / DS) & 1;
        // dV += P^T dO of tile i, P^T read from tensor memory.  P^T(i) being
        // stored says that S^T(i), hence Q(i), is done, but not that dO(i)
        // has landed: wait for its slot here too.  (Its next fill needs this
        // thread's release, so the parity cannot alias.)  dK(i) needs no such
        // wait: dS^T(i) comes from dP^T(i), which read dO(i) after Q(i).
        if (!sync.wait(p_full, i & 1) || !sync.wait(&do_full[ds], dph)) { ok = false; break; }
        tc_fence_after();
        const uint64_t bo = dOm + ds * kStage;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          umma_bf16_tmem_a(tmem + 128, tmem + 384 + kk * 8, bo + moff(kk), idG,
                           (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(pt_free);
        umma_commit(&do_empty[ds]);
        issued = true;
        // dK += dS^T Q of tile i
        if (!sync.wait(ds_full, i & 1)) { ok = false; break; }
        tc_fence_after();
        const uint64_t bq = dQm + qs * kStage;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          umma_bf16_tmem_a(tmem + 256, tmem + 448 + kk * 8, bq + moff(kk), idG,
                           (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(dst_free);
        umma_commit(&q_empty[qs]);
      }
    }
    if ((!ok || *abort_flag) && issued) {
      int none = 0;
      uint64_t* d = &drain[warp == 1 ? 0 : 1];
      umma_commit(d);
      mbar_wait_bounded(d, 0, &none, err, SITE_ATTN, timeout_ns / 8);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax warps
    // Warp 4 + 4 half + quarter owns key rows 32 quarter .. 32 quarter + 31
    // (its TMEM lanes) and query columns 64 half .. 64 half + 63.
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int krow = quarter * 32 + lane;  // key inside the tile
    const int key = j0 + krow;
    const bool kvalid = key < T;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = rsqrtf((float)HD) * kLog2e;
    bool ok = true;
    for (int i = 0; i < n_rt; ++i) {
      const int st = i & 1;
      // packed rows rowbase .. rowbase + 63 are this thread's query columns
      const long rowbase = (rt0 + i) * BQ + half * 64;
      if (!sync.wait_warp(sc_full, 0) || !sync.wait_warp(&info_full[st], (i >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[64];
      {
        uint32_t r0_[32], r1_[32];
        tmem_ld_32cols_nowait(tmem + lane_off + half * 64, r0_);
        tmem_ld_32cols_nowait(tmem + lane_off + half * 64 + 32, r1_);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0_[c]);
          x[32 + c] = __uint_as_float(r1_[c]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sc_free);
      const float* il = info_lse + st * 128 + half * 64;
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = reinterpret_cast<const float4*>(il)[c4];
        x[c4 * 4 + 0] = ex2(fmaf(x[c4 * 4 + 0], sl2, -l4.x));
        x[c4 * 4 + 1] = ex2(fmaf(x[c4 * 4 + 1], sl2, -l4.y));
        x[c4 * 4 + 2] = ex2(fmaf(x[c4 * 4 + 2], sl2, -l4.z));
        x[c4 * 4 + 3] = ex2(fmaf(x[c4 * 4 + 3], sl2, -l4.w));
      }
      // Row rr (token rr / H) sees this key iff rr >= key * H; rows at or past
      // T H are padding.  Warp-uniform test: only tiles on the diagonal or at
      // the end of the sequence mask anything.
      if (rowbase < (long)(j0 + BKV - 1) * H || rowbase + 64 > TH) {
        const long lo = (long)key * H - rowbase, hi = TH - rowbase;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < lo || c >= hi) x[c] = 0.f;
      }
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) pk[j] = pack2(x[2 * j], x[2 * j + 1]);
      if (i > 0 && !sync.wait_warp(pt_free, (i - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      pairs_to_tmem(tmem + lane_off + 384 + half * 32, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // dS^T = P^T (dP^T - delta), with P^T as stored (bf16)
      if (!sync.wait_warp(sc_full, 1)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t r0_[32], r1_[32];
        tmem_ld_32cols_nowait(tmem + lane_off + half * 64, r0_);
        tmem_ld_32cols_nowait(tmem + lane_off + half * 64 + 32, r1_);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0_[c]);
          x[32 + c] = __uint_as_float(r1_[c]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sc_free);
      const float* id = info_dl + st * 128 + half * 64;
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 d4 = reinterpret_cast<const float4*>(id)[c4];
        const uint32_t p01 = pk[c4 * 2], p23 = pk[c4 * 2 + 1];
        float a0, a1, a2, a3;
        sub_mul2(a0, a1, x[c4 * 4 + 0], x[c4 * 4 + 1], d4.x, d4.y, __uint_as_float(p01 << 16),
                 __uint_as_float(p01 & 0xffff0000u));
        sub_mul2(a2, a3, x[c4 * 4 + 2], x[c4 * 4 + 3], d4.z, d4.w, __uint_as_float(p23 << 16),
                 __uint_as_float(p23 & 0xffff0000u));
        pk[c4 * 2] = pack2(a0, a1);
        pk[c4 * 2 + 1] = pack2(a2, a3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&info_free[st]);
      if (i > 0 && !sync.wait_warp(dst_free, (i - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      pairs_to_tmem(tmem + lane_off + 448 + half * 32, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    if (ok && n_rt > 0 && sync.wait_warp(dst_free, (n_rt - 1) & 1)) {
      tc_fence_after();
      const float scale = rsqrtf((float)HD);
      const long tok = (long)b * T + key;
#pragma unroll 1
      for (int c = 2 * half; c < 2 * half + 2; ++c) {
        float v[32];
        tmem_ld_32cols(tmem + lane_off + 128 + c * 32, v);
        if (kvalid) store_bf16_32(dv + tok * ldv + c * 32, v, 1.f);
        tmem_ld_32cols(tmem + lane_off + 256 + c * 32, v);
        if (kvalid) store_bf16_32(dk + tok * ldk + c * 32, v, scale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// 3-D map over a (B, rows, 128) bf16 tensor: box {64, box_rows, 1}; rows past
// `rows` read as zero, so a tile never sees the next sequence.
bool map3(CUtensorMap* m, const void* base, long rows, int B, int box_rows) {
  const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)rows, (uint64_t)B};
  const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)rows * HD * 2};
  const uint32_t box[3] = {64, (uint32_t)box_rows, 1};
  return make_tmap_bf16(m, base, 3, dims, strides, box);
}

template <class K>
cudaError_t set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t attention_fwd_tc(int B, int T, int H, const void* q, const void* k, const void* v,
                             void* o, float* lse, const Ctx& ctx) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(attn_fwd_tc_kernel, fwd::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const long TH = (long)T * H;
  CUtensorMap mq, mk, mv;
  if (!map3(&mq, q, TH, B, fwd::BQ) || !map3(&mk, k, T, B, fwd::BKV) ||
      !map3(&mv, v, T, B, fwd::BKV))
    return cudaErrorInvalidValue;
  const long items = (long)B * ((TH + 2 * fwd::BQ - 1) / (2 * fwd::BQ));
  const unsigned grid = (unsigned)std::min<long>(items, std::max(ctx.num_sms, 1));
  attn_fwd_tc_kernel<<<grid, fwd::NTF, fwd::SMEM, ctx.stream>>>(mq, mk, mv, (nc::bf16*)o, lse, B, T,
                                                          H, ctx.err, ctx.timeout_ns);
  return launched(1);
}

cudaError_t attention_bwd_tc(int B, int T, int H, const void* q, const void* k, const void* v,
                             const void* o, const float* lse, const void* dout, void* dq,
                             long ldq, void* dk, long ldk, void* dv, long ldv, float* delta,
                             const Ctx& ctx) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(attn_bwd_dq_tc_kernel, bdq::SMEM);
    if (e == cudaSuccess) e = set_smem(attn_bwd_dkdv_tc_kernel, bkv::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const long TH = (long)T * H;
  CUtensorMap mq, mdo, mk, mv;
  static_assert(bkv::BKV == bdq::BKV && bkv::BQ == bdq::BQ, "both passes share their maps");
  if (!map3(&mk, k, T, B, bdq::BKV) || !map3(&mv, v, T, B, bdq::BKV) ||
      !map3(&mq, q, TH, B, bdq::BQ) || !map3(&mdo, dout, TH, B, bdq::BQ))
    return cudaErrorInvalidValue;
  const long rows = (long)B * TH;
  attn_delta_kernel<<<(unsigned)((rows * 16 + 255) / 256), 256, 0, ctx.stream>>>(
      (const nc::bf16*)o, (const nc::bf16*)dout, delta, rows);
  note_launch(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long dq_tiles = (long)B * ((TH + bdq::BQ - 1) / bdq::BQ);
  const unsigned gq = (unsigned)std::min<long>(dq_tiles, std::max(ctx.num_sms, 1));
  attn_bwd_dq_tc_kernel<<<gq, NT, bdq::SMEM, ctx.stream>>>(
      mk, mv, mq, mdo, lse, delta, (nc::bf16*)dq, ldq, B, T, H, ctx.err, ctx.timeout_ns);
  note_launch(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned gk = (unsigned)B * (unsigned)((T + bkv::BKV - 1) / bkv::BKV);
  attn_bwd_dkdv_tc_kernel<<<gk, NT, bkv::SMEM, ctx.stream>>>(
      mq, mdo, mk, mv, lse, delta, (nc::bf16*)dk, ldk,
      (nc::bf16*)dv, ldv, T, H, ctx.err, ctx.timeout_ns);
  return launched(1);
}

}  // namespace nc
