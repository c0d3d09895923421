// Persistent bf16 GEMM on the 5th-generation tensor cores (sm_100 family,
// built for sm_103a): TMA -> 128B-swizzled shared memory -> tcgen05.mma ->
// fp32 accumulator in tensor memory -> tcgen05.ld -> fused epilogue.
//
//   C[m][n] = sum_k A(m, k) B(n, k)
//   A(m, k) = A[m * lda + k] (K-major)  or  A[k * lda + m] (A_MN: M-major)
//   B(n, k) = B[n * ldb + k] (K-major)  or  B[k * ldb + n] (B_MN: N-major)
//
// Two CTAs of a cluster (a CTA pair on two SMs) compute one 256 x 256 output
// tile with cta_group::2 MMAs: each CTA loads 128 rows of the A tile and 128
// rows of the B tile (64 K-columns a stage, 32 KB, 6 stages), the even CTA
// issues the MMAs, and each CTA's tensor memory holds its 128 output rows x
// 256 columns (two accumulators, so the epilogue of one tile overlaps the
// main loop of the next).  Per FLOP this moves 1.5x fewer operand bytes from
// L2 into shared memory than one CTA working a 128 x 256 tile alone.  Each
// pair walks work units (m-tile, n-tile, k-split) with a grid stride; m-tiles
// are visited in groups so that concurrently running pairs share tiles in L2.
//
// Warp roles (256 threads per CTA): warp 0 lane 0 issues TMA (both CTAs;
// completion is counted on the even CTA's barrier), warp 1 lane 0 of the
// even CTA issues tcgen05.mma, warp 2 owns the TMEM allocation, warps 4..7
// run the epilogue (warp 4 + i reads TMEM lanes 32i..32i+31, i.e. tile rows).
// The epilogue transforms one 128-byte-wide column chunk of its 128 rows at a
// time in registers, writes it to a 128B-swizzled staging buffer and lets one
// thread store the chunk with a TMA bulk store (or bulk reduce-add for the
// float32 residual / gradient accumulation), so global writes go out as
// whole lines; two staging buffers alternate.  Every wait is
// bounded: on timeout the CTA records DEV_TIMEOUT, its roles stop, in-flight
// work is drained (bounded) and TMEM is released before the pair exits.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "epilogue.cuh"
#include "nc_common.cuh"
#include "tc_common.cuh"

namespace nc {
namespace tc {

constexpr int BM = 256;              // output rows per CTA pair
constexpr int BN = 256;              // output columns
constexpr int BK = 64;
constexpr int HALF_ROWS = 128;       // rows of the A and of the B tile each CTA loads
constexpr int A_BYTES = HALF_ROWS * BK * 2;  // 16 KB
constexpr int B_BYTES = HALF_ROWS * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 256;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
// Epilogue staging: two 128-row x 128-byte chunks of the output tile, and
// for epilogues with an auxiliary operand (same layout as C) two more for
// its chunks, loaded by TMA ahead of use; those run a 5-stage operand ring.
// Head-pair epilogues use the same two extra chunks for their per-row table.
constexpr int STAGE_OUT_BYTES = HALF_ROWS * 128;  // 16 KB
template <bool kAux>
struct SmemPlan {
  static constexpr int kStages = kAux ? 5 : 6;
  static constexpr int OUT_OFF = kStages * STAGE_BYTES;
  static constexpr int AUX_OFF = OUT_OFF + 2 * STAGE_OUT_BYTES;
  static constexpr int BAR_OFF = AUX_OFF + (kAux ? 2 * STAGE_OUT_BYTES : 0);
  static constexpr int BYTES = BAR_OFF + 256 /*barriers*/ + 1024 /*align slack*/;
  static_assert(BYTES <= 232448, "GEMM shared memory exceeds 227 KB");
};
constexpr int STAGES_MAX = 6;
// Swizzle-128B atom: 8 rows of 128 bytes.  An MN-major operand half-tile is
// stored as 128/64 = 2 column blocks of 64 elements, each BK rows of 128 B.
constexpr int MN_BLOCK_BYTES = BK * 128;  // 8 KB

// Work units, batch outermost (the tiles of one batch entry run together and
// share its operands in L2), then k-split, then grouped (m, n) tiles.
struct Sched {
  int m_tiles, n_tiles, splits, k_blocks, kb_per_split, group_m, units, batches;

  // z: destination slab (batch * splits + split); batch: operand slice.
  __device__ __forceinline__ void decode(int u, int& mt, int& nt, int& z, int& batch, int& kb0,
                                         int& kb1) const {
    const int per_split = m_tiles * n_tiles;
    const int per_batch = per_split * splits;
    batch = u / per_batch;
    u -= batch * per_batch;
    const int split = u / per_split;
    z = batch * splits + split;
    const int r = u - split * per_split;
    const int group_size = group_m * n_tiles;
    const int group = r / group_size;
    const int first_m = group * group_m;
    const int gm = min(group_m, m_tiles - first_m);
    const int in = r - group * group_size;
    mt = first_m + in % gm;
    nt = in / gm;
    kb0 = split * kb_per_split;
    kb1 = min(k_blocks, kb0 + kb_per_split);
  }
};

// K-major tile (rows of 64 K-elements = 128 B, 8-row swizzle atoms 1 KB apart):
// LBO unused for swizzled K-major, SBO = 1 KB.  MMA step k (16 elements) starts
// 32 B further inside the atom.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int k) {
  return sdesc_sw128(tile + k * 32, 16, 1024);
}
// MN-major tile (column blocks of 64 MN-elements, BK rows of 128 B each):
// LBO = distance between 64-wide MN blocks, SBO = distance between 8-row
// K groups.  MMA step k covers K rows 16k..16k+15 = 2 K groups.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int k) {
  return sdesc_sw128(tile + k * 2048, MN_BLOCK_BYTES, 1024);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, M = 256 (pair), N = 256.
__host__ __device__ constexpr uint32_t idesc_bf16(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
// kind::f8f6f4 with both operands E4M3 (format code 0 in bits 7-9 and 10-12),
// both K-major, fp32 accumulator (bits 4-5 = 1).
__host__ __device__ constexpr uint32_t idesc_e4m3() {
  return (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
// One k-block is 128 bytes of every operand row: 64 bf16 or 128 E4M3 values.
template <bool kFp8>
__host__ __device__ constexpr int kblock_elems() { return kFp8 ? 128 : BK; }

// Epilogues that declare kAuxTma read a second operand with C's layout
// (ReLU^2 backward: the saved activation; AXPBY: the addend); the kernel
// brings its chunks in by TMA ahead of use and passes them to compute_aux.
template <class E, class = void>
struct HasAuxTma {
  static constexpr bool value = false;
};
template <class E>
struct HasAuxTma<E, std::void_t<decltype(E::kAuxTma)>> {
  static constexpr bool value = E::kAuxTma;
};
// Epilogues that declare kHeadPairs take two 64-column chunks of a row at a
// time (compute_head) and choose each chunk's destination map (dest).
template <class E, class = void>
struct HasHeadPairs {
  static constexpr bool value = false;
};
template <class E>
struct HasHeadPairs<E, std::void_t<decltype(E::kHeadPairs)>> {
  static constexpr bool value = E::kHeadPairs;
};

enum WaitSite : int {
  SITE_PROD_EMPTY = 101, SITE_MMA_ACC_EMPTY = 102, SITE_MMA_FULL = 103,
  SITE_EPI_ACC_FULL = 104, SITE_DRAIN = 105
};

// 128 bytes of one output row (W elements of Out) into row `r` of a
// [128 rows][128 B] staging chunk with the TMA 128-byte swizzle.
template <typename Out, int W>
__device__ __forceinline__ void stage_row(uint8_t* chunk, int r, const float (&v)[W]) {
  uint8_t* base = chunk + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint4 w;
    if constexpr (sizeof(Out) == 4) {
      w.x = __float_as_uint(v[q * 4 + 0]);
      w.y = __float_as_uint(v[q * 4 + 1]);
      w.z = __float_as_uint(v[q * 4 + 2]);
      w.w = __float_as_uint(v[q * 4 + 3]);
    } else {
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (std::is_same<Out, __half>::value) {
          const __half2 t = __floats2half2_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
          h[e] = *reinterpret_cast<const uint32_t*>(&t);
        } else {
          const __nv_bfloat162 t = __floats2bfloat162_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
          h[e] = *reinterpret_cast<const uint32_t*>(&t);
        }
      }
      w = make_uint4(h[0], h[1], h[2], h[3]);
    }
    *reinterpret_cast<uint4*>(base + ((q ^ (r & 7)) << 4)) = w;
  }
}

// Inverse of stage_row for a 16-bit type: the 64 values of row `r` of a
// 128B-swizzled [128 rows][128 B] chunk written by TMA.
template <typename T>
__device__ __forceinline__ void unstage_row(const uint8_t* chunk, int r, float (&a)[64]) {
  const uint8_t* base = chunk + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 w = *reinterpret_cast<const uint4*>(base + ((q ^ (r & 7)) << 4));
    const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
    for (int i = 0; i < 8; ++i) a[q * 8 + i] = to_f(e[i]);
  }
}

template <bool A_MN, bool B_MN, class Epi, bool kFp8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmAux, const Sched sch, const int M,
                        const int N, const __grid_constant__ Epi epi, int* err,
                        const long long timeout_ns) {
  static_assert(!kFp8 || (!A_MN && !B_MN), "8-bit operands are K-major");
  constexpr bool kAux = HasAuxTma<Epi>::value;
  constexpr bool kHeads = HasHeadPairs<Epi>::value;
  using Plan = SmemPlan<kAux || kHeads>;
  constexpr int STAGES = Plan::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Plan::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_ok = abort_flag + 1;  // [4]: the epilogue warps' accumulator waits
  uint64_t* aux_full = reinterpret_cast<uint64_t*>(smem + Plan::BAR_OFF + 192);  // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs, 1: its peer
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // used on the even CTA: both CTAs' bytes
      mbar_init(&empty[s], 1);  // one multicast commit per phase, in each CTA
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // used on the even CTA: 4 epilogue warps x 2 CTAs
    }
    mbar_init(drain, 1);
    mbar_init(&aux_full[0], 1);
    mbar_init(&aux_full[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (kAux || kHeads) tma_prefetch_desc(&tmAux);
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    int stage = 0;
    uint32_t phase = 0;
    int armed_phase[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) armed_phase[s] = -1;
    bool ok = true;
    for (int u = pair; u < sch.units && ok; u += npairs) {
      int mt, nt, split, batch, kb0, kb1;
      sch.decode(u, mt, nt, split, batch, kb0, kb1);
      const int row_a = mt * BM + (int)rank * HALF_ROWS;
      const int row_b = nt * BN + (int)rank * HALF_ROWS;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_flag, err, SITE_PROD_EMPTY,
                               timeout_ns)) {
          ok = false;
          break;
        }
        if (rank == 0) {
          mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          armed_phase[stage] = (int)phase;
        }
        const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
        uint8_t* a = sA + stage * A_BYTES;
        uint8_t* b = sB + stage * B_BYTES;
        const int k0 = kb * kblock_elems<kFp8>();
        if (!A_MN) {
          tma_load_3d_pair(a, &tmA, bar, k0, row_a, batch);
        } else {
#pragma unroll
          for (int j = 0; j < HALF_ROWS / 64; ++j)
            tma_load_3d_pair(a + j * MN_BLOCK_BYTES, &tmA, bar, row_a + 64 * j, k0, batch);
        }
        if (!B_MN) {
          tma_load_3d_pair(b, &tmB, bar, k0, row_b, batch);
        } else {
#pragma unroll
          for (int j = 0; j < HALF_ROWS / 64; ++j)
            tma_load_3d_pair(b + j * MN_BLOCK_BYTES, &tmB, bar, row_b + 64 * j, k0, batch);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if ((!ok || *abort_flag) && rank == 0) {
      // Drain: the copies of both CTAs that this barrier counted land before
      // the pair exits.  (The peer's own waits give up only after the limit,
      // long after any copy it issued has landed.)
      int dummy_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if (armed_phase[s] >= 0)
          mbar_wait_cluster(&full[s], (uint32_t)armed_phase[s], &dummy_abort, err, SITE_DRAIN,
                            timeout_ns / 8);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (even CTA) ----------------
    constexpr uint32_t idesc = kFp8 ? idesc_e4m3() : idesc_bf16(A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true, issued = false;
    for (int u = pair; u < sch.units && ok; u += npairs) {
      int mt, nt, split, batch, kb0, kb1;
      sch.decode(u, mt, nt, split, batch, kb0, kb1);
      if (!mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1u, abort_flag, err,
                             SITE_MMA_ACC_EMPTY, timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_cluster(&full[stage], phase, abort_flag, err, SITE_MMA_FULL,
                               timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
        const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t ad = A_MN ? desc_mnmajor(a_addr, k) : desc_kmajor(a_addr, k);
          const uint64_t bd = B_MN ? desc_mnmajor(b_addr, k) : desc_kmajor(b_addr, k);
          if constexpr (kFp8)  // K = 32 E4M3 values: the same 32 bytes per step
            umma_f8_pair(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          else
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        }
        issued = true;
        umma_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit_pair(&acc_full[acc], 0x3);  // both halves of the tile are ready
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if ((!ok || *abort_flag) && issued) {
      // Drain: wait until every MMA issued so far has completed.
      int dummy_abort = 0;
      umma_commit_pair(drain, 0x1);
      mbar_wait_cluster(drain, 0, &dummy_abort, err, SITE_DRAIN, timeout_ns / 8);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs, 128 rows each) ----------------
    using Out = typename Epi::Out;
    constexpr int W = 128 / (int)sizeof(Out);  // columns per staging chunk
    constexpr int NCH = BN / W;
    const int quarter = warp & 3;
    const bool issuer = warp == 4 && lane == 0;
    const uint32_t acc_empty_leader0 = mapa_shared(smem_u32(&acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = mapa_shared(smem_u32(&acc_empty[1]), 0);
    const bool reduce = epi.reduce();
    int acc = 0, chunk_no = 0;
    int aux_no = 0;                   // auxiliary chunks consumed so far
    uint32_t aux_uses[2] = {0, 0};    // loads consumed per auxiliary buffer
    uint32_t aux_issued[2] = {0, 0};  // loads issued per auxiliary buffer (issuer)
    uint32_t acc_phase = 0;
    uint32_t tab_loads = 0;           // head pairs: table loads waited for so far
    for (int u = pair; u < sch.units; u += npairs) {
      int mt, nt, split, batch, kb0, kb1;
      sch.decode(u, mt, nt, split, batch, kb0, kb1);
      const int r_in = quarter * 32 + lane;
      const int row0 = mt * BM + (int)rank * HALF_ROWS;
      const int row = row0 + r_in;
      // Chunks of this tile that lie inside C (a prefix of the NCH chunks).
      const int nvalid = row0 >= M ? 0 : min(NCH, (N - nt * BN + W - 1) / W);
      const int aux_base = aux_no;    // chunk c of this tile uses buffer (aux_base + c) & 1
      auto issue_aux = [&](int c) {
        const int bsel = (aux_base + c) & 1;
        ++aux_issued[bsel];
        mbar_arrive_expect_tx(&aux_full[bsel], STAGE_OUT_BYTES);
        tma_load_3d(smem + Plan::AUX_OFF + bsel * STAGE_OUT_BYTES, &tmAux, &aux_full[bsel],
                    nt * BN + c * W, row0, batch);
      };
      if constexpr (kAux) {
        // The first two auxiliary chunks load while the tile still accumulates.
        if (issuer)
          for (int c = 0; c < min(2, nvalid); ++c) issue_aux(c);
      }
      if constexpr (kHeads) {
        // The half tile's 128 table rows, while the tile still accumulates.
        // Every thread finished reading the previous unit's rows before the
        // named barrier that preceded its first staged chunk; tiles without
        // a head (nvalid == 0) neither load nor wait.
        if (issuer && nvalid > 0) {
          ++aux_issued[0];
          mbar_arrive_expect_tx(&aux_full[0], 2 * STAGE_OUT_BYTES);
          const int t0 = row0 % epi.T;
          tma_load_3d(smem + Plan::AUX_OFF, &tmAux, &aux_full[0], 0, t0, 0);
          tma_load_3d(smem + Plan::AUX_OFF + STAGE_OUT_BYTES, &tmAux, &aux_full[0], 64, t0, 0);
        }
      }
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_cluster(&acc_full[acc], acc_phase, abort_flag, err, SITE_EPI_ACC_FULL,
                               timeout_ns);
      // The four warps leave together or not at all (they meet at named
      // barriers below).
      if (lane == 0) epi_ok[quarter] = ok;
      named_bar_sync<128>();
      ok = epi_ok[0] & epi_ok[1] & epi_ok[2] & epi_ok[3];
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      float row_acc = 0.f;
      if constexpr (HasHeadPairs<Epi>::value) {
        // One head (two 64-column chunks) at a time; each chunk is staged and
        // stored like any other, to the destination the epilogue names.
        static_assert(W == 64 && !kAux, "head pairs are 64-column bf16 chunks");
        int tok = 1;
        if (nvalid > 0) {
          if (lane == 0)
            tok = mbar_wait_bounded(&aux_full[0], tab_loads & 1u, abort_flag, err,
                                    SITE_EPI_ACC_FULL, timeout_ns);
          tok = __shfl_sync(0xffffffffu, tok, 0);
          if (tok) mbar_try_wait(smem_u32(&aux_full[0]), tab_loads & 1u);  // acquire in every lane
          ++tab_loads;
        }
#pragma unroll 1
        for (int c = 0; c + 1 < nvalid; c += 2) {
          const int col = nt * BN + c * W;
          float v0[64], v1[64];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_ld_32cols(taddr + c * W + h * 32, *reinterpret_cast<float(*)[32]>(v0 + h * 32));
            tmem_ld_32cols(taddr + (c + 1) * W + h * 32,
                           *reinterpret_cast<float(*)[32]>(v1 + h * 32));
          }
          if (row < M && tok)
            epi.compute_head(row, col >> 7, v0, v1, smem + Plan::AUX_OFF, r_in);
#pragma unroll 1
          for (int q2 = 0; q2 < 2; ++q2) {
            uint8_t* chunk = smem + Plan::OUT_OFF + (chunk_no & 1) * STAGE_OUT_BYTES;
            ++chunk_no;
            if (issuer) bulk_wait_group_read<1>();  // the store issued from this buffer is done reading
            named_bar_sync<128>();
            if (q2 == 0)
              stage_row<Out, W>(chunk, r_in, v0);
            else
              stage_row<Out, W>(chunk, r_in, v1);
            fence_proxy_async_smem();
            named_bar_sync<128>();
            if (issuer) {
              int x = 0;
              const CUtensorMap* dmap = epi.dest(col + q2 * W, x);
              tma_store_3d(dmap, chunk, x, row0, 0);
              bulk_commit_group();
            }
          }
        }
      } else {
#pragma unroll 1
      for (int c = 0; c < nvalid; ++c) {
        const int col = nt * BN + c * W;
        float v[W];
#pragma unroll
        for (int h = 0; h < W / 32; ++h)
          tmem_ld_32cols(taddr + c * W + h * 32, *reinterpret_cast<float(*)[32]>(v + h * 32));
        if constexpr (kAux) {
          const int bsel = aux_no & 1;
          int aok = 1;
          if (lane == 0)
            aok = mbar_wait_bounded(&aux_full[bsel], aux_uses[bsel] & 1u, abort_flag, err,
                                    SITE_EPI_ACC_FULL, timeout_ns);
          aok = __shfl_sync(0xffffffffu, aok, 0);
          if (aok) {
            mbar_try_wait(smem_u32(&aux_full[bsel]), aux_uses[bsel] & 1u);  // acquire in every lane
            float av[64];
            unstage_row<Out>(smem + Plan::AUX_OFF + bsel * STAGE_OUT_BYTES, r_in, av);
            if (row < M) row_acc += epi.template compute_aux<W>(row, col, v, batch, av);
          }
          ++aux_uses[bsel];
          ++aux_no;
        } else {
          if (row < M) row_acc += epi.template compute<W>(row, col, v, batch);
        }
        uint8_t* chunk = smem + Plan::OUT_OFF + (chunk_no & 1) * STAGE_OUT_BYTES;
        ++chunk_no;
        if (issuer) bulk_wait_group_read<1>();  // the store issued from this buffer is done reading
        named_bar_sync<128>();
        stage_row<Out, W>(chunk, r_in, v);
        fence_proxy_async_smem();
        named_bar_sync<128>();
        if (issuer) {
          if (reduce)
            tma_reduce_add_3d(&tmC, chunk, col, row0, split);
          else
            tma_store_3d(&tmC, chunk, col, row0, split);
          bulk_commit_group();
          // Every thread is past its read of this chunk's auxiliary buffer:
          // refill it with chunk c + 2.
          if constexpr (kAux) {
            if (c + 2 < nvalid) issue_aux(c + 2);
          }
        }
      }
      }
      if (Epi::kRowReduce && row < M) epi.row_end(row, nt * BN, row_acc);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? acc_empty_leader1 : acc_empty_leader0);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (issuer) {
      bulk_wait_group_all();
      // After an abort: let auxiliary loads already issued land before exit.
      if constexpr (kHeads) {
        int none = 0;
        for (; tab_loads < aux_issued[0]; ++tab_loads)
          mbar_wait_bounded(&aux_full[0], tab_loads & 1u, &none, err, SITE_DRAIN,
                            timeout_ns / 8);
      }
      if constexpr (kAux) {
        int none = 0;
        for (int b2 = 0; b2 < 2; ++b2)
          for (; aux_uses[b2] < aux_issued[b2]; ++aux_uses[b2])
            mbar_wait_bounded(&aux_full[b2], aux_uses[b2] & 1u, &none, err, SITE_DRAIN,
                              timeout_ns / 8);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still touch it
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace tc
}  // namespace nc
