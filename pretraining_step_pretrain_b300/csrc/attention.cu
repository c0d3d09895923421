// Causal multi-query attention, forward and backward (launch article,
// architecture list: multi-query attention -- H query heads share one K/V
// head; causal because the objective is next-token prediction).
//
//   o_h[i] = sum_{j<=i} softmax_j(q_h[i] . k[j] / sqrt(h)) v[j]
//
// Query rows of one sequence are packed as r = t * H + head (the natural
// (B, T, H, h) layout of q), so one (T*H) x h matrix faces the single
// T x h K and V: every K/V tile brought on chip serves all H heads, and the
// causal rule becomes "key j is visible to packed row r iff j <= r / H".
//
// bf16 path (h = 128): flash-style tiles on mma.sync m16n8k16 (fp32
// accumulation) with an online softmax; the backward recomputes P from the
// saved log-sum-exp and runs two passes -- a Q-major pass for dQ (which also
// writes delta = rowsum(dO * O)) and a KV-major pass for dK, dV that sums
// over every packed row, hence over all heads, without atomics.
// fp32 path (debug mode, h in {64, 128}): one warp per row, plain loops.
#include <algorithm>
#include <mutex>

#include "nc_common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ===================================================================
// fp32 SIMT kernels
// ===================================================================
template <int E>  // elements per lane, h = 32 E
__global__ void attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                    const float* __restrict__ v, float* __restrict__ o,
                                    float* __restrict__ lse, int B, int T, int H) {
  constexpr int h = 32 * E;
  const long row = blockIdx.x * 4L + (threadIdx.x >> 5);  // global packed row over (B, T, H)
  const int lane = threadIdx.x & 31;
  if (row >= (long)B * T * H) return;
  const int b = (int)(row / ((long)T * H));
  const int t = (int)((row / H) % T);
  const float scale = rsqrtf((float)h);
  float qv[E], acc[E];
  for (int e = 0; e < E; ++e) {
    qv[e] = q[row * h + lane * E + e];
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j <= t; ++j) {
    const float* kr = k + ((long)b * T + j) * h + lane * E;
    float s = 0.f;
    for (int e = 0; e < E; ++e) s += qv[e] * kr[e];
    s = warp_sum(s) * scale;
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn), p = expf(s - mn);
    l = l * corr + p;
    const float* vr = v + ((long)b * T + j) * h + lane * E;
    for (int e = 0; e < E; ++e) acc[e] = acc[e] * corr + p * vr[e];
    m = mn;
  }
  for (int e = 0; e < E; ++e) o[row * h + lane * E + e] = acc[e] / l;
  if (lane == 0) lse[row] = m + logf(l);
}

// dq for one packed row; also writes delta = rowsum(dO * O).
template <int E>
__global__ void attn_bwd_dq_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                       const float* __restrict__ v, const float* __restrict__ o,
                                       const float* __restrict__ lse,
                                       const float* __restrict__ dout, float* __restrict__ dq,
                                       long ldq, float* __restrict__ delta, int B, int T, int H) {
  constexpr int h = 32 * E;
  const long row = blockIdx.x * 4L + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long)B * T * H) return;
  const int b = (int)(row / ((long)T * H));
  const int t = (int)((row / H) % T);
  const int head = (int)(row % H);
  const float scale = rsqrtf((float)h);
  float qv[E], dov[E], acc[E];
  float dl = 0.f;
  for (int e = 0; e < E; ++e) {
    qv[e] = q[row * h + lane * E + e];
    dov[e] = dout[row * h + lane * E + e];
    dl += dov[e] * o[row * h + lane * E + e];
    acc[e] = 0.f;
  }
  dl = warp_sum(dl);
  const float L = lse[row];
  for (int j = 0; j <= t; ++j) {
    const float* kr = k + ((long)b * T + j) * h + lane * E;
    const float* vr = v + ((long)b * T + j) * h + lane * E;
    float s = 0.f, dp = 0.f;
    for (int e = 0; e < E; ++e) {
      s += qv[e] * kr[e];
      dp += dov[e] * vr[e];
    }
    s = warp_sum(s) * scale;
    dp = warp_sum(dp);
    const float p = expf(s - L);
    const float ds = p * (dp - dl);
    for (int e = 0; e < E; ++e) acc[e] += ds * kr[e];
  }
  const long tok = (long)b * T + t;
  for (int e = 0; e < E; ++e) dq[tok * ldq + (long)head * h + lane * E + e] = acc[e] * scale;
  if (lane == 0) delta[row] = dl;
}

// dk, dv for one key: sums over every packed row r with r / H >= j.
template <int E>
__global__ void attn_bwd_dkdv_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                         const float* __restrict__ v,
                                         const float* __restrict__ lse,
                                         const float* __restrict__ dout,
                                         const float* __restrict__ delta, float* __restrict__ dk,
                                         long ldk, float* __restrict__ dv, long ldv, int B, int T,
                                         int H) {
  constexpr int h = 32 * E;
  const long key = blockIdx.x * 4L + (threadIdx.x >> 5);  // over (B, T)
  const int lane = threadIdx.x & 31;
  if (key >= (long)B * T) return;
  const int b = (int)(key / T), j = (int)(key % T);
  const float scale = rsqrtf((float)h);
  float kv[E], vv[E], adk[E], adv[E];
  for (int e = 0; e < E; ++e) {
    kv[e] = k[key * h + lane * E + e];
    vv[e] = v[key * h + lane * E + e];
    adk[e] = adv[e] = 0.f;
  }
  const long rbase = (long)b * T * H;
  for (long r = (long)j * H; r < (long)T * H; ++r) {
    const float* qr = q + (rbase + r) * h + lane * E;
    const float* dr = dout + (rbase + r) * h + lane * E;
    float s = 0.f, dp = 0.f;
    for (int e = 0; e < E; ++e) {
      s += qr[e] * kv[e];
      dp += dr[e] * vv[e];
    }
    s = warp_sum(s) * scale;
    dp = warp_sum(dp);
    const float p = expf(s - lse[rbase + r]);
    const float ds = p * (dp - delta[rbase + r]);
    for (int e = 0; e < E; ++e) {
      adv[e] += p * dr[e];
      adk[e] += ds * qr[e];
    }
  }
  for (int e = 0; e < E; ++e) {
    dk[key * ldk + lane * E + e] = adk[e] * scale;
    dv[key * ldv + lane * E + e] = adv[e];
  }
}

// ===================================================================
// bf16 mma.sync kernels (h = 128)
// ===================================================================
constexpr int HD = 128;       // head dim
constexpr int TILE = 64;      // packed rows / keys per tile
constexpr int TILE_BYTES = TILE * HD * 2;  // 16 KB

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// [64][128] bf16 tile, 256-byte rows, 16-byte chunks XOR-swizzled by row % 8.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}

// Rows [row0, row0 + 64) of a row-major bf16 matrix (row stride ld); rows at
// or beyond `limit` are zero-filled and not read.
__device__ __forceinline__ void load_tile(uint32_t sbase, const bf16* g, long ld, long row0,
                                          long limit, int tid, int nthreads) {
  for (int i = tid; i < TILE * 16; i += nthreads) {
    const int r = i >> 4, ch = i & 15;
    const long gr = row0 + r;
    const bool ok = gr < limit;
    cp_async16(sbase + swz(r, ch), g + (ok ? gr : 0) * ld + ch * 8, ok);
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Fragment addresses (lane i) inside a swizzled tile:
//  A operand, 16 x 16 block at (row r0, col k0), row-major source:
__device__ __forceinline__ uint32_t addr_a(uint32_t base, int r0, int k0, int lane) {
  return base + swz(r0 + (lane & 7) + ((lane >> 3) & 1) * 8, (k0 >> 3) + (lane >> 4));
}
//  B operand for X . Y^T with Y row-major [n][k]: n-tiles n0 and n0 + 8, k chunk k0.
__device__ __forceinline__ uint32_t addr_bt(uint32_t base, int n0, int k0, int lane) {
  return base + swz(n0 + (lane & 7) + (lane >> 4) * 8, (k0 >> 3) + ((lane >> 3) & 1));
}
//  B operand for X . Y with Y row-major [k][n] (ldmatrix.trans): k chunk k0,
//  n-tiles n0 and n0 + 8.
__device__ __forceinline__ uint32_t addr_bn(uint32_t base, int k0, int n0, int lane) {
  return base + swz(k0 + (lane & 7) + ((lane >> 3) & 1) * 8, (n0 >> 3) + (lane >> 4));
}

// ---------------- forward ----------------
// grid (ceil(T*H / 64), B), 128 threads; warp w owns packed rows r0 + 16w..+15.
__global__ void __launch_bounds__(128) attn_fwd_bf16_kernel(const bf16* __restrict__ q,
                                                            const bf16* __restrict__ k,
                                                            const bf16* __restrict__ v,
                                                            bf16* __restrict__ o,
                                                            float* __restrict__ lse, int T, int H) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + TILE_BYTES;  // K[2], V[2] follow
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.y;
  const long TH = (long)T * H;
  const int n_qtiles = (int)((TH + TILE - 1) / TILE);
  const long r0 = (long)(n_qtiles - 1 - blockIdx.x) * TILE;  // heaviest tiles first
  const bf16* qb = q + (long)b * TH * HD;
  const bf16* kb = k + (long)b * T * HD;
  const bf16* vb = v + (long)b * T * HD;

  const long r_last = min(r0 + TILE - 1, TH - 1);
  const int t_max = (int)(r_last / H);
  const int t_min = (int)(r0 / H);
  const int n_kv = t_max / TILE + 1;

  load_tile(sQ, qb, HD, r0, TH, tid, 128);
  load_tile(sK0, kb, HD, 0, T, tid, 128);
  load_tile(sK0 + 2 * TILE_BYTES, vb, HD, 0, T, tid, 128);
  cp_async_commit();

  const float sl2 = rsqrtf((float)HD) * kLog2e;  // scale in log2 units
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const long my_r[2] = {r0 + warp * 16 + g, r0 + warp * 16 + g + 8};
  const int my_t[2] = {(int)(my_r[0] / H), (int)(my_r[1] / H)};
  uint32_t qf[8][4];

  for (int it = 0; it < n_kv; ++it) {
    const int buf = it & 1;
    if (it + 1 < n_kv) {
      const uint32_t nk = sK0 + (buf ^ 1) * TILE_BYTES;
      load_tile(nk, kb, HD, (long)(it + 1) * TILE, T, tid, 128);
      load_tile(nk + 2 * TILE_BYTES, vb, HD, (long)(it + 1) * TILE, T, tid, 128);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) ldsm_x4(qf[kk], addr_a(sQ, warp * 16, kk * 16, lane));
    }
    const uint32_t sK = sK0 + buf * TILE_BYTES;
    const uint32_t sV = sK + 2 * TILE_BYTES;
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        uint32_t bf[4];
        ldsm_x4(bf, addr_bt(sK, jp * 16, kk * 16, lane));
        mma16816(s[2 * jp], qf[kk], bf[0], bf[1]);
        mma16816(s[2 * jp + 1], qf[kk], bf[2], bf[3]);
      }
    }
    const int key0 = it * TILE;
    const bool need_mask = key0 + TILE - 1 > t_min || key0 + TILE > T;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const int key = key0 + j * 8 + 2 * c + (e & 1);
        float x = s[j][e] * sl2;
        if (need_mask && (key > my_t[hr] || key >= T)) x = -INFINITY;
        s[j][e] = x;
        mx[hr] = fmaxf(mx[hr], x);
      }
    }
    float corr[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float m_new = fmaxf(m_run[hr], mx[hr]);
      corr[hr] = (m_run[hr] == -INFINITY) ? 0.f : exp2f(m_run[hr] - m_new);
      m_run[hr] = m_new;
    }
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const float p = (s[j][e] == -INFINITY) ? 0.f : exp2f(s[j][e] - m_run[hr]);
        s[j][e] = p;
        ls[hr] += p;
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) l_run[hr] = l_run[hr] * corr[hr] + ls[hr];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc[i][0] *= corr[0]; acc[i][1] *= corr[0];
      acc[i][2] *= corr[1]; acc[i][3] *= corr[1];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t bf[4];
        ldsm_x4_t(bf, addr_bn(sV, kk * 16, dp * 16, lane));
        mma16816(acc[2 * dp], pa, bf[0], bf[1]);
        mma16816(acc[2 * dp + 1], pa, bf[2], bf[3]);
      }
    }
    __syncthreads();  // buffer `buf` is refilled at the next iteration
  }

#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const long r = my_r[hr];
    if (r >= TH) continue;
    const float inv = 1.f / l_run[hr];
    bf16* orow = o + ((long)b * TH + r) * HD;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t pk = pack_bf16(acc[i][2 * hr] * inv, acc[i][2 * hr + 1] * inv);
      *reinterpret_cast<uint32_t*>(orow + i * 8 + 2 * c) = pk;
    }
    if (c == 0) lse[(long)b * TH + r] = (m_run[hr] + log2f(l_run[hr])) * kLn2;
  }
}

// ---------------- backward: dQ (+ delta) ----------------
// grid (ceil(T*H / 64), B), 128 threads.  smem: Q, dO, K[2], V[2].
__global__ void __launch_bounds__(128) attn_bwd_dq_bf16_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
    const bf16* __restrict__ o, const float* __restrict__ lse, const bf16* __restrict__ dout,
    bf16* __restrict__ dq, long ldq, float* __restrict__ delta, int T, int H) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sdO = sQ + TILE_BYTES;
  const uint32_t sK0 = sdO + TILE_BYTES;  // K[2] then V[2]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.y;
  const long TH = (long)T * H;
  const int n_qtiles = (int)((TH + TILE - 1) / TILE);
  const long r0 = (long)(n_qtiles - 1 - blockIdx.x) * TILE;
  const bf16* qb = q + (long)b * TH * HD;
  const bf16* ob = o + (long)b * TH * HD;
  const bf16* dob = dout + (long)b * TH * HD;
  const bf16* kb = k + (long)b * T * HD;
  const bf16* vb = v + (long)b * T * HD;
  const long r_last = min(r0 + TILE - 1, TH - 1);
  const int t_max = (int)(r_last / H), t_min = (int)(r0 / H);
  const int n_kv = t_max / TILE + 1;

  load_tile(sQ, qb, HD, r0, TH, tid, 128);
  load_tile(sdO, dob, HD, r0, TH, tid, 128);
  load_tile(sK0, kb, HD, 0, T, tid, 128);
  load_tile(sK0 + 2 * TILE_BYTES, vb, HD, 0, T, tid, 128);
  cp_async_commit();

  // delta for this warp's 16 rows: lane pairs (2 lanes per row, 64 dims each)
  __shared__ float s_delta[TILE];
  {
    const int rr = lane >> 1, half = lane & 1;
    const long r = r0 + warp * 16 + rr;
    float dsum = 0.f;
    if (r < TH) {
      const bf16* orow = ob + r * HD + half * 64;
      const bf16* drow = dob + r * HD + half * 64;
      for (int i = 0; i < 64; i += 4) {
        float a[4], bb[4];
        Vec4<bf16>::load(orow + i, a);
        Vec4<bf16>::load(drow + i, bb);
        dsum += a[0] * bb[0] + a[1] * bb[1] + a[2] * bb[2] + a[3] * bb[3];
      }
    }
    dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
    if (half == 0) {
      s_delta[warp * 16 + rr] = dsum;
      if (r < TH) delta[(long)b * TH + r] = dsum;
    }
  }
  __syncwarp();
  const float sl2 = rsqrtf((float)HD) * kLog2e;
  const long my_r[2] = {r0 + warp * 16 + g, r0 + warp * 16 + g + 8};
  const int my_t[2] = {(int)(my_r[0] / H), (int)(my_r[1] / H)};
  float lse2[2], dl[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lse2[hr] = my_r[hr] < TH ? lse[(long)b * TH + my_r[hr]] * kLog2e : 0.f;
    dl[hr] = s_delta[warp * 16 + g + 8 * hr];
  }
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  for (int it = 0; it < n_kv; ++it) {
    const int buf = it & 1;
    if (it + 1 < n_kv) {
      const uint32_t nk = sK0 + (buf ^ 1) * TILE_BYTES;
      load_tile(nk, kb, HD, (long)(it + 1) * TILE, T, tid, 128);
      load_tile(nk + 2 * TILE_BYTES, vb, HD, (long)(it + 1) * TILE, T, tid, 128);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sK = sK0 + buf * TILE_BYTES;
    const uint32_t sV = sK + 2 * TILE_BYTES;
    float s[8][4], dp[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = dp[j][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t qa[4], da[4];
      ldsm_x4(qa, addr_a(sQ, warp * 16, kk * 16, lane));
      ldsm_x4(da, addr_a(sdO, warp * 16, kk * 16, lane));
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        uint32_t kf[4], vf[4];
        ldsm_x4(kf, addr_bt(sK, jp * 16, kk * 16, lane));
        ldsm_x4(vf, addr_bt(sV, jp * 16, kk * 16, lane));
        mma16816(s[2 * jp], qa, kf[0], kf[1]);
        mma16816(s[2 * jp + 1], qa, kf[2], kf[3]);
        mma16816(dp[2 * jp], da, vf[0], vf[1]);
        mma16816(dp[2 * jp + 1], da, vf[2], vf[3]);
      }
    }
    const int key0 = it * TILE;
    const bool need_mask = key0 + TILE - 1 > t_min || key0 + TILE > T;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const int key = key0 + j * 8 + 2 * c + (e & 1);
        float p = exp2f(s[j][e] * sl2 - lse2[hr]);
        if ((need_mask && (key > my_t[hr] || key >= T)) || my_r[hr] >= TH) p = 0.f;
        s[j][e] = p * (dp[j][e] - dl[hr]);  // dS
      }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp2 = 0; dp2 < 8; ++dp2) {
        uint32_t bf[4];
        ldsm_x4_t(bf, addr_bn(sK, kk * 16, dp2 * 16, lane));
        mma16816(acc[2 * dp2], pa, bf[0], bf[1]);
        mma16816(acc[2 * dp2 + 1], pa, bf[2], bf[3]);
      }
    }
    __syncthreads();
  }
  const float scale = rsqrtf((float)HD);
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const long r = my_r[hr];
    if (r >= TH) continue;
    const long tok = (long)b * T + r / H;
    const int head = (int)(r % H);
    bf16* row = dq + tok * ldq + (long)head * HD;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      *reinterpret_cast<uint32_t*>(row + i * 8 + 2 * c) =
          pack_bf16(acc[i][2 * hr] * scale, acc[i][2 * hr + 1] * scale);
  }
}

// ---------------- backward: dK, dV ----------------
// grid (ceil(T / 64), B), 128 threads; warp w owns keys j0 + 16w..+15 and walks
// every packed row r >= j0 * H in sub-tiles of 32 rows.
// smem: K, V, then Q[2], dO[2] (64-row tiles), lse2[2][64], delta[2][64].
__global__ void __launch_bounds__(128) attn_bwd_dkdv_bf16_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
    const float* __restrict__ lse, const bf16* __restrict__ dout, const float* __restrict__ delta,
    bf16* __restrict__ dk, long ldk, bf16* __restrict__ dv, long ldv, int T, int H) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + TILE_BYTES;
  const uint32_t sQ0 = sV + TILE_BYTES;    // Q[2]
  const uint32_t sD0 = sQ0 + 2 * TILE_BYTES;  // dO[2]
  float* s_lse = reinterpret_cast<float*>(smem + 6 * TILE_BYTES);  // [2][64]
  float* s_dl = s_lse + 2 * TILE;                                  // [2][64]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.y;
  const int j0 = blockIdx.x * TILE;
  const long TH = (long)T * H;
  const bf16* qb = q + (long)b * TH * HD;
  const bf16* dob = dout + (long)b * TH * HD;
  const float* lseb = lse + (long)b * TH;
  const float* dlb = delta + (long)b * TH;
  const long rt0 = ((long)j0 * H) / TILE;  // first packed-row tile
  const long n_rt = (TH + TILE - 1) / TILE - rt0;

  load_tile(sK, k + (long)b * T * HD, HD, j0, T, tid, 128);
  load_tile(sV, v + (long)b * T * HD, HD, j0, T, tid, 128);
  auto load_rows = [&](long rt, int buf) {
    const long r0 = rt * TILE;
    load_tile(sQ0 + buf * TILE_BYTES, qb, HD, r0, TH, tid, 128);
    load_tile(sD0 + buf * TILE_BYTES, dob, HD, r0, TH, tid, 128);
    if (tid < TILE) {
      const long r = r0 + tid;
      s_lse[buf * TILE + tid] = r < TH ? lseb[r] * kLog2e : 0.f;
      s_dl[buf * TILE + tid] = r < TH ? dlb[r] : 0.f;
    }
  };
  load_rows(rt0, 0);
  cp_async_commit();

  const float sl2 = rsqrtf((float)HD) * kLog2e;
  const int my_key[2] = {j0 + warp * 16 + g, j0 + warp * 16 + g + 8};
  float adk[16][4], adv[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) adk[i][e] = adv[i][e] = 0.f;

  for (long it = 0; it < n_rt; ++it) {
    const int buf = (int)(it & 1);
    if (it + 1 < n_rt) {
      load_rows(rt0 + it + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sQ = sQ0 + buf * TILE_BYTES;
    const uint32_t sD = sD0 + buf * TILE_BYTES;
    const long r_tile = (rt0 + it) * TILE;
#pragma unroll 1
    for (int sub = 0; sub < 2; ++sub) {
      const int rs = sub * 32;  // row offset inside the 64-row tile
      float st[4][4], dpt[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[j][e] = dpt[j][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t ka[4], va[4];
        ldsm_x4(ka, addr_a(sK, warp * 16, kk * 16, lane));
        ldsm_x4(va, addr_a(sV, warp * 16, kk * 16, lane));
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          uint32_t qf[4], df[4];
          ldsm_x4(qf, addr_bt(sQ, rs + jp * 16, kk * 16, lane));
          ldsm_x4(df, addr_bt(sD, rs + jp * 16, kk * 16, lane));
          mma16816(st[2 * jp], ka, qf[0], qf[1]);
          mma16816(st[2 * jp + 1], ka, qf[2], qf[3]);
          mma16816(dpt[2 * jp], va, df[0], df[1]);
          mma16816(dpt[2 * jp + 1], va, df[2], df[3]);
        }
      }
      // P^T and dS^T (rows = keys, cols = packed rows)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kr = e >> 1;
          const int lr = rs + j * 8 + 2 * c + (e & 1);  // row inside the tile
          const long r = r_tile + lr;
          const int key = my_key[kr];
          float p = exp2f(st[j][e] * sl2 - s_lse[buf * TILE + lr]);
          if (r >= TH || key >= T || (long)key > r / H) p = 0.f;
          st[j][e] = p;
          dpt[j][e] = p * (dpt[j][e] - s_dl[buf * TILE + lr]);
        }
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t pa[4], sa[4];
        pa[0] = pack_bf16(st[2 * kk][0], st[2 * kk][1]);
        pa[1] = pack_bf16(st[2 * kk][2], st[2 * kk][3]);
        pa[2] = pack_bf16(st[2 * kk + 1][0], st[2 * kk + 1][1]);
        pa[3] = pack_bf16(st[2 * kk + 1][2], st[2 * kk + 1][3]);
        sa[0] = pack_bf16(dpt[2 * kk][0], dpt[2 * kk][1]);
        sa[1] = pack_bf16(dpt[2 * kk][2], dpt[2 * kk][3]);
        sa[2] = pack_bf16(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
        sa[3] = pack_bf16(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
        for (int dp2 = 0; dp2 < 8; ++dp2) {
          uint32_t df[4], qf[4];
          ldsm_x4_t(df, addr_bn(sD, rs + kk * 16, dp2 * 16, lane));
          ldsm_x4_t(qf, addr_bn(sQ, rs + kk * 16, dp2 * 16, lane));
          mma16816(adv[2 * dp2], pa, df[0], df[1]);
          mma16816(adv[2 * dp2 + 1], pa, df[2], df[3]);
          mma16816(adk[2 * dp2], sa, qf[0], qf[1]);
          mma16816(adk[2 * dp2 + 1], sa, qf[2], qf[3]);
        }
      }
    }
    __syncthreads();
  }
  const float scale = rsqrtf((float)HD);
#pragma unroll
  for (int kr = 0; kr < 2; ++kr) {
    const int key = my_key[kr];
    if (key >= T) continue;
    const long tok = (long)b * T + key;
    bf16* krow = dk + tok * ldk;
    bf16* vrow = dv + tok * ldv;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      *reinterpret_cast<uint32_t*>(krow + i * 8 + 2 * c) =
          pack_bf16(adk[i][2 * kr] * scale, adk[i][2 * kr + 1] * scale);
      *reinterpret_cast<uint32_t*>(vrow + i * 8 + 2 * c) =
          pack_bf16(adv[i][2 * kr], adv[i][2 * kr + 1]);
    }
  }
}

constexpr int kFwdSmem = 5 * TILE_BYTES;                       // Q, K[2], V[2]
constexpr int kDqSmem = 6 * TILE_BYTES;                        // Q, dO, K[2], V[2]
constexpr int kDkdvSmem = 6 * TILE_BYTES + 4 * TILE * 4;       // K, V, Q[2], dO[2], lse, delta

}  // namespace

size_t attention_scratch_bytes(int B, int T, int H) { return (size_t)B * T * H * 4 + 256; }

cudaError_t attention_fwd(bool bf16, int B, int T, int H, int h, const void* q, const void* k,
                          const void* v, void* o, float* lse, const Ctx& ctx) {
  if (!bf16) {
    const long rows = (long)B * T * H;
    const int blocks = (int)((rows + 3) / 4);
    if (h == 128)
      attn_fwd_f32_kernel<4><<<blocks, 128, 0, ctx.stream>>>(
          (const float*)q, (const float*)k, (const float*)v, (float*)o, lse, B, T, H);
    else
      attn_fwd_f32_kernel<2><<<blocks, 128, 0, ctx.stream>>>(
          (const float*)q, (const float*)k, (const float*)v, (float*)o, lse, B, T, H);
    return launched(1);
  }
  if (h != HD) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((unsigned)(((long)T * H + TILE - 1) / TILE), B);
  attn_fwd_bf16_kernel<<<grid, 128, kFwdSmem, ctx.stream>>>(
      (const nc::bf16*)q, (const nc::bf16*)k, (const nc::bf16*)v, (nc::bf16*)o, lse, T, H);
  return launched(1);
}

cudaError_t attention_bwd(bool bf16, int B, int T, int H, int h, const void* q, const void* k,
                          const void* v, const void* o, const float* lse, const void* dout,
                          void* dq, long ldq, void* dk, long ldk, void* dv, long ldv,
                          float* delta, const Ctx& ctx) {
  if (!bf16) {
    const long rows = (long)B * T * H;
    const long keys = (long)B * T;
#define NC_ATTB(EE)                                                                          \
  attn_bwd_dq_f32_kernel<EE><<<(unsigned)((rows + 3) / 4), 128, 0, ctx.stream>>>(            \
      (const float*)q, (const float*)k, (const float*)v, (const float*)o, lse,               \
      (const float*)dout, (float*)dq, ldq, delta, B, T, H);                                  \
  attn_bwd_dkdv_f32_kernel<EE><<<(unsigned)((keys + 3) / 4), 128, 0, ctx.stream>>>(          \
      (const float*)q, (const float*)k, (const float*)v, lse, (const float*)dout, delta,     \
      (float*)dk, ldk, (float*)dv, ldv, B, T, H)
    if (h == 128) { NC_ATTB(4); } else { NC_ATTB(2); }
#undef NC_ATTB
    return launched(2);
  }
  if (h != HD) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dkdv_bf16_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kDkdvSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 gq((unsigned)(((long)T * H + TILE - 1) / TILE), B);
  attn_bwd_dq_bf16_kernel<<<gq, 128, kDqSmem, ctx.stream>>>(
      (const nc::bf16*)q, (const nc::bf16*)k, (const nc::bf16*)v, (const nc::bf16*)o, lse,
      (const nc::bf16*)dout, (nc::bf16*)dq, ldq, delta, T, H);
  dim3 gk((unsigned)((T + TILE - 1) / TILE), B);
  attn_bwd_dkdv_bf16_kernel<<<gk, 128, kDkdvSmem, ctx.stream>>>(
      (const nc::bf16*)q, (const nc::bf16*)k, (const nc::bf16*)v, lse, (const nc::bf16*)dout,
      delta, (nc::bf16*)dk, ldk, (nc::bf16*)dv, ldv, T, H);
  return launched(2);
}

// ---------------------------------------------------------------------------
// Allocation-free attention backward.
//
// The backward needs one float of scratch per packed query row (delta =
// rowsum(dO * O)).  nc_attention_bwd takes that scratch from the caller's
// workspace; the variant below instead uses this fixed array in device
// memory, which is part of the library image: every GPU that loads the
// library holds these 8 MB until the process exits, and no call allocates
// anything.  Every call shares the one array, so two calls that overlap on
// the GPU (for example on two streams) race; callers must order them.  Each
// call rewrites every delta entry it later reads, so nothing has to be
// cleared between calls.
static __device__ __align__(256) float g_noalloc_attn_delta[kNoAllocAttnMaxRows];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

// Device address of the array on the current device.  In host code the name
// g_noalloc_attn_delta is only a host-side stand-in, never a device address,
// so it is looked up here once per device (with that device current) and
// cached.
static cudaError_t noalloc_delta_ptr(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_attn_delta);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

cudaError_t attention_bwd_noalloc(bool bf16, int B, int T, int H, int h, const void* q,
                                  const void* k, const void* v, const void* o, const float* lse,
                                  const void* dout, void* dq, long ldq, void* dk, long ldk,
                                  void* dv, long ldv, const Ctx& ctx) {
  if ((long)B * T * H > kNoAllocAttnMaxRows) return cudaErrorInvalidValue;
  float* delta = nullptr;
  cudaError_t e = noalloc_delta_ptr(&delta);
  if (e != cudaSuccess) return e;
  return attention_bwd(bf16, B, T, H, h, q, k, v, o, lse, dout, dq, ldq, dk, ldk, dv, ldv, delta,
                       ctx);
}

}  // namespace nc
