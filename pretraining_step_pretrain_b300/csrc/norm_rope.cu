// Memory-bound kernels of the step: parameter-free RMSNorm forward/backward,
// the post-embedding norm, QK-norm + rotary embedding forward/backward, the
// RoPE table and a float32 -> activation cast.  One warp per row (or per
// (token, head)), 16-byte loads of fp32 / 8-byte loads of 16-bit data,
// warp-shuffle reductions.  Activation type A is bf16 or float.
//
// RMSNorm (launch article, architecture list: RMSNorm carries no learnable
// gain): y = x * r, r = 1/sqrt(mean(x^2) + eps).
// Backward (from y = x r(x)): dx = r (dy - y * mean(dy * y)).
#include <algorithm>

#include "nc_common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float rms_inv(float sumsq, int n, float eps) {
  return rsqrtf(sumsq / (float)n + eps);
}

// E consecutive elements (E = 4: one 8- or 16-byte access; E = 2: scalars).
template <typename A, int E>
__device__ __forceinline__ void load_vec(const A* p, float (&x)[E]) {
  if constexpr (E == 4) {
    Vec4<A>::load(p, x);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = to_f(p[e]);
  }
}
template <typename A, int E>
__device__ __forceinline__ void store_vec(A* p, const float (&x)[E]) {
  if constexpr (E == 4) {
    Vec4<A>::store(p, x);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) p[e] = from_f<A>(x[e]);
  }
}

// ---- RoPE table: tab[t * h/2 + i] = (cos, sin)(t * base^(-2i/h)), fp64 math.
__global__ void rope_table_kernel(float2* tab, __half2* tab16, int T, int half, int h,
                                  double base) {
  const long n = (long)T * half;
  for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < n;
       idx += (long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / half), i = (int)(idx % half);
    const double theta = pow(base, -2.0 * (double)i / (double)h);
    double s, c;
    sincos((double)t * theta, &s, &c);
    tab[idx] = make_float2((float)c, (float)s);
    if (tab16) tab16[idx] = __floats2half2_rn((float)c, (float)s);
  }
}

// ---- embedding gather + RMSNorm -> float32 residual.
template <typename W>
__global__ void embed_norm_kernel(const int* __restrict__ ids, const W* __restrict__ wte,
                                  float* __restrict__ x, float* __restrict__ rstd, int M, int d,
                                  int V, float eps, int* err) {
  const int row = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const int id = ids[row];
  float* xr = x + (long)row * d;
  if (id < 0 || id >= V) {
    if (lane == 0) {
      raise_error(err, DEV_TOKEN_RANGE, 1, row);
      rstd[row] = 0.f;
    }
    for (int c = lane * 4; c < d; c += 128) {
      const float z[4] = {0.f, 0.f, 0.f, 0.f};
      Vec4<float>::store(xr + c, z);
    }
    return;
  }
  const W* wr = wte + (long)id * d;
  float ss = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float v[4];
    Vec4<W>::load(wr + c, v);
    ss += v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
  }
  const float r = rms_inv(warp_sum(ss), d, eps);
  for (int c = lane * 4; c < d; c += 128) {
    float v[4];
    Vec4<W>::load(wr + c, v);
    for (int i = 0; i < 4; ++i) v[i] *= r;
    Vec4<float>::store(xr + c, v);
  }
  if (lane == 0) rstd[row] = r;
}

// ---- RMSNorm forward: float32 residual row -> activation row.
template <typename A>
__global__ void rmsnorm_fwd_kernel(const float* __restrict__ x, A* __restrict__ y,
                                   float* __restrict__ rstd, int M, int d, float eps) {
  const int row = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const float* xr = x + (long)row * d;
  float ss = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float v[4];
    Vec4<float>::load(xr + c, v);
    ss += v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
  }
  const float r = rms_inv(warp_sum(ss), d, eps);
  A* yr = y + (long)row * d;
  for (int c = lane * 4; c < d; c += 128) {
    float v[4];
    Vec4<float>::load(xr + c, v);
    for (int i = 0; i < 4; ++i) v[i] *= r;
    Vec4<A>::store(yr + c, v);
  }
  if (lane == 0) rstd[row] = r;
}

// ---- RMSNorm backward (+ residual): dx (+)= r (dy - y mean(dy y)); also
// writes the activation-type copy of dx used as the next GEMM operand.
template <typename A>
__global__ void rmsnorm_bwd_kernel(const A* __restrict__ dy, const A* __restrict__ y,
                                   const float* __restrict__ rstd, float* __restrict__ dx,
                                   A* __restrict__ dx_act, int add, int M, int d) {
  const int row = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const A* dyr = dy + (long)row * d;
  const A* yr = y + (long)row * d;
  float dot = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float a[4], b[4];
    Vec4<A>::load(dyr + c, a);
    Vec4<A>::load(yr + c, b);
    dot += a[0] * b[0] + a[1] * b[1] + a[2] * b[2] + a[3] * b[3];
  }
  const float mean = warp_sum(dot) / (float)d;
  const float r = rstd[row];
  float* dxr = dx + (long)row * d;
  A* dar = dx_act + (long)row * d;
  for (int c = lane * 4; c < d; c += 128) {
    float a[4], b[4], o[4];
    Vec4<A>::load(dyr + c, a);
    Vec4<A>::load(yr + c, b);
    if (add) Vec4<float>::load(dxr + c, o);
    for (int i = 0; i < 4; ++i) {
      const float g = r * (a[i] - b[i] * mean);
      o[i] = add ? o[i] + g : g;
    }
    Vec4<float>::store(dxr + c, o);
    Vec4<A>::store(dar + c, o);
  }
}

template <typename A>
__global__ void cast_kernel(const float* __restrict__ x, A* __restrict__ y, long n4) {
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4;
       i += (long)gridDim.x * blockDim.x) {
    float v[4];
    Vec4<float>::load(x + 4 * i, v);
    Vec4<A>::store(y + 4 * i, v);
  }
}

// ---- QK-norm + RoPE forward.  One warp per (token m, head j), j in [0, H+2):
// j < H query heads and j == H the key head are RMS-normalised over their h
// values and rotated; j == H+1 (value) is copied.  Lane l holds elements
// [E l, E l + E); the rotation partner of element i < h/2 is i + h/2, held by
// lane l ^ 16 at the same slot.
template <typename A, int E>
__global__ void qknorm_rope_fwd_kernel(const A* __restrict__ qkv, const float2* __restrict__ tab,
                                       A* __restrict__ q, A* __restrict__ k, A* __restrict__ v,
                                       float* __restrict__ rstd_qk, int M, int T, int H,
                                       float eps) {
  // One warp per token: H query heads, the key head, the value head.  The
  // token's (cos, sin) pairs are read once; four heads are loaded before any
  // is used so that several loads are in flight per lane.
  constexpr int h = 32 * E, half = h / 2;
  const int m = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= M) return;
  const int t = m % T;
  const bool lo = lane < 16;
  float2 cs[E];
#pragma unroll
  for (int e = 0; e < E; ++e) cs[e] = tab[(long)t * half + (lane & 15) * E + e];
  const int nh = H + 2;
  const A* src = qkv + (long)m * nh * h + lane * E;
  for (int j0 = 0; j0 < nh; j0 += 4) {
    float x[4][E];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j0 + u < nh) load_vec<A, E>(src + (long)(j0 + u) * h, x[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      if (j >= nh) break;
      if (j == H + 1) {
        store_vec<A, E>(v + (long)m * h + lane * E, x[u]);
        continue;
      }
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) ss += x[u][e] * x[u][e];
      const float r = rms_inv(warp_sum(ss), h, eps);
      float out[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float y = x[u][e] * r;
        const float pr = __shfl_xor_sync(0xffffffffu, y, 16);
        out[e] = lo ? (y * cs[e].x - pr * cs[e].y) : (pr * cs[e].y + y * cs[e].x);
      }
      A* dst = (j < H) ? q + ((long)m * H + j) * h + lane * E : k + (long)m * h + lane * E;
      store_vec<A, E>(dst, out);
      if (lane == 0) rstd_qk[(long)m * (H + 1) + j] = r;
    }
  }
}

// ---- QK-norm + RoPE backward, in place on the (M, (H+2)h) gradient buffer.
// With z = R(y) the saved rotated output and g = dL/dz:
//   dx = r * R^T (g - z * mean(g z))      (R orthogonal, so g.z = R^T g . R^T z)
template <typename A, int E>
__global__ void qknorm_rope_bwd_kernel(A* __restrict__ dqkv, const A* __restrict__ q,
                                       const A* __restrict__ k, const float* __restrict__ rstd_qk,
                                       const float2* __restrict__ tab, int M, int T, int H) {
  // One warp per token (H query heads + the key head; the value gradient
  // passes through), four heads' loads in flight before any is used.
  constexpr int h = 32 * E, half = h / 2;
  const int m = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= M) return;
  const int t = m % T;
  const bool lo = lane < 16;
  float2 cs[E];
#pragma unroll
  for (int e = 0; e < E; ++e) cs[e] = tab[(long)t * half + (lane & 15) * E + e];
  const int nh = H + 1;
  A* grow = dqkv + (long)m * (H + 2) * h + lane * E;
  for (int j0 = 0; j0 < nh; j0 += 4) {
    float g[4][E], z[4][E];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      if (j < nh) {
        load_vec<A, E>(grow + (long)j * h, g[u]);
        load_vec<A, E>((j < H) ? q + ((long)m * H + j) * h + lane * E : k + (long)m * h + lane * E,
                       z[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      if (j >= nh) break;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot += g[u][e] * z[u][e];
      const float mean = warp_sum(dot) / (float)h;
      const float r = rstd_qk[(long)m * (H + 1) + j];
      float out[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float w = g[u][e] - z[u][e] * mean;
        const float pr = __shfl_xor_sync(0xffffffffu, w, 16);
        out[e] = r * (lo ? (w * cs[e].x + pr * cs[e].y) : (w * cs[e].x - pr * cs[e].y));
      }
      store_vec<A, E>(grow + (long)j * h, out);
    }
  }
}

// ---- QK-norm + RoPE backward, staged: each warp streams whole tokens (the
// gradient rows and the saved q, k rows) through a ring of kStages
// shared-memory slots filled by bulk copies (one mbarrier per slot), so every
// warp keeps kStages - 1 tokens of loads in flight without holding them in
// registers.  Same arithmetic as qknorm_rope_bwd_kernel, which remains the
// path for shapes whose slots do not fit in shared memory.  (The same
// staging of the forward measured no faster than its register version.)
constexpr int kStages = 3;
constexpr int kStagedWarps = 4;
constexpr int SITE_QKNORM = 400;

// Order this thread's generic-proxy shared-memory reads before a later bulk
// copy (async proxy) into the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Elements lane*E .. lane*E + E - 1 of a head row held in shared memory.
template <typename A, int E>
__device__ __forceinline__ void load_vec_s(const uint8_t* p, float (&x)[E]) {
  load_vec<A, E>(reinterpret_cast<const A*>(p), x);
}

// A warp-private ring: slot s of warp w at sm + (w * kStages + s) * slot_bytes.
struct WarpRing {
  uint8_t* base;
  uint64_t* bars;  // [kStages]
  uint32_t slot_bytes;
  __device__ uint8_t* slot(int s) const { return base + (size_t)s * slot_bytes; }
};

// On a timed-out wait: wait (bounded) for this warp's other copies in flight
// (armed[s]: the parity slot s's pending fill completes with, or -1), then the
// caller returns.
__device__ __forceinline__ void ring_drain(const WarpRing& r, const int (&armed)[kStages],
                                           int* err, long long timeout_ns) {
  int none = 0;
  for (int s = 0; s < kStages; ++s)
    if (armed[s] >= 0)
      mbar_wait_bounded(&r.bars[s], (uint32_t)armed[s], &none, err, SITE_QKNORM, timeout_ns / 8);
}

template <typename A, int E>
__global__ void __launch_bounds__(32 * kStagedWarps)
    qknorm_rope_bwd_staged_kernel(A* __restrict__ dqkv, const A* __restrict__ q,
                                  const A* __restrict__ k, const float* __restrict__ rstd_qk,
                                  const float2* __restrict__ tab, int M, int T, int H, int* err,
                                  long long timeout_ns) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint64_t bars[kStagedWarps][kStages];
  constexpr int h = 32 * E, half = h / 2;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nh = H + 1;  // query heads + the key head (the value gradient passes through)
  const uint32_t row = (uint32_t)h * sizeof(A);
  // slot: g (nh rows of the gradient) then z (H rows of q, one of k)
  const WarpRing r{sm + (size_t)w * kStages * 2 * nh * row, bars[w], 2 * nh * row};
  const long stride = (long)gridDim.x * kStagedWarps;
  const long m0 = (long)blockIdx.x * kStagedWarps + w;
  auto fill = [&](long m, int s) {
    uint8_t* d = r.slot(s);
    mbar_arrive_expect_tx(&r.bars[s], r.slot_bytes);
    bulk_g2s(d, dqkv + m * (H + 2) * h, nh * row, &r.bars[s]);
    bulk_g2s(d + nh * row, q + m * H * h, H * row, &r.bars[s]);
    bulk_g2s(d + (2 * nh - 1) * row, k + m * h, row, &r.bars[s]);
  };
  int armed[kStages];
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&r.bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  for (int s = 0; s < kStages; ++s) {
    const long m = m0 + s * stride;
    armed[s] = m < M ? 0 : -1;
    if (lane == 0 && m < M) fill(m, s);
  }
  const bool lo = lane < 16;
  int s = 0;
  uint32_t ph = 0;
  for (long m = m0; m < M; m += stride) {
    const int t = (int)(m % T);
    float2 cs[E];
#pragma unroll
    for (int e = 0; e < E; ++e) cs[e] = tab[(long)t * half + (lane & 15) * E + e];
    const float rl = lane < nh ? rstd_qk[m * nh + lane] : 0.f;
    int none = 0;
    if (!mbar_wait_bounded(&r.bars[s], ph, &none, err, SITE_QKNORM, timeout_ns)) {
      armed[s] = -1;
      ring_drain(r, armed, err, timeout_ns);
      return;
    }
    const uint8_t* gs = r.slot(s) + lane * E * sizeof(A);
    const uint8_t* zs = gs + nh * row;
    A* grow = dqkv + m * (H + 2) * h + lane * E;
    for (int j = 0; j < nh; ++j) {
      float g[E], z[E];
      load_vec_s<A, E>(gs + (size_t)j * row, g);
      load_vec_s<A, E>(zs + (size_t)j * row, z);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot += g[e] * z[e];
      const float mean = warp_sum(dot) / (float)h;
      const float rr = j < 32 ? __shfl_sync(0xffffffffu, rl, j) : rstd_qk[m * nh + j];
      float out[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float wv = g[e] - z[e] * mean;
        const float pr = __shfl_xor_sync(0xffffffffu, wv, 16);
        out[e] = rr * (lo ? (wv * cs[e].x + pr * cs[e].y) : (wv * cs[e].x - pr * cs[e].y));
      }
      store_vec<A, E>(grow + (size_t)j * h, out);
    }
    __syncwarp();
    const long mn = m + kStages * stride;
    if (mn < M) {
      if (lane == 0) {
        fence_proxy_async_shared();
        fill(mn, s);
      }
      armed[s] = (int)(ph ^ 1u);  // the parity this refill completes with
    } else {
      armed[s] = -1;
    }
    if (++s == kStages) { s = 0; ph ^= 1u; }
  }
}

inline int row_blocks(long rows) { return (int)((rows + kWarpsPerBlock - 1) / kWarpsPerBlock); }

// Dynamic shared memory of a staged launch, or 0 when its slots do not fit.
constexpr int kStagedMaxSmem = 200 * 1024;
inline int staged_smem(long slot_bytes) {
  const long bytes = slot_bytes * kStages * kStagedWarps;
  return bytes <= kStagedMaxSmem ? (int)bytes : 0;
}
inline int staged_blocks(long M, int smem, int num_sms) {
  const int per_sm = std::max(1, std::min(8, (int)((227L * 1024) / (smem + 1024))));
  return (int)std::max<long>(1, std::min<long>((M + kStagedWarps - 1) / kStagedWarps,
                                               (long)num_sms * per_sm));
}

}  // namespace

cudaError_t rope_table(float2* tab, void* tab16, int T, int h, float base, const Ctx& ctx) {
  const long n = (long)T * (h / 2);
  const int blocks = (int)std::min<long>((n + 255) / 256, 4096);
  rope_table_kernel<<<blocks, 256, 0, ctx.stream>>>(tab, static_cast<__half2*>(tab16), T, h / 2,
                                                    h, (double)base);
  return launched(1);
}

cudaError_t embed_norm_fwd(bool bf16, const int* ids, const void* wte, float* x, float* rstd,
                           int M, int d, int V, float eps, const Ctx& ctx) {
  if (bf16)
    embed_norm_kernel<nc::bf16><<<row_blocks(M), 32 * kWarpsPerBlock, 0, ctx.stream>>>(
        ids, static_cast<const nc::bf16*>(wte), x, rstd, M, d, V, eps, ctx.err);
  else
    embed_norm_kernel<float><<<row_blocks(M), 32 * kWarpsPerBlock, 0, ctx.stream>>>(
        ids, static_cast<const float*>(wte), x, rstd, M, d, V, eps, ctx.err);
  return launched(1);
}

cudaError_t rmsnorm_fwd(bool bf16, const float* x, void* y, float* rstd, int M, int d, float eps,
                        const Ctx& ctx) {
  if (bf16)
    rmsnorm_fwd_kernel<nc::bf16><<<row_blocks(M), 32 * kWarpsPerBlock, 0, ctx.stream>>>(
        x, static_cast<nc::bf16*>(y), rstd, M, d, eps);
  else
    rmsnorm_fwd_kernel<float><<<row_blocks(M), 32 * kWarpsPerBlock, 0, ctx.stream>>>(
        x, static_cast<float*>(y), rstd, M, d, eps);
  return launched(1);
}

cudaError_t rmsnorm_bwd(bool bf16, const void* dy, const void* y, const float* rstd, float* dx,
                        void* dx_act, int add, int M, int d, const Ctx& ctx) {
  if (bf16)
    rmsnorm_bwd_kernel<nc::bf16><<<row_blocks(M), 32 * kWarpsPerBlock, 0, ctx.stream>>>(
        static_cast<const nc::bf16*>(dy), static_cast<const nc::bf16*>(y), rstd, dx,
        static_cast<nc::bf16*>(dx_act), add, M, d);
  else
    rmsnorm_bwd_kernel<float><<<row_blocks(M), 32 * kWarpsPerBlock, 0, ctx.stream>>>(
        static_cast<const float*>(dy), static_cast<const float*>(y), rstd, dx,
        static_cast<float*>(dx_act), add, M, d);
  return launched(1);
}

cudaError_t cast_f32_to_act(bool bf16, const float* x, void* y, long n, const Ctx& ctx) {
  const long n4 = n / 4;
  const int blocks = (int)std::max<long>(1, std::min<long>((n4 + 255) / 256, (long)ctx.num_sms * 16));
  if (bf16)
    cast_kernel<nc::bf16><<<blocks, 256, 0, ctx.stream>>>(x, static_cast<nc::bf16*>(y), n4);
  else
    cast_kernel<float><<<blocks, 256, 0, ctx.stream>>>(x, static_cast<float*>(y), n4);
  return launched(1);
}

template <typename A, int E>
cudaError_t qknorm_bwd_staged(void* dqkv, const void* q, const void* k, const float* rstd_qk,
                              const float2* tab, int M, int T, int H, int blocks, int smem,
                              const Ctx& ctx) {
  static bool attr = false;  // the opt-in shared-memory limit, set once per instantiation
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(qknorm_rope_bwd_staged_kernel<A, E>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kStagedMaxSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  qknorm_rope_bwd_staged_kernel<A, E><<<blocks, 32 * kStagedWarps, smem, ctx.stream>>>(
      static_cast<A*>(dqkv), static_cast<const A*>(q), static_cast<const A*>(k), rstd_qk, tab, M,
      T, H, ctx.err, ctx.timeout_ns);
  return launched(1);
}

cudaError_t qknorm_rope_fwd(bool bf16, const void* qkv, const float2* tab, void* q, void* k,
                            void* v, float* rstd_qk, int B, int T, int H, int h, float eps,
                            const Ctx& ctx) {
  const int M = B * T;
  const int blocks = row_blocks(M);
#define NC_QKF(TA, EE)                                                                      \
  qknorm_rope_fwd_kernel<TA, EE><<<blocks, 32 * kWarpsPerBlock, 0, ctx.stream>>>(          \
      static_cast<const TA*>(qkv), tab, static_cast<TA*>(q), static_cast<TA*>(k),          \
      static_cast<TA*>(v), rstd_qk, M, T, H, eps)
  if (bf16) {
    if (h == 128) NC_QKF(nc::bf16, 4); else NC_QKF(nc::bf16, 2);
  } else {
    if (h == 128) NC_QKF(float, 4); else NC_QKF(float, 2);
  }
#undef NC_QKF
  return launched(1);
}

cudaError_t qknorm_rope_bwd(bool bf16, void* dqkv, const void* q, const void* k,
                            const float* rstd_qk, const float2* tab, int B, int T, int H, int h,
                            const Ctx& ctx) {
  const int M = B * T;
  const int smem = staged_smem(2L * (H + 1) * h * (bf16 ? 2 : 4));
  if (smem > 0) {
    const int blocks = staged_blocks(M, smem, ctx.num_sms);
    if (bf16) {
      if (h == 128) return qknorm_bwd_staged<nc::bf16, 4>(dqkv, q, k, rstd_qk, tab, M, T, H, blocks, smem, ctx);
      return qknorm_bwd_staged<nc::bf16, 2>(dqkv, q, k, rstd_qk, tab, M, T, H, blocks, smem, ctx);
    }
    if (h == 128) return qknorm_bwd_staged<float, 4>(dqkv, q, k, rstd_qk, tab, M, T, H, blocks, smem, ctx);
    return qknorm_bwd_staged<float, 2>(dqkv, q, k, rstd_qk, tab, M, T, H, blocks, smem, ctx);
  }
  const int blocks = row_blocks(M);
#define NC_QKB(TA, EE)                                                                      \
  qknorm_rope_bwd_kernel<TA, EE><<<blocks, 32 * kWarpsPerBlock, 0, ctx.stream>>>(          \
      static_cast<TA*>(dqkv), static_cast<const TA*>(q), static_cast<const TA*>(k), rstd_qk, \
      tab, M, T, H)
  if (bf16) {
    if (h == 128) NC_QKB(nc::bf16, 4); else NC_QKB(nc::bf16, 2);
  } else {
    if (h == 128) NC_QKB(float, 4); else NC_QKB(float, 2);
  }
#undef NC_QKB
  return launched(1);
}

}  // namespace nc
