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
// bf16 path (h = 128): tcgen05 tensor-core kernels in attention_tc.cu (online
// softmax forward; backward as a Q-major dQ pass that also writes
// delta = rowsum(dO * O) and a KV-major dK/dV pass summing over every packed
// row, hence over all heads, without atomics).
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
  if (h != 128) return cudaErrorInvalidValue;
  return attention_fwd_tc(B, T, H, q, k, v, o, lse, ctx);
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
  if (h != 128) return cudaErrorInvalidValue;
  return attention_bwd_tc(B, T, H, q, k, v, o, lse, dout, dq, ldq, dk, ldk, dv, ldv, delta, ctx);
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

// The device error word of the allocation-free calls, laid out like the one
// at the start of a workspace ([0] status, first writer wins; [1] site; [2]
// detail).  The kernels' bounded waits record a timeout here; it starts at
// zero when the library loads and is read and cleared by
// noalloc_read_status().  Shared by every call, like the array above.
static __device__ __align__(16) int g_noalloc_err[4];

namespace {
constexpr int kMaxDevices = 64;
struct NoAllocPtrs {
  float* delta = nullptr;
  int* err = nullptr;
};
std::mutex g_noalloc_mu;
NoAllocPtrs g_noalloc_ptr[kMaxDevices];
}  // namespace

// Device addresses of the array and the error word on the current device.
// In host code their names are only host-side stand-ins, never device
// addresses, so they are looked up here once per device (with that device
// current) and cached.
static cudaError_t noalloc_ptrs(NoAllocPtrs* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocPtrs& p = g_noalloc_ptr[dev];
  if (!p.delta) {
    void* d = nullptr;
    void* w = nullptr;
    e = cudaGetSymbolAddress(&d, g_noalloc_attn_delta);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(&w, g_noalloc_err);
    if (e != cudaSuccess) return e;
    p.delta = static_cast<float*>(d);
    p.err = static_cast<int*>(w);
  }
  *out = p;
  return cudaSuccess;
}

cudaError_t noalloc_error_word(int** err) {
  NoAllocPtrs p;
  cudaError_t e = noalloc_ptrs(&p);
  if (e == cudaSuccess) *err = p.err;
  return e;
}

cudaError_t noalloc_read_status(cudaStream_t stream, int word[4]) {
  int* err = nullptr;
  cudaError_t e = noalloc_error_word(&err);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(word, err, 4 * sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(err, 0, 4 * sizeof(int));
  return e;
}

cudaError_t attention_bwd_noalloc(bool bf16, int B, int T, int H, int h, const void* q,
                                  const void* k, const void* v, const void* o, const float* lse,
                                  const void* dout, void* dq, long ldq, void* dk, long ldk,
                                  void* dv, long ldv, const Ctx& ctx) {
  if ((long)B * T * H > kNoAllocAttnMaxRows) return cudaErrorInvalidValue;
  NoAllocPtrs p;
  cudaError_t e = noalloc_ptrs(&p);
  if (e != cudaSuccess) return e;
  Ctx c = ctx;
  c.err = p.err;
  return attention_bwd(bf16, B, T, H, h, q, k, v, o, lse, dout, dq, ldq, dk, ldk, dv, ldv,
                       p.delta, c);
}

}  // namespace nc
