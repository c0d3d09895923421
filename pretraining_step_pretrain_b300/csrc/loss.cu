// Softcap + log-softmax + next-token cross-entropy and its backward
// (launch article, architecture list: untied unembedding with a logit softcap;
// walkthrough section "预训练": next-token prediction).
//
//   s = c tanh(z / c),   loss = mean over targets >= 0 of [lse(s_t) - s_t[y_t]]
//   dz = (softmax(s) - onehot(y)) * (1 - (s/c)^2) / N_valid
//
// Tensor-core path: the LM-head GEMM epilogue already wrote fp16 s, per-row
// partial sums of exp(s) for every 256-column tile, and s at the target; the
// kernels below reduce the partials (fixed order), form the loss, and turn s
// into bf16 dz in place.  fp32 debug path: the GEMM wrote z; a row kernel
// applies the cap and computes lse in fp32.
#include <algorithm>

#include "nc_common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

__device__ __forceinline__ float block_reduce_max(float v, float* sh) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) sh[w] = v;
  __syncthreads();
  float r = (l < (int)(blockDim.x >> 5)) ? sh[l] : -INFINITY;
  r = warp_max(r);
  __syncthreads();
  return r;
}
__device__ __forceinline__ float block_reduce_sum(float v, float* sh) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) sh[w] = v;
  __syncthreads();
  float r = (l < (int)(blockDim.x >> 5)) ? sh[l] : 0.f;
  r = warp_sum(r);
  __syncthreads();
  return r;
}

// fp32 path: one CTA per row; z -> s in place, lse and s[target].
__global__ void softcap_rows_f32_kernel(float* __restrict__ s, const int* __restrict__ targets,
                                        float* __restrict__ lse, float* __restrict__ s_tgt, int V,
                                        float cap) {
  __shared__ float sh[32];
  const long row = blockIdx.x;
  float* sr = s + row * V;
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < V; c += blockDim.x) {
    const float v = cap * tanhf(sr[c] / cap);
    sr[c] = v;
    mx = fmaxf(mx, v);
  }
  mx = block_reduce_max(mx, sh);
  float sum = 0.f;
  for (int c = threadIdx.x; c < V; c += blockDim.x) sum += expf(sr[c] - mx);
  sum = block_reduce_sum(sum, sh);
  if (threadIdx.x == 0) {
    lse[row] = mx + logf(sum);
    const int y = targets[row];
    s_tgt[row] = (y >= 0 && y < V) ? sr[y] : 0.f;
  }
}

// tensor-core path: lse from the per-tile partial sums, summed in tile order.
__global__ void ce_rows_kernel(const float* __restrict__ part, int n_part,
                               float* __restrict__ lse, int M) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= M) return;
  const float* p = part + (long)row * n_part;
  float sum = 0.f;
  for (int i = 0; i < n_part; ++i) sum += p[i];
  lse[row] = logf(sum);
}

// Deterministic mean over valid rows (fixed-order tree in one CTA).
// A target outside [-1, V) counts as ignored and records DEV_TOKEN_RANGE.
__global__ void ce_loss_kernel(const float* __restrict__ lse, const float* __restrict__ s_tgt,
                               const int* __restrict__ targets, int M, int V, float* loss,
                               float* inv_n, int* err) {
  __shared__ double sh_sum[1024];
  __shared__ int sh_cnt[1024];
  double acc = 0.0;
  int cnt = 0;
  for (int i = threadIdx.x; i < M; i += blockDim.x) {
    const int y = targets[i];
    if (y >= 0 && y < V) {
      acc += (double)lse[i] - (double)s_tgt[i];
      ++cnt;
    } else if (y >= V || y < -1) {
      raise_error(err, DEV_TOKEN_RANGE, 2, i);
    }
  }
  sh_sum[threadIdx.x] = acc;
  sh_cnt[threadIdx.x] = cnt;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      sh_sum[threadIdx.x] += sh_sum[threadIdx.x + s];
      sh_cnt[threadIdx.x] += sh_cnt[threadIdx.x + s];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int n = sh_cnt[0] > 0 ? sh_cnt[0] : 1;
    *loss = (float)(sh_sum[0] / n);
    *inv_n = 1.f / (float)n;
  }
}

// 8 consecutive elements: one 16-byte access for 16-bit types, two for fp32.
__device__ __forceinline__ void load8(const __half* p, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  Vec4<float>::load(p, *reinterpret_cast<float(*)[4]>(v));
  Vec4<float>::load(p + 4, *reinterpret_cast<float(*)[4]>(v + 4));
}
__device__ __forceinline__ void store8(bf16* p, const float (&v)[8]) {
  uint4 q;
  uint32_t* w = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(p) = q;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  Vec4<float>::store(p, *reinterpret_cast<const float(*)[4]>(v));
  Vec4<float>::store(p + 4, *reinterpret_cast<const float(*)[4]>(v + 4));
}

// Forward-only evaluation: mean loss over valid targets and bits per byte
// (fixed-order tree in one CTA).  out[0] = sum(loss_t) / n in nats;
// out[1] = sum over targets with byte length > 0 of loss_t / (ln 2 * sum of
// their byte lengths), or NaN without a byte table.
__global__ void eval_loss_kernel(const float* __restrict__ lse, const float* __restrict__ s_tgt,
                                 const int* __restrict__ targets,
                                 const int* __restrict__ token_bytes, int M, int V,
                                 float* out, int* err) {
  __shared__ double sh_l[1024], sh_lb[1024];
  __shared__ long long sh_n[1024], sh_b[1024];
  double acc = 0.0, acc_b = 0.0;
  long long cnt = 0, nbytes = 0;
  for (int i = threadIdx.x; i < M; i += blockDim.x) {
    const int y = targets[i];
    if (y >= 0 && y < V) {
      const double nats = (double)lse[i] - (double)s_tgt[i];
      acc += nats;
      ++cnt;
      if (token_bytes) {
        const int nb = token_bytes[y];
        if (nb > 0) {
          acc_b += nats;
          nbytes += nb;
        }
      }
    } else if (y >= V || y < -1) {
      raise_error(err, DEV_TOKEN_RANGE, 3, i);
    }
  }
  sh_l[threadIdx.x] = acc;
  sh_lb[threadIdx.x] = acc_b;
  sh_n[threadIdx.x] = cnt;
  sh_b[threadIdx.x] = nbytes;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      sh_l[threadIdx.x] += sh_l[threadIdx.x + s];
      sh_lb[threadIdx.x] += sh_lb[threadIdx.x + s];
      sh_n[threadIdx.x] += sh_n[threadIdx.x + s];
      sh_b[threadIdx.x] += sh_b[threadIdx.x + s];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const long long n = sh_n[0] > 0 ? sh_n[0] : 1;
    out[0] = (float)(sh_l[0] / (double)n);
    out[1] = (token_bytes && sh_b[0] > 0)
                 ? (float)(sh_lb[0] / (0.6931471805599453 * (double)sh_b[0]))
                 : __int_as_float(0x7fc00000);
  }
}

// dz in place.  TS: stored capped logit type, TG: gradient type written over
// it (same size).  One CTA per row; 8 elements (16 B of fp16/bf16, two 16 B
// vectors of fp32) per thread and step.
template <typename TS, typename TG, bool kFastExp>
__global__ void __launch_bounds__(256) ce_dlogits_kernel(TS* __restrict__ s,
                                                         const float* __restrict__ lse,
                                                         const int* __restrict__ targets,
                                                         const float* __restrict__ inv_n, int V,
                                                         float cap) {
  const long row = blockIdx.x;
  int y = targets[row];
  if (y >= V) y = -1;
  const float scale = y >= 0 ? *inv_n : 0.f;  // ignored rows get a zero gradient
  const float inv_c = 1.f / cap;
  const float l = lse[row];
  TS* sr = s + row * V;
  TG* gr = reinterpret_cast<TG*>(sr);
  const int v8 = V & ~7;
  for (int c = threadIdx.x * 8; c < v8; c += blockDim.x * 8) {
    float v[8];
    load8(sr + c, v);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float sv = v[k];
      const float p = kFastExp ? __expf(sv - l) : expf(sv - l);
      const float t = sv * inv_c;
      v[k] = (p - (c + k == y ? 1.f : 0.f)) * (1.f - t * t) * scale;
    }
    store8(gr + c, v);
  }
  for (int c = v8 + threadIdx.x; c < V; c += blockDim.x) {
    const float sv = to_f(sr[c]);
    const float p = kFastExp ? __expf(sv - l) : expf(sv - l);
    const float t = sv * inv_c;
    gr[c] = from_f<TG>((p - (c == y ? 1.f : 0.f)) * (1.f - t * t) * scale);
  }
}

}  // namespace

cudaError_t softcap_rows_f32(float* s, const int* targets, float* lse, float* s_tgt, int M,
                             int V, float cap, const Ctx& ctx) {
  softcap_rows_f32_kernel<<<M, 256, 0, ctx.stream>>>(s, targets, lse, s_tgt, V, cap);
  return launched(1);
}

cudaError_t ce_rows_from_partials(const float* part, int n_part, float* lse, int M,
                                  const Ctx& ctx) {
  ce_rows_kernel<<<(M + 255) / 256, 256, 0, ctx.stream>>>(part, n_part, lse, M);
  return launched(1);
}

cudaError_t ce_loss(const float* lse, const float* s_tgt, const int* targets, int M, int V,
                    float* loss, float* inv_n, const Ctx& ctx) {
  ce_loss_kernel<<<1, 1024, 0, ctx.stream>>>(lse, s_tgt, targets, M, V, loss, inv_n, ctx.err);
  return launched(1);
}

cudaError_t eval_loss(const float* lse, const float* s_tgt, const int* targets,
                      const int* token_bytes, int M, int V, float* out, const Ctx& ctx) {
  eval_loss_kernel<<<1, 1024, 0, ctx.stream>>>(lse, s_tgt, targets, token_bytes, M, V, out,
                                               ctx.err);
  return launched(1);
}

cudaError_t ce_dlogits(bool bf16, void* s, const float* lse, const int* targets,
                       const float* inv_n, int M, int V, float cap, const Ctx& ctx) {
  if (M <= 0) return cudaSuccess;
  if (bf16)
    ce_dlogits_kernel<__half, nc::bf16, true><<<M, 256, 0, ctx.stream>>>(
        static_cast<__half*>(s), lse, targets, inv_n, V, cap);
  else
    ce_dlogits_kernel<float, float, false><<<M, 256, 0, ctx.stream>>>(
        static_cast<float*>(s), lse, targets, inv_n, V, cap);
  return launched(1);
}

}  // namespace nc
