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

// dz in place.  TS: stored capped logit type, TG: gradient type written over it.
template <typename TS, typename TG, bool kFastExp>
__global__ void ce_dlogits_kernel(TS* __restrict__ s, const float* __restrict__ lse,
                                  const int* __restrict__ targets, const float* __restrict__ inv_n,
                                  int M, int V, float cap) {
  const long n4 = (long)M * V / 4;
  const float scale = *inv_n;
  const float inv_c = 1.f / cap;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4;
       i += (long)gridDim.x * blockDim.x) {
    const long e0 = 4 * i;
    const int row = (int)(e0 / V), col = (int)(e0 % V);
    int y = targets[row];
    if (y >= V) y = -1;
    float v[4];
    Vec4<TS>::load(s + e0, v);
    const float l = lse[row];
    for (int k = 0; k < 4; ++k) {
      const float sv = v[k];
      const float p = kFastExp ? __expf(sv - l) : expf(sv - l);
      const float t = sv * inv_c;
      float g = (p - (col + k == y ? 1.f : 0.f)) * (1.f - t * t) * scale;
      v[k] = y >= 0 ? g : 0.f;
    }
    Vec4<TG>::store(reinterpret_cast<TG*>(s) + e0, v);
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

cudaError_t ce_dlogits(bool bf16, void* s, const float* lse, const int* targets,
                       const float* inv_n, int M, int V, float cap, const Ctx& ctx) {
  const long n4 = (long)M * V / 4;
  const int blocks = (int)std::max<long>(1, std::min<long>((n4 + 255) / 256, (long)ctx.num_sms * 32));
  if (bf16)
    ce_dlogits_kernel<__half, nc::bf16, true><<<blocks, 256, 0, ctx.stream>>>(
        static_cast<__half*>(s), lse, targets, inv_n, M, V, cap);
  else
    ce_dlogits_kernel<float, float, false><<<blocks, 256, 0, ctx.stream>>>(
        static_cast<float*>(s), lse, targets, inv_n, M, V, cap);
  return launched(1);
}

}  // namespace nc
