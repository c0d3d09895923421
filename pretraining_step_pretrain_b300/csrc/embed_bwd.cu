// Backward of the token embedding + post-embedding RMSNorm (launch article,
// architecture list: untied embedding, norm right after the embedding).
//
//   dx0[t]  = r0[t] (dx[t] - y[t] mean(dx[t] y[t])),  y[t] = wte[id_t] r0[t]
//   dwte[v] = sum over tokens t with id_t == v of dx0[t]
//
// The scatter-add is made deterministic: token indices are sorted by id with
// a stable LSD radix sort (8-bit digits), then every vocabulary row sums its
// tokens in increasing token order.  No floating-point atomics are used.
#include <algorithm>

#include "nc_common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

constexpr int kSortTile = 1024;     // keys per CTA in the radix passes
constexpr int kSortThreads = 256;

template <typename W>
__global__ void embed_bwd_rows_kernel(const int* __restrict__ ids, const W* __restrict__ wte,
                                      const float* __restrict__ rstd0, const float* __restrict__ dx,
                                      float* __restrict__ dx0, uint32_t* __restrict__ keys,
                                      uint32_t* __restrict__ vals, int M, int d, int V) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  int id = ids[row];
  const bool valid = id >= 0 && id < V;
  if (!valid) id = 0;  // its gradient row is zero; nc_embed_norm reported the id
  if (lane == 0) {
    keys[row] = (uint32_t)id;
    vals[row] = (uint32_t)row;
  }
  const float r = valid ? rstd0[row] : 0.f;
  const W* wr = wte + (long)id * d;
  const float* dxr = dx + (long)row * d;
  float dot = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float a[4], w[4];
    Vec4<float>::load(dxr + c, a);
    Vec4<W>::load(wr + c, w);
    dot += (a[0] * w[0] + a[1] * w[1] + a[2] * w[2] + a[3] * w[3]) * r;
  }
  const float mean = warp_sum(dot) / (float)d;
  float* out = dx0 + (long)row * d;
  for (int c = lane * 4; c < d; c += 128) {
    float a[4], w[4], o[4];
    Vec4<float>::load(dxr + c, a);
    Vec4<W>::load(wr + c, w);
    for (int i = 0; i < 4; ++i) o[i] = r * (a[i] - w[i] * r * mean);
    Vec4<float>::store(out + c, o);
  }
}

__global__ void radix_hist_kernel(const uint32_t* __restrict__ keys, int M, int shift,
                                  uint32_t* __restrict__ hist, int ntiles) {
  __shared__ uint32_t cnt[256];
  cnt[threadIdx.x] = 0;
  __syncthreads();
  const int base = blockIdx.x * kSortTile;
  for (int i = threadIdx.x; i < kSortTile; i += kSortThreads) {
    if (base + i < M) atomicAdd(&cnt[(keys[base + i] >> shift) & 255u], 1u);
  }
  __syncthreads();
  hist[threadIdx.x * ntiles + blockIdx.x] = cnt[threadIdx.x];
}

// Exclusive scan of n counters in one CTA of 1024 threads.
__global__ void radix_scan_kernel(uint32_t* __restrict__ data, int n) {
  __shared__ uint32_t sums[1024];
  const int per = (n + 1023) / 1024;
  const int lo = threadIdx.x * per, hi = min(n, lo + per);
  uint32_t s = 0;
  for (int i = lo; i < hi; ++i) s += data[i];
  sums[threadIdx.x] = s;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const uint32_t v = threadIdx.x >= off ? sums[threadIdx.x - off] : 0u;
    __syncthreads();
    sums[threadIdx.x] += v;
    __syncthreads();
  }
  uint32_t run = sums[threadIdx.x] - s;
  for (int i = lo; i < hi; ++i) {
    const uint32_t v = data[i];
    data[i] = run;
    run += v;
  }
}

// Stable scatter: within a tile, keys keep their order (round-major, thread
// order within a round); warp peers with equal digits are ranked by lane.
__global__ void radix_scatter_kernel(const uint32_t* __restrict__ keys_in,
                                     const uint32_t* __restrict__ vals_in,
                                     uint32_t* __restrict__ keys_out,
                                     uint32_t* __restrict__ vals_out, int M, int shift,
                                     const uint32_t* __restrict__ offsets, int ntiles) {
  __shared__ uint32_t base[256];
  __shared__ uint32_t running[256];
  __shared__ uint32_t wcount[kSortThreads / 32][257];
  const int t = threadIdx.x, w = t >> 5, lane = t & 31;
  base[t] = offsets[t * ntiles + blockIdx.x];
  running[t] = 0;
  for (int i = 0; i < kSortThreads / 32; ++i) wcount[i][t] = 0;
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = 0; r < kSortTile / kSortThreads; ++r) {
    const int idx = blockIdx.x * kSortTile + r * kSortThreads + t;
    const bool valid = idx < M;
    const uint32_t key = valid ? keys_in[idx] : 0u;
    const uint32_t val = valid ? vals_in[idx] : 0u;
    const uint32_t digit = valid ? ((key >> shift) & 255u) : 256u;
    const unsigned peers = __match_any_sync(0xffffffffu, digit);
    const uint32_t rank = __popc(peers & lt_mask);
    if ((peers & lt_mask) == 0) wcount[w][digit] = __popc(peers);
    __syncthreads();
    if (valid) {
      uint32_t prefix = 0;
      for (int i = 0; i < w; ++i) prefix += wcount[i][digit];
      const uint32_t dst = base[digit] + running[digit] + prefix + rank;
      keys_out[dst] = key;
      vals_out[dst] = val;
    }
    __syncthreads();
    uint32_t total = 0;
    for (int i = 0; i < kSortThreads / 32; ++i) {
      total += wcount[i][t];
      wcount[i][t] = 0;
    }
    running[t] += total;
    __syncthreads();
  }
}

// One CTA per vocabulary row: sum its (sorted) tokens in token order.
__global__ void segment_sum_kernel(const uint32_t* __restrict__ keys,
                                   const uint32_t* __restrict__ vals,
                                   const float* __restrict__ dx0, float* __restrict__ dwte, int M,
                                   int d, int accumulate) {
  __shared__ int range[2];
  const uint32_t v = blockIdx.x;
  if (threadIdx.x < 2) {
    const uint32_t target = v + threadIdx.x;  // lower_bound(v), lower_bound(v + 1)
    int lo = 0, hi = M;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (keys[mid] < target) lo = mid + 1; else hi = mid;
    }
    range[threadIdx.x] = lo;
  }
  __syncthreads();
  const int b = range[0], e = range[1];
  float* out = dwte + (long)v * d;
  for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = b; i < e; ++i) {
      float t[4];
      Vec4<float>::load(dx0 + (long)vals[i] * d + c, t);
      for (int k = 0; k < 4; ++k) acc[k] += t[k];
    }
    if (accumulate) {
      float o[4];
      Vec4<float>::load(out + c, o);
      for (int k = 0; k < 4; ++k) acc[k] += o[k];
    }
    Vec4<float>::store(out + c, acc);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t embed_bwd_scratch_bytes(int M, int d) {
  const int ntiles = (M + kSortTile - 1) / kSortTile;
  return align256((size_t)M * d * 4) + 4 * align256((size_t)M * 4) +
         align256((size_t)256 * ntiles * 4);
}

cudaError_t embed_norm_bwd(bool bf16, const int* ids, const void* wte, const float* rstd0,
                           const float* dx, float* dwte, int accumulate, int M, int d, int V,
                           void* scratch, const Ctx& ctx) {
  uint8_t* p = static_cast<uint8_t*>(scratch);
  float* dx0 = reinterpret_cast<float*>(p);
  p += align256((size_t)M * d * 4);
  uint32_t* k0 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)M * 4);
  uint32_t* v0 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)M * 4);
  uint32_t* k1 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)M * 4);
  uint32_t* v1 = reinterpret_cast<uint32_t*>(p); p += align256((size_t)M * 4);
  uint32_t* hist = reinterpret_cast<uint32_t*>(p);
  const int ntiles = (M + kSortTile - 1) / kSortTile;

  const int rblocks = (M + 7) / 8;
  if (bf16)
    embed_bwd_rows_kernel<nc::bf16><<<rblocks, 256, 0, ctx.stream>>>(
        ids, static_cast<const nc::bf16*>(wte), rstd0, dx, dx0, k0, v0, M, d, V);
  else
    embed_bwd_rows_kernel<float><<<rblocks, 256, 0, ctx.stream>>>(
        ids, static_cast<const float*>(wte), rstd0, dx, dx0, k0, v0, M, d, V);
  note_launch(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  int bits = 1;
  while ((1 << bits) < V) ++bits;
  for (int shift = 0; shift < bits; shift += 8) {
    radix_hist_kernel<<<ntiles, kSortThreads, 0, ctx.stream>>>(k0, M, shift, hist, ntiles);
    radix_scan_kernel<<<1, 1024, 0, ctx.stream>>>(hist, 256 * ntiles);
    radix_scatter_kernel<<<ntiles, kSortThreads, 0, ctx.stream>>>(k0, v0, k1, v1, M, shift, hist,
                                                                  ntiles);
    note_launch(3);
    std::swap(k0, k1);
    std::swap(v0, v1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  segment_sum_kernel<<<V, 128, 0, ctx.stream>>>(k0, v0, dx0, dwte, M, d, accumulate);
  return launched(1);
}

}  // namespace nc
