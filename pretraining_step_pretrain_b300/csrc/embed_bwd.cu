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

// Segmented sum over the sorted token list, cut into fixed slices of kSlice
// tokens (one CTA each).  Inside a slice every run of equal ids is summed in
// token order.  A run that is a whole segment (its neighbours on both sides
// carry other ids) is written to dwte directly; a run cut by a slice edge is
// a partial: the first run of slice s goes to part_first[s], the last to
// part_last[s] (a slice that is one single cut run uses part_first).
constexpr int kSlice = 64;
constexpr int kSegThreads = 128;

__global__ void __launch_bounds__(kSegThreads)
    segment_slice_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals,
                         const float* __restrict__ dx0, float* __restrict__ dwte,
                         float* __restrict__ part_first, float* __restrict__ part_last, int M,
                         int d, int accumulate) {
  __shared__ uint32_t k_s[kSlice], v_s[kSlice];
  const int s = blockIdx.x;
  const int i0 = s * kSlice, n = min(kSlice, M - i0);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    k_s[i] = keys[i0 + i];
    v_s[i] = vals[i0 + i];
  }
  const uint32_t prev = i0 > 0 ? keys[i0 - 1] : 0xFFFFFFFFu;
  const uint32_t next = i0 + n < M ? keys[i0 + n] : 0xFFFFFFFFu;
  __syncthreads();
  for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int run0 = 0;
    for (int g = 0; g < n; g += 8) {
      float t[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (g + j < n) Vec4<float>::load(dx0 + (long)v_s[g + j] * d + c, t[j]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = g + j;
        if (i >= n) break;
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] += t[j][k];
        const uint32_t v = k_s[i];
        const uint32_t after = i + 1 < n ? k_s[i + 1] : next;
        if (after == v) continue;  // the run goes on
        // The run ends at i.  It is a whole segment unless it began before
        // this slice; such a run is the slice's first run (a partial).
        float* out;
        if (run0 > 0 || prev != v) {
          out = dwte + (long)v * d + c;
          if (accumulate) {
            float o[4];
            Vec4<float>::load(out, o);
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] += o[k];
          }
        } else {
          out = part_first + (long)s * d + c;
        }
        Vec4<float>::store(out, acc);
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = 0.f;
        run0 = i + 1;
      }
    }
    if (run0 < n) {
      // The last run continues into the next slice.
      float* out = (run0 == 0 ? part_first : part_last) + (long)s * d;
      Vec4<float>::store(out + c, acc);
    }
  }
}

// One CTA per (slice, group of columns): if a segment cut by slice edges
// starts in this slice, sum its partials slice by slice (fixed order) and
// write its dwte row.  The segment's last slice comes from a binary search
// of the sorted ids, and the partials are loaded eight slices at a time
// before they are added in order, so a long segment (the most frequent
// token spans hundreds of slices) keeps several loads in flight.
constexpr int kJoinThreads = 64;
constexpr int kJoinBatch = 8;

__global__ void __launch_bounds__(kJoinThreads)
    segment_join_kernel(const uint32_t* __restrict__ keys, const float* __restrict__ part_first,
                        const float* __restrict__ part_last, float* __restrict__ dwte, int M,
                        int d, int accumulate) {
  const int s = blockIdx.x;
  const int i0 = s * kSlice, n = min(kSlice, M - i0);
  const uint32_t v = keys[i0 + n - 1];
  if (i0 + n >= M || keys[i0 + n] != v) return;  // the last run ends in this slice
  const bool whole_slice = keys[i0] == v;
  if (whole_slice && i0 > 0 && keys[i0 - 1] == v) return;  // began in an earlier slice
  const int c = (blockIdx.y * kJoinThreads + threadIdx.x) * 4;
  if (c >= d) return;
  // last index holding v: the keys are sorted
  int lo = i0 + n, hi = M;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (keys[mid] <= v) lo = mid + 1; else hi = mid;
  }
  const int s_end = (lo - 1) / kSlice;
  float acc[4];
  Vec4<float>::load((whole_slice ? part_first : part_last) + (long)s * d + c, acc);
  for (int s2 = s + 1; s2 <= s_end; s2 += kJoinBatch) {
    float t[kJoinBatch][4];
#pragma unroll
    for (int j = 0; j < kJoinBatch; ++j)
      if (s2 + j <= s_end) Vec4<float>::load(part_first + (long)(s2 + j) * d + c, t[j]);
#pragma unroll
    for (int j = 0; j < kJoinBatch; ++j)
      if (s2 + j <= s_end)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] += t[j][k];
  }
  float* out = dwte + (long)v * d + c;
  if (accumulate) {
    float o[4];
    Vec4<float>::load(out, o);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] += o[k];
  }
  Vec4<float>::store(out, acc);
}

// Rows of dwte whose id occurs in no token: zero (or left as they are when
// accumulating).  One warp per vocabulary row; lane 0 binary-searches the
// sorted ids.
__global__ void segment_zero_kernel(const uint32_t* __restrict__ keys, float* __restrict__ dwte,
                                    int M, int d, int V) {
  const int v = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (v >= V) return;
  int present = 0;
  if (lane == 0) {
    int lo = 0, hi = M;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (keys[mid] < (uint32_t)v) lo = mid + 1; else hi = mid;
    }
    present = lo < M && keys[lo] == (uint32_t)v;
  }
  present = __shfl_sync(0xffffffffu, present, 0);
  if (present) return;
  float* out = dwte + (long)v * d;
  const float z[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = lane * 4; c < d; c += 128) Vec4<float>::store(out + c, z);
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t embed_bwd_scratch_bytes(int M, int d) {
  const int ntiles = (M + kSortTile - 1) / kSortTile;
  const size_t nslices = (M + kSlice - 1) / kSlice;
  return align256((size_t)M * d * 4) + 4 * align256((size_t)M * 4) +
         align256((size_t)256 * ntiles * 4) + 2 * align256(nslices * d * 4);
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
  const int ntiles_ = (M + kSortTile - 1) / kSortTile;
  p += align256((size_t)256 * ntiles_ * 4);
  const int nslices = (M + kSlice - 1) / kSlice;
  float* part_first = reinterpret_cast<float*>(p); p += align256((size_t)nslices * d * 4);
  float* part_last = reinterpret_cast<float*>(p);
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
  if (!accumulate) {
    segment_zero_kernel<<<(V + 7) / 8, 256, 0, ctx.stream>>>(k0, dwte, M, d, V);
    note_launch(1);
  }
  segment_slice_kernel<<<nslices, kSegThreads, 0, ctx.stream>>>(k0, v0, dx0, dwte, part_first,
                                                                part_last, M, d, accumulate);
  const dim3 jgrid(nslices, (unsigned)((d + 4 * kJoinThreads - 1) / (4 * kJoinThreads)));
  segment_join_kernel<<<jgrid, kJoinThreads, 0, ctx.stream>>>(k0, part_first, part_last, dwte, M,
                                                              d, accumulate);
  return launched(2);
}

}  // namespace nc
