// GEMM epilogues shared by the tcgen05 kernel (bf16) and the SIMT kernel (fp32).
//
// Each epilogue receives W consecutive fp32 accumulators of one output row,
// starting at column `col`, and returns a per-chunk contribution to a row
// reduction that only the softcap/cross-entropy epilogue uses.  The caller
// guarantees row < M and col + W <= N.
//
//   apply<W>    (SIMT kernel, W = 4): transform and store to global memory.
//   compute<W>  (tensor-core kernel, W = 128 bytes of Out): transform in
//               registers only; the kernel stages the chunk in shared memory
//               and writes it with one TMA bulk store, or a TMA bulk
//               reduce-add into the destination when reduce() is true.
//   Out         element type of the destination.
#pragma once

#include <cuda.h>

#include "nc_common.cuh"

namespace nc {

template <typename T, int W>
__device__ __forceinline__ void store_row_chunk(T* p, const float (&v)[W]) {
#pragma unroll
  for (int i = 0; i < W; i += 4) {
    float t[4] = {v[i], v[i + 1], v[i + 2], v[i + 3]};
    Vec4<T>::store(p + i, t);
  }
}
template <typename T, int W>
__device__ __forceinline__ void load_row_chunk(const T* p, float (&v)[W]) {
#pragma unroll
  for (int i = 0; i < W; i += 4) {
    float t[4];
    Vec4<T>::load(p + i, t);
    v[i] = t[0]; v[i + 1] = t[1]; v[i + 2] = t[2]; v[i + 3] = t[3];
  }
}

// C = acc (activation type: bf16 or fp32).
template <typename TOut>
struct EpiStore {
  static constexpr bool kRowReduce = false;
  using Out = TOut;
  TOut* c;
  long ldc;
  __device__ __forceinline__ bool reduce() const { return false; }
  template <int W>
  __device__ __forceinline__ float compute(int, int, float (&)[W], int) const { return 0.f; }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int) const {
    store_row_chunk<TOut, W>(c + (long)row * ldc + col, v);
    return 0.f;
  }
  __device__ __forceinline__ void row_end(int, int, float) const {}
};

// Scaled store: C = scale * acc (the dequantisation of a product of 8-bit
// operands: scale = s_A s_B).
template <typename TOut>
struct EpiScaleStore {
  static constexpr bool kRowReduce = false;
  using Out = TOut;
  TOut* c;
  long ldc;
  float scale;
  __device__ __forceinline__ bool reduce() const { return false; }
  template <int W>
  __device__ __forceinline__ float compute(int, int, float (&v)[W], int) const {
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] *= scale;
    return 0.f;
  }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int) const {
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] *= scale;
    store_row_chunk<TOut, W>(c + (long)row * ldc + col, v);
    return 0.f;
  }
  __device__ __forceinline__ void row_end(int, int, float) const {}
};

// Float32 store for weight gradients.  With split-K each split writes its own
// slab (c + split * split_stride) and a reduction kernel sums the slabs in a
// fixed order; with one split the epilogue writes (or accumulates into) C.
struct EpiStoreF32 {
  static constexpr bool kRowReduce = false;
  using Out = float;
  float* c;
  long ldc;
  long split_stride;
  int accumulate;
  __device__ __forceinline__ bool reduce() const { return accumulate != 0; }
  template <int W>
  __device__ __forceinline__ float compute(int, int, float (&)[W], int) const { return 0.f; }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int split) const {
    float* p = c + split * split_stride + (long)row * ldc + col;
    if (accumulate) {
      float o[W];
      load_row_chunk<float, W>(p, o);
#pragma unroll
      for (int i = 0; i < W; ++i) v[i] += o[i];
    }
    store_row_chunk<float, W>(p, v);
    return 0.f;
  }
  __device__ __forceinline__ void row_end(int, int, float) const {}
};

// Residual add into the float32 stream: X += acc.
struct EpiAddF32 {
  static constexpr bool kRowReduce = false;
  using Out = float;
  float* x;
  long ldx;
  __device__ __forceinline__ bool reduce() const { return true; }
  template <int W>
  __device__ __forceinline__ float compute(int, int, float (&)[W], int) const { return 0.f; }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int) const {
    float* p = x + (long)row * ldx + col;
    float o[W];
    load_row_chunk<float, W>(p, o);
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] += o[i];
    store_row_chunk<float, W>(p, v);
    return 0.f;
  }
  __device__ __forceinline__ void row_end(int, int, float) const {}
};

// ReLU^2 MLP activation: a = max(u, 0)^2.  Only `a` is kept: backward needs
// relu(u) = sqrt(a), which is recovered from `a` (see EpiRelu2Bwd).
template <typename TOut>
struct EpiRelu2 {
  static constexpr bool kRowReduce = false;
  using Out = TOut;
  TOut* a;
  long lda;
  __device__ __forceinline__ bool reduce() const { return false; }
  template <int W>
  __device__ __forceinline__ float compute(int, int, float (&v)[W], int) const {
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const float r = fmaxf(v[i], 0.f);
      v[i] = r * r;
    }
    return 0.f;
  }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int) const {
#pragma unroll
    for (int i = 0; i < W; ++i) {
      float r = fmaxf(v[i], 0.f);
      v[i] = r * r;
    }
    store_row_chunk<TOut, W>(a + (long)row * lda + col, v);
    return 0.f;
  }
  __device__ __forceinline__ void row_end(int, int, float) const {}
};

// Backward of ReLU^2 fused after dA = dY Wproj: dU = dA * 2 relu(u), with
// relu(u) = sqrt(a) read from the saved activation a = relu(u)^2.
template <typename TOut>
struct EpiRelu2Bwd {
  static constexpr bool kRowReduce = false;
  using Out = TOut;
  // The tensor-core kernel brings this tile's `a` in by TMA, one 128-byte
  // chunk per row at a time, ahead of the accumulator (compute_aux).
  static constexpr bool kAuxTma = true;
  TOut* du;
  const TOut* a;
  long ld;
  __device__ __forceinline__ bool reduce() const { return false; }
  __device__ __forceinline__ static float two_sqrt(float x) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return 2.f * r;
  }
  template <int W>
  __device__ __forceinline__ float compute_aux(int, int, float (&v)[W], int,
                                               const float (&av)[W]) const {
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] *= two_sqrt(av[i]);
    return 0.f;
  }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int) const {
    float av[W];
    load_row_chunk<TOut, W>(a + (long)row * ld + col, av);
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] *= 2.f * sqrtf(av[i]);
    store_row_chunk<TOut, W>(du + (long)row * ld + col, v);
    return 0.f;
  }
  __device__ __forceinline__ void row_end(int, int, float) const {}
};

// C = alpha * aux + beta * acc (aux of the output type, same layout as C;
// batch entry z reads aux + z * aux_bstride).  The Newton-Schulz steps of
// the Muon update use it: B = b A + c A A and X' = a X + B X.
template <typename TOut>
struct EpiAxpby {
  static constexpr bool kRowReduce = false;
  using Out = TOut;
  static constexpr bool kAuxTma = true;  // aux chunks come in by TMA (compute_aux)
  TOut* c;
  const TOut* aux;
  long ld;
  long aux_bstride;
  float alpha, beta;
  __device__ __forceinline__ bool reduce() const { return false; }
  template <int W>
  __device__ __forceinline__ float compute_aux(int, int, float (&v)[W], int,
                                               const float (&av)[W]) const {
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = alpha * av[i] + beta * v[i];
    return 0.f;
  }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int z) const {
    float av[W];
    load_row_chunk<TOut, W>(aux + (long)z * aux_bstride + (long)row * ld + col, av);
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = alpha * av[i] + beta * v[i];
    store_row_chunk<TOut, W>(c + (long)z * aux_bstride + (long)row * ld + col, v);
    return 0.f;
  }
  __device__ __forceinline__ void row_end(int, int, float) const {}
};

// LM head epilogue (tensor-core path): s = c tanh(z / c) stored as fp16 --
// |s| <= c = 15 lies well inside fp16's range and fp16 keeps 3 more mantissa
// bits than bf16 there; the per-row sum of exp(s) over this tile's columns
// goes to part[row * n_part + col_tile]; no max shift is needed because
// |s| <= c bounds exp(s) by e^c.  The capped logit at the row's target column
// is kept in fp32 (s_tgt) for the loss.
struct EpiSoftcapCE {
  static constexpr bool kRowReduce = true;
  using Out = __half;
  __half* s;
  long lds;
  float* part;
  int n_part;
  int tile_n;
  const int* targets;
  float* s_tgt;
  float cap, inv_cap;
  __device__ __forceinline__ bool reduce() const { return false; }
  template <int W>
  __device__ __forceinline__ float compute(int row, int col, float (&v)[W], int) const {
    const int y = __ldg(targets + row);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      float t;
      asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(v[i] * inv_cap));
      v[i] = cap * t;
      sum += __expf(v[i]);
      if (col + i == y) s_tgt[row] = v[i];
    }
    return sum;
  }
  template <int W>
  __device__ __forceinline__ float apply(int row, int col, float (&v)[W], int) const {
    const int y = __ldg(targets + row);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      float t;
      asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(v[i] * inv_cap));
      v[i] = cap * t;
      sum += __expf(v[i]);
      if (col + i == y) s_tgt[row] = v[i];
    }
    store_row_chunk<__half, W>(s + (long)row * lds + col, v);
    return sum;
  }
  __device__ __forceinline__ void row_end(int row, int col0, float sum) const {
    part[(long)row * n_part + col0 / tile_n] = sum;
  }
};

// QK-norm + RoPE fused into the QKV projection (launch article, architecture
// list: QK norm -- RMSNorm of every query head and of the key head -- and
// rotary embeddings).  The tensor-core kernel hands this epilogue one head at
// a time: the 128 fp32 accumulators of a row's head, as two 64-column chunks.
// Query heads (head < H) and the key head (head == H) are RMS-normalised over
// their 128 values and rotated by the token's position t = row % T: the
// half-split pairs (i, i + 64) are element i of the first chunk and element i
// of the second, rotated by angle t theta_i with (cos, sin) from the step's
// table; rstd_qk[row][head] keeps the normaliser for the backward.  The value
// head passes through.  Each chunk goes by its own tensor map to q (M, H h),
// k (M, h) or v (M, h), the layouts the attention kernels read.
struct EpiQkNormRope {
  static constexpr bool kRowReduce = false;
  static constexpr bool kHeadPairs = true;
  using Out = bf16;
  CUtensorMap mq, mk, mv;
  // (T, 64) pairs (cos, sin) of t theta_i as fp16 (an fp16 value carries a
  // 2^-11 relative error, a quarter of the bf16 rounding of the stored q and
  // k).  The kernel copies the 128 rows of a half tile into shared memory by
  // TMA (two 128-byte-swizzled [128 rows][128 B] chunks: pairs 0-31 and
  // 32-63), so T must be a multiple of 128.
  const __half2* tab;
  float* rstd_qk;     // (M, H + 1)
  int T, H;
  float eps;
  __device__ __forceinline__ bool reduce() const { return false; }
  __device__ __forceinline__ void row_end(int, int, float) const {}
  // Head `head` of output row `row`: a = its columns 0-63, b = 64-127; `tab`
  // holds the table rows of the half tile, this row's at index r.
  __device__ __forceinline__ void compute_head(int row, int head, float (&a)[64],
                                               float (&b)[64], const uint8_t* tab,
                                               int r) const {
    if (head > H) return;  // the value head: stored as computed
    float s8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s8[i] = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) s8[i & 7] = fmaf(a[i], a[i], fmaf(b[i], b[i], s8[i & 7]));
    const float ss = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
    const float rs = rsqrtf(ss / 128.f + eps);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint8_t* trow = tab + j * (128 * 128) + r * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 w = *reinterpret_cast<const uint4*>(trow + ((q ^ (r & 7)) << 4));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 c2 = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
          const int k = 32 * j + 4 * q + e;
          const float y0 = a[k] * rs, y1 = b[k] * rs;
          a[k] = y0 * c2.x - y1 * c2.y;
          b[k] = y0 * c2.y + y1 * c2.x;
        }
      }
    }
    rstd_qk[(long)row * (H + 1) + head] = rs;
  }
  // Destination of the 64-column chunk starting at column `col` of the
  // (M, (H + 2) 128) product, and the chunk's first column there.
  __device__ __forceinline__ const CUtensorMap* dest(int col, int& x) const {
    const int head = col >> 7;
    if (head < H) {
      x = col;
      return &mq;
    }
    x = col & 127;
    return head == H ? &mk : &mv;
  }
};

}  // namespace nc
