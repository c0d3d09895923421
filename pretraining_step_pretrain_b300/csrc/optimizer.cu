// The optimizer step that follows the pretraining step (launch article's
// Q&A, architecture list: Muon + AdamW after modded-nanoGPT; walkthrough,
// section "预训练": Muon for the matrices, AdamW for the embedding and the
// unembedding, learning rates scaled by 1/sqrt(dim), lrm decaying linearly
// to 0 at the end).
//
// Master weights, gradients and optimizer state are fp32; every update also
// rewrites the compute copy (bf16, or fp32 in the debug mode) that the next
// forward pass reads.
//
//   AdamW (embedding, LM head): one element-wise pass, float4 accesses.
//   Muon (every block matrix, r x c):
//     1. b <- mu b + g; u = g + mu b; per-block partial sums of u^2
//     2. X0 = u / (||u||_F + 1e-7) in bf16, wide orientation (transposed
//        when r > c), all layers of one shape in one batch
//     3. Newton-Schulz steps X <- a X + (b A + c A A) X, A = X X^T, as batched
//        tcgen05 GEMMs (gemm.cu)
//     4. W <- W - lr sqrt(max(1, r/c)) X (transposed back), compute copy.
// The partial sums are reduced in a fixed order, so a step is bit-reproducible.
#include <algorithm>
#include <cmath>
#include <vector>

#include "nc.h"
#include "nc_common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

template <typename C>
__global__ void adamw_kernel(float* __restrict__ p, const float* __restrict__ g,
                             float* __restrict__ m, float* __restrict__ v, C* __restrict__ pc,
                             long n4, AdamWArgs a) {
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4;
       i += (long)gridDim.x * blockDim.x) {
    float pv[4], gv[4], mv[4], vv[4];
    Vec4<float>::load(p + 4 * i, pv);
    Vec4<float>::load(g + 4 * i, gv);
    Vec4<float>::load(m + 4 * i, mv);
    Vec4<float>::load(v + 4 * i, vv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      mv[k] = a.beta1 * mv[k] + (1.f - a.beta1) * gv[k];
      vv[k] = a.beta2 * vv[k] + (1.f - a.beta2) * gv[k] * gv[k];
      const float mhat = mv[k] * a.inv_bc1;
      const float vhat = vv[k] * a.inv_bc2;
      pv[k] = pv[k] - a.lr * a.wd * pv[k] - a.lr * mhat / (sqrtf(vhat) + a.eps);
    }
    Vec4<float>::store(p + 4 * i, pv);
    Vec4<float>::store(m + 4 * i, mv);
    Vec4<float>::store(v + 4 * i, vv);
    Vec4<C>::store(pc + 4 * i, pv);
  }
}

constexpr int kNormBlocks = 256;  // partial sums per matrix
constexpr int kNormThreads = 256;

// b <- mu b + g (in place) and per-block partial sums of u^2, u = g + mu b.
__global__ void __launch_bounds__(kNormThreads)
    muon_momentum_kernel(const float* __restrict__ g, float* __restrict__ b, long n4, float mu,
                         float* __restrict__ partial) {
  __shared__ float red[kNormThreads / 32];
  float ss = 0.f;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4;
       i += (long)gridDim.x * blockDim.x) {
    float gv[4], bv[4];
    Vec4<float>::load(g + 4 * i, gv);
    Vec4<float>::load(b + 4 * i, bv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      bv[k] = mu * bv[k] + gv[k];
      const float u = gv[k] + mu * bv[k];
      ss += u * u;
    }
    Vec4<float>::store(b + 4 * i, bv);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kNormThreads / 32; ++w) t += red[w];
    partial[blockIdx.x] = t;
  }
}

// X0 = u / (||u||_F + 1e-7) (activation type), u = g + mu b, in the wide orientation:
// X0[i][j] = u[i][j] (r <= c) or u[j][i] (r > c, X0 is c x r).  32 x 32 tiles
// through shared memory keep both sides coalesced.
template <typename X>
__global__ void muon_prepare_kernel(const float* __restrict__ g, const float* __restrict__ b,
                                    float mu, const float* __restrict__ partial, int r, int c,
                                    int transpose, X* __restrict__ x) {
  __shared__ float tile[32][33];
  __shared__ float inv_norm;
  if (threadIdx.x == 0 && threadIdx.y == 0) {
    float t = 0.f;
    for (int i = 0; i < kNormBlocks; ++i) t += partial[i];  // fixed order
    inv_norm = 1.f / (sqrtf(t) + 1e-7f);
  }
  __syncthreads();
  const float s = inv_norm;
  const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 32;  // tile of u (r x c)
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    const int i = i0 + k, j = j0 + threadIdx.x;
    float u = 0.f;
    if (i < r && j < c) {
      const long o = (long)i * c + j;
      u = (g[o] + mu * b[o]) * s;
    }
    tile[k][threadIdx.x] = u;
  }
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    if (!transpose) {
      const int i = i0 + k, j = j0 + threadIdx.x;
      if (i < r && j < c) x[(long)i * c + j] = from_f<X>(tile[k][threadIdx.x]);
    } else {
      const int jj = j0 + k, ii = i0 + threadIdx.x;  // X0 is c x r: X0[jj][ii] = u[ii][jj]
      if (ii < r && jj < c) x[(long)jj * r + ii] = from_f<X>(tile[threadIdx.x][k]);
    }
  }
}

// W <- W - step X^T-or-X, compute copy rewritten.  X is the final
// Newton-Schulz iterate in the wide orientation (activation type C).
template <typename C>
__global__ void muon_update_kernel(float* __restrict__ p, const C* __restrict__ x, int r, int c,
                                   int transpose, float step, C* __restrict__ pc) {
  __shared__ float tile[32][33];
  const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 32;  // tile of W (r x c)
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    float o = 0.f;
    if (!transpose) {
      const int i = i0 + k, j = j0 + threadIdx.x;
      if (i < r && j < c) o = to_f(x[(long)i * c + j]);
      tile[k][threadIdx.x] = o;
    } else {
      const int jj = j0 + k, ii = i0 + threadIdx.x;
      if (ii < r && jj < c) o = to_f(x[(long)jj * r + ii]);
      tile[threadIdx.x][k] = o;
    }
  }
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    const int i = i0 + k, j = j0 + threadIdx.x;
    if (i < r && j < c) {
      const long o = (long)i * c + j;
      const float w = p[o] - step * tile[k][threadIdx.x];
      p[o] = w;
      pc[o] = from_f<C>(w);
    }
  }
}

}  // namespace

cudaError_t adamw_step(bool bf16_copy, float* p, const float* g, float* m, float* v, void* pc,
                       long n, const AdamWArgs& a, const Ctx& ctx) {
  const long n4 = n / 4;  // n is a multiple of 64 (vocab x d_model)
  const int blocks = (int)std::max<long>(1, std::min<long>((n4 + 255) / 256, (long)ctx.num_sms * 8));
  if (bf16_copy)
    adamw_kernel<nc::bf16><<<blocks, 256, 0, ctx.stream>>>(p, g, m, v, static_cast<nc::bf16*>(pc),
                                                           n4, a);
  else
    adamw_kernel<float><<<blocks, 256, 0, ctx.stream>>>(p, g, m, v, static_cast<float*>(pc), n4,
                                                        a);
  return launched(1);
}

cudaError_t muon_momentum(const float* g, float* b, long n, float mu, float* partial,
                          const Ctx& ctx) {
  muon_momentum_kernel<<<kNormBlocks, kNormThreads, 0, ctx.stream>>>(g, b, n / 4, mu, partial);
  return launched(1);
}

int muon_partials() { return kNormBlocks; }

cudaError_t muon_prepare(bool bf16, const float* g, const float* b, float mu,
                         const float* partial, int r, int c, bool transpose, void* x,
                         const Ctx& ctx) {
  dim3 grid((c + 31) / 32, (r + 31) / 32), block(32, 8);
  if (bf16)
    muon_prepare_kernel<nc::bf16><<<grid, block, 0, ctx.stream>>>(
        g, b, mu, partial, r, c, transpose ? 1 : 0, static_cast<nc::bf16*>(x));
  else
    muon_prepare_kernel<float><<<grid, block, 0, ctx.stream>>>(g, b, mu, partial, r, c,
                                                               transpose ? 1 : 0,
                                                               static_cast<float*>(x));
  return launched(1);
}

cudaError_t muon_update(bool bf16, float* p, const void* x, int r, int c, bool transpose,
                        float step, void* pc, const Ctx& ctx) {
  dim3 grid((c + 31) / 32, (r + 31) / 32), block(32, 8);
  if (bf16)
    muon_update_kernel<nc::bf16><<<grid, block, 0, ctx.stream>>>(
        p, static_cast<const nc::bf16*>(x), r, c, transpose ? 1 : 0, step,
        static_cast<nc::bf16*>(pc));
  else
    muon_update_kernel<float><<<grid, block, 0, ctx.stream>>>(
        p, static_cast<const float*>(x), r, c, transpose ? 1 : 0, step, static_cast<float*>(pc));
  return launched(1);
}

// ---------------------------------------------------------------- host side
namespace {

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Block matrices of one layer: 0 w_qkv, 1 w_o, 2 w_fc, 3 w_proj (rows, cols).
void kind_shape(const nc_config& c, int kind, int& r, int& cc) {
  const int d = c.d_model, Hh = c.n_head * c.head_dim, q = (c.n_head + 2) * c.head_dim,
            f = c.d_mlp;
  switch (kind) {
    case 0: r = q; cc = d; break;
    case 1: r = d; cc = Hh; break;
    case 2: r = f; cc = d; break;
    default: r = d; cc = f; break;
  }
}

// Groups of kinds whose wide orientation (m = min, n = max) coincides: every
// layer's matrices of a group go through the Newton-Schulz GEMMs as one batch.
struct MuonGroup {
  int m, n;
  std::vector<int> kinds;
};
std::vector<MuonGroup> muon_groups(const nc_config& c) {
  std::vector<MuonGroup> gs;
  for (int k = 0; k < 4; ++k) {
    int r, cc;
    kind_shape(c, k, r, cc);
    const int m = std::min(r, cc), n = std::max(r, cc);
    bool found = false;
    for (auto& g : gs)
      if (g.m == m && g.n == n) {
        g.kinds.push_back(k);
        found = true;
      }
    if (!found) gs.push_back({m, n, {k}});
  }
  return gs;
}

struct OptLayout {
  size_t partial, x0, x1, a, bm, total;
};
OptLayout opt_layout(const nc_config& c) {
  const size_t es = c.dtype == NC_BF16 ? 2 : 4;
  size_t max_x = 0, max_a = 0;
  for (const auto& g : muon_groups(c)) {
    const size_t cnt = (size_t)c.depth * g.kinds.size();
    max_x = std::max(max_x, cnt * g.m * g.n);
    max_a = std::max(max_a, cnt * g.m * g.m);
  }
  OptLayout L;
  size_t o = 256;  // device error word
  L.partial = o;
  o += al256((size_t)4 * c.depth * kNormBlocks * 4);
  L.x0 = o;
  o += al256(max_x * es);
  L.x1 = o;
  o += al256(max_x * es);
  L.a = o;
  o += al256(max_a * es);
  L.bm = o;
  o += al256(max_a * es);
  L.total = o;
  return L;
}

template <typename T>
T pick(const nc_layer_f& l, int kind) {
  switch (kind) {
    case 0: return l.w_qkv;
    case 1: return l.w_o;
    case 2: return l.w_fc;
    default: return l.w_proj;
  }
}
void* pick_c(const nc_layer_wc& l, int kind) {
  switch (kind) {
    case 0: return l.w_qkv;
    case 1: return l.w_o;
    case 2: return l.w_fc;
    default: return l.w_proj;
  }
}
const float* pick_g(const nc_layer_g& l, int kind) {
  switch (kind) {
    case 0: return l.d_qkv;
    case 1: return l.d_o;
    case 2: return l.d_fc;
    default: return l.d_proj;
  }
}

}  // namespace

size_t optimizer_ws_bytes(const nc_config& c) { return opt_layout(c).total; }

cudaError_t optimizer_step(const nc_config& c, const nc_opt_config& oc, int t, float lrm,
                           const OptTensors& w, void* ws, const Ctx& ctx) {
  const bool bf = c.dtype == NC_BF16;
  const size_t es = bf ? 2 : 4;
  const OptLayout L = opt_layout(c);
  uint8_t* base = static_cast<uint8_t*>(ws);
  cudaError_t e;

  // AdamW: embedding and LM head, rates scaled by lrm / sqrt(d_model).
  AdamWArgs a;
  a.beta1 = oc.beta1;
  a.beta2 = oc.beta2;
  a.eps = oc.eps;
  a.wd = oc.weight_decay;
  a.inv_bc1 = (float)(1.0 / (1.0 - std::pow((double)oc.beta1, (double)t)));
  a.inv_bc2 = (float)(1.0 / (1.0 - std::pow((double)oc.beta2, (double)t)));
  const long nvd = (long)c.vocab * c.d_model;
  const float width = (float)(1.0 / std::sqrt((double)c.d_model));
  a.lr = oc.lr_embed * lrm * width;
  if ((e = adamw_step(bf, w.wte, w.dwte, w.m_wte, w.v_wte, w.wte_c, nvd, a, ctx)) != cudaSuccess)
    return e;
  a.lr = oc.lr_lm * lrm * width;
  if ((e = adamw_step(bf, w.w_lm, w.dw_lm, w.m_lm, w.v_lm, w.w_lm_c, nvd, a, ctx)) != cudaSuccess)
    return e;

  // Muon: every block matrix, one batch per shape group.
  float* partial = reinterpret_cast<float*>(base + L.partial);
  int slot = 0;
  for (const auto& g : muon_groups(c)) {
    const int cnt = c.depth * (int)g.kinds.size();
    uint8_t* X = base + L.x0;
    uint8_t* Xn = base + L.x1;
    uint8_t* A = base + L.a;
    uint8_t* Bm = base + L.bm;
    const long mn = (long)g.m * g.n, mm = (long)g.m * g.m;
    // momentum, norm, first iterate (wide orientation)
    for (int i = 0; i < cnt; ++i) {
      const int layer = i / (int)g.kinds.size(), kind = g.kinds[i % g.kinds.size()];
      int r, cc;
      kind_shape(c, kind, r, cc);
      const float* gr = pick_g(w.grads[layer], kind);
      float* mb = pick<float*>(w.mom[layer], kind);
      float* pt = partial + (size_t)(slot + i) * kNormBlocks;
      if ((e = muon_momentum(gr, mb, (long)r * cc, oc.momentum, pt, ctx)) != cudaSuccess) return e;
      if ((e = muon_prepare(bf, gr, mb, oc.momentum, pt, r, cc, r > cc, X + i * mn * es, ctx)) !=
          cudaSuccess)
        return e;
    }
    // Newton-Schulz: A = X X^T; B = b A + c A A; X <- a X + B X (batched)
    for (int s = 0; s < oc.ns_steps; ++s) {
      GemmArgs g1{};
      g1.layout = GEMM_NT; g1.epi = EPI_STORE;
      g1.M = g.m; g1.N = g.m; g1.K = g.n;
      g1.A = X; g1.lda = g.n; g1.B = X; g1.ldb = g.n; g1.C = A; g1.ldc = g.m;
      g1.batch = cnt; g1.a_bstride = mn; g1.b_bstride = mn; g1.c_bstride = mm;
      GemmArgs g2{};
      g2.layout = GEMM_NT; g2.epi = EPI_AXPBY;
      g2.M = g.m; g2.N = g.m; g2.K = g.m;
      g2.A = A; g2.lda = g.m; g2.B = A; g2.ldb = g.m; g2.C = Bm; g2.ldc = g.m; g2.aux = A;
      g2.alpha = oc.ns_b; g2.beta = oc.ns_c;
      g2.batch = cnt; g2.a_bstride = mm; g2.b_bstride = mm; g2.c_bstride = mm;
      GemmArgs g3{};
      g3.layout = GEMM_NN; g3.epi = EPI_AXPBY;
      g3.M = g.m; g3.N = g.n; g3.K = g.m;
      g3.A = Bm; g3.lda = g.m; g3.B = X; g3.ldb = g.n; g3.C = Xn; g3.ldc = g.n; g3.aux = X;
      g3.alpha = oc.ns_a; g3.beta = 1.f;
      g3.batch = cnt; g3.a_bstride = mm; g3.b_bstride = mn; g3.c_bstride = mn;
      for (GemmArgs* ga : {&g1, &g2, &g3}) {
        e = bf ? gemm_bf16(*ga, ctx) : gemm_f32(*ga, ctx);
        if (e != cudaSuccess) return e;
      }
      std::swap(X, Xn);
    }
    // W <- W - lr lrm sqrt(max(1, r/c)) X
    for (int i = 0; i < cnt; ++i) {
      const int layer = i / (int)g.kinds.size(), kind = g.kinds[i % g.kinds.size()];
      int r, cc;
      kind_shape(c, kind, r, cc);
      const float step =
          (float)(oc.lr_muon * lrm * std::sqrt(std::max(1.0, (double)r / (double)cc)));
      if ((e = muon_update(bf, pick<float*>(w.layers[layer], kind), X + i * mn * es, r, cc,
                           r > cc, step, pick_c(w.layers_c[layer], kind), ctx)) != cudaSuccess)
        return e;
    }
    slot += cnt;
  }
  return cudaSuccess;
}

}  // namespace nc
