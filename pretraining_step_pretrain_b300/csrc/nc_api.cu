// C-ABI entry points (include/nc.h): argument validation, the workspace
// layout, and the order in which one step's kernels are enqueued.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <atomic>
#include <string>
#include <vector>

#include "../../include/nc.h"
#include "nc_common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

thread_local std::string g_last_error;

nc_status fail(nc_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
nc_status fail(nc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

#define NC_CUDA(expr)                                                                   \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(NC_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));         \
  } while (0)

// ---------------------------------------------------------------- profiling
// While on, every named launch group is bracketed by CUDA events recorded on
// the launching stream (host-side event objects only; no device memory).
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  std::vector<ProfRec> recs;
};
Profiler g_prof;

template <class F>
cudaError_t timed(const char* name, cudaStream_t stream, F&& f) {
  if (!g_prof.on || g_prof.used + 2 > g_prof.pool.size()) return f();
  cudaEvent_t a = g_prof.pool[g_prof.used++], b = g_prof.pool[g_prof.used++];
  cudaEventRecord(a, stream);
  cudaError_t e = f();
  cudaEventRecord(b, stream);
  g_prof.recs.push_back({name, a, b});
  return e;
}

#define NC_RUN(name, expr) NC_CUDA(timed(name, ctx.stream, [&]() -> cudaError_t { return (expr); }))

inline size_t al(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- validation
nc_status check_cfg(const nc_config* c, int B, int T) {
  if (!c) return fail(NC_ERR_INVALID_ARG, "cfg is null");
  if (c->dtype != NC_BF16 && c->dtype != NC_F32)
    return fail(NC_ERR_INVALID_ARG, "dtype %d is not NC_BF16 or NC_F32", c->dtype);
  if (c->depth < 1 || c->n_head < 1)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "depth %d, n_head %d must be >= 1", c->depth, c->n_head);
  if (c->d_model < 64 || c->d_model % 64)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "d_model %d must be a positive multiple of 64", c->d_model);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "head_dim %d must be 64 or 128", c->head_dim);
  if (c->dtype == NC_BF16 && c->head_dim != 128)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "bf16 mode needs head_dim 128 (got %d)", c->head_dim);
  if (c->d_mlp < 64 || c->d_mlp % 64)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "d_mlp %d must be a positive multiple of 64", c->d_mlp);
  if (c->vocab < 64 || c->vocab % 64 || c->vocab > (1 << 24))
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "vocab %d must be a multiple of 64 in [64, 2^24]", c->vocab);
  if (B < 1 || T < 1 || (long)B * T > (1L << 24))
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "B=%d T=%d: need B, T >= 1 and B*T <= 2^24", B, T);
  if ((long)T * c->n_head > kMaxAttnRowsPerSeq)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "T*n_head = %ld exceeds %ld query rows per sequence",
                (long)T * c->n_head, kMaxAttnRowsPerSeq);
  if (!(c->softcap > 0.f) || !(c->eps >= 0.f) || !(c->rope_base > 0.f))
    return fail(NC_ERR_INVALID_ARG, "softcap, rope_base must be > 0 and eps >= 0");
  return NC_OK;
}

nc_status check_ptrs(std::initializer_list<const void*> ps) {
  int i = 0;
  for (const void* p : ps) {
    if (!p) return fail(NC_ERR_INVALID_ARG, "pointer argument %d is null", i);
    if (!aligned16(p)) return fail(NC_ERR_INVALID_ARG, "pointer argument %d is not 16-byte aligned", i);
    ++i;
  }
  return NC_OK;
}

// ---------------------------------------------------------------- workspace
struct LayerBufs {
  void *xn, *q, *k, *v, *o, *xn2, *a;
  float *rstd1, *rstd_qk, *lse, *rstd2;
};

struct Layout {
  size_t total = 0;
  size_t err, rope, rope16, rstd0, x, dx, xf, rstdf, big, part, lse_row, s_tgt, loss_misc;
  size_t qkv, dx_act, dxn, du, dact, delta, split;
  size_t layer0, layer_stride;
  size_t l_xn, l_q, l_k, l_v, l_o, l_xn2, l_a, l_rstd1, l_rstd_qk, l_lse, l_rstd2;
  size_t split_elems;
  int M, n_part;
};

Layout make_layout(const nc_config& c, int B, int T) {
  Layout L;
  const size_t M = (size_t)B * T, d = c.d_model, H = c.n_head, h = c.head_dim, f = c.d_mlp,
               V = c.vocab;
  const bool bf = c.dtype == NC_BF16;
  const size_t es = bf ? 2 : 4;
  const size_t qkvw = (H + 2) * h;
  L.M = (int)M;
  L.n_part = (int)((V + kTileN - 1) / kTileN);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += al(bytes); return r; };
  L.err = take(256);
  L.rope = take(T * (h / 2) * 8);
  L.rope16 = take(T * (h / 2) * 4);
  L.rstd0 = take(M * 4);
  L.x = take(M * d * 4);
  L.dx = take(M * d * 4);
  L.xf = take(M * d * es);
  L.rstdf = take(M * 4);
  const size_t logits = M * V * es;
  L.big = take(std::max(logits, embed_bwd_scratch_bytes((int)M, (int)d)));
  L.part = take(bf ? M * L.n_part * 4 : 0);
  L.lse_row = take(M * 4);
  L.s_tgt = take(M * 4);
  L.loss_misc = take(64);
  L.qkv = take(M * qkvw * es);
  L.dx_act = take(M * d * es);
  L.dxn = take(M * d * es);
  L.du = take(M * f * es);
  L.dact = take(M * H * h * es);
  L.delta = take(M * H * 4);
  size_t se = 0;
  if (bf) {
    const int Mi = (int)M;
    se = std::max({gemm_bf16_split_elems(GEMM_TN, EPI_STORE_F32, (int)qkvw, (int)d, Mi),
                   gemm_bf16_split_elems(GEMM_TN, EPI_STORE_F32, (int)d, (int)(H * h), Mi),
                   gemm_bf16_split_elems(GEMM_TN, EPI_STORE_F32, (int)f, (int)d, Mi),
                   gemm_bf16_split_elems(GEMM_TN, EPI_STORE_F32, (int)d, (int)f, Mi),
                   gemm_bf16_split_elems(GEMM_TN, EPI_STORE_F32, (int)V, (int)d, Mi)});
  }
  L.split_elems = se;
  L.split = take(se * 4);
  L.layer0 = o;
  size_t lo = 0;
  auto ltake = [&](size_t bytes) { size_t r = lo; lo += al(bytes); return r; };
  L.l_xn = ltake(M * d * es);
  L.l_q = ltake(M * H * h * es);
  L.l_k = ltake(M * h * es);
  L.l_v = ltake(M * h * es);
  L.l_o = ltake(M * H * h * es);
  L.l_xn2 = ltake(M * d * es);
  L.l_a = ltake(M * f * es);
  L.l_rstd1 = ltake(M * 4);
  L.l_rstd_qk = ltake(M * (H + 1) * 4);
  L.l_lse = ltake(M * H * 4);
  L.l_rstd2 = ltake(M * 4);
  L.layer_stride = lo;
  L.total = L.layer0 + (size_t)c.depth * lo;
  return L;
}

template <typename T = void>
inline T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

LayerBufs layer_bufs(void* ws, const Layout& L, int layer) {
  uint8_t* base = static_cast<uint8_t*>(ws) + L.layer0 + (size_t)layer * L.layer_stride;
  LayerBufs b;
  b.xn = base + L.l_xn;
  b.q = base + L.l_q;
  b.k = base + L.l_k;
  b.v = base + L.l_v;
  b.o = base + L.l_o;
  b.xn2 = base + L.l_xn2;
  b.a = base + L.l_a;
  b.rstd1 = reinterpret_cast<float*>(base + L.l_rstd1);
  b.rstd_qk = reinterpret_cast<float*>(base + L.l_rstd_qk);
  b.lse = reinterpret_cast<float*>(base + L.l_lse);
  b.rstd2 = reinterpret_cast<float*>(base + L.l_rstd2);
  return b;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

Ctx make_ctx(void* ws, void* stream, long long timeout_ns = kWaitTimeoutNs) {
  Ctx c;
  c.stream = static_cast<cudaStream_t>(stream);
  c.err = static_cast<int*>(ws);
  c.timeout_ns = timeout_ns;
  c.num_sms = sm_count();
  return c;
}

GemmArgs gemm_args(int layout, int epi, int M, int N, int K, const void* A, long lda,
                   const void* B, long ldb, void* C, long ldc) {
  GemmArgs g;
  std::memset(&g, 0, sizeof g);
  g.layout = layout;
  g.epi = epi;
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda;
  g.B = B; g.ldb = ldb;
  g.C = C; g.ldc = ldc;
  return g;
}

cudaError_t run_gemm(bool bf16, GemmArgs g, const Layout* L, void* ws, const Ctx& ctx) {
  if (bf16 && L) {
    g.split_buf = at<float>(ws, L->split);
    g.split_buf_elems = L->split_elems;
  }
  return bf16 ? gemm_bf16(g, ctx) : gemm_f32(g, ctx);
}

// ---------------------------------------------------------------- the step's pieces
nc_status embed_fwd_impl(const nc_config& c, int B, int T, const int32_t* ids, const void* wte,
                         float* x, void* ws, const Layout& L, const Ctx& ctx) {
  const bool bf = c.dtype == NC_BF16;
  NC_CUDA(cudaMemsetAsync(ws, 0, 16, ctx.stream));
  NC_RUN("embed.rope_table", rope_table(at<float2>(ws, L.rope), at(ws, L.rope16), T, c.head_dim, c.rope_base, ctx));
  NC_RUN("embed.norm", embed_norm_fwd(bf, ids, wte, x, at<float>(ws, L.rstd0), L.M, c.d_model, c.vocab, c.eps,
                         ctx));
  return NC_OK;
}

nc_status block_fwd_impl(const nc_config& c, int layer, int B, int T, const nc_layer_w& w,
                         float* x, void* ws, const Layout& L, const Ctx& ctx) {
  const bool bf = c.dtype == NC_BF16;
  const int M = L.M, d = c.d_model, H = c.n_head, h = c.head_dim, f = c.d_mlp;
  const int qkvw = (H + 2) * h;
  LayerBufs lb = layer_bufs(ws, L, layer);
  void* qkv = at(ws, L.qkv);
  NC_RUN("fwd.norm1", rmsnorm_fwd(bf, x, lb.xn, lb.rstd1, M, d, c.eps, ctx));
  if (bf && h == 128 && T % 128 == 0) {
    // QK-norm + RoPE in the QKV GEMM's epilogue, straight into q, k, v (each
    // 128-row half tile reads 128 consecutive positions of the RoPE table).
    GemmArgs g = gemm_args(GEMM_NT, EPI_QKNORM_ROPE, M, qkvw, d, lb.xn, d, w.w_qkv, d, qkv, qkvw);
    g.qk_q = lb.q;
    g.qk_k = lb.k;
    g.qk_v = lb.v;
    g.qk_rstd = lb.rstd_qk;
    g.qk_tab = at(ws, L.rope16);
    g.qk_T = T;
    g.qk_H = H;
    g.qk_eps = c.eps;
    NC_RUN("fwd.qkv_gemm", run_gemm(bf, g, &L, ws, ctx));
  } else {
    NC_RUN("fwd.qkv_gemm", run_gemm(bf, gemm_args(GEMM_NT, EPI_STORE, M, qkvw, d, lb.xn, d, w.w_qkv, d, qkv, qkvw),
                     &L, ws, ctx));
    NC_RUN("fwd.qknorm_rope", qknorm_rope_fwd(bf, qkv, at<float2>(ws, L.rope), lb.q, lb.k, lb.v, lb.rstd_qk, B, T, H,
                            h, c.eps, ctx));
  }
  NC_RUN("fwd.attention", attention_fwd(bf, B, T, H, h, lb.q, lb.k, lb.v, lb.o, lb.lse, ctx));
  NC_RUN("fwd.out_gemm", run_gemm(bf, gemm_args(GEMM_NT, EPI_ADD_F32, M, d, H * h, lb.o, H * h, w.w_o, H * h, x, d),
                   &L, ws, ctx));
  NC_RUN("fwd.norm2", rmsnorm_fwd(bf, x, lb.xn2, lb.rstd2, M, d, c.eps, ctx));
  NC_RUN("fwd.fc_gemm", run_gemm(bf, gemm_args(GEMM_NT, EPI_RELU2, M, f, d, lb.xn2, d, w.w_fc, d, lb.a, f), &L,
                   ws, ctx));
  NC_RUN("fwd.proj_gemm", run_gemm(bf, gemm_args(GEMM_NT, EPI_ADD_F32, M, d, f, lb.a, f, w.w_proj, f, x, d), &L,
                   ws, ctx));
  return NC_OK;
}

// Final norm, logits, softcap, per-row log-sum-exp and capped target logit.
nc_status lm_fwd_impl(const nc_config& c, const float* x_L, const void* w_lm,
                      const int32_t* targets, void* ws, const Layout& L, const Ctx& ctx) {
  const bool bf = c.dtype == NC_BF16;
  const int M = L.M, d = c.d_model, V = c.vocab;
  void* xf = at(ws, L.xf);
  float* rstdf = at<float>(ws, L.rstdf);
  void* logits = at(ws, L.big);
  float* lse = at<float>(ws, L.lse_row);
  float* s_tgt = at<float>(ws, L.s_tgt);
  NC_RUN("lm.norm", rmsnorm_fwd(bf, x_L, xf, rstdf, M, d, c.eps, ctx));
  if (bf) {
    GemmArgs g = gemm_args(GEMM_NT, EPI_SOFTCAP_CE, M, V, d, xf, d, w_lm, d, logits, V);
    g.part = at<float>(ws, L.part);
    g.n_part = L.n_part;
    g.targets = targets;
    g.s_tgt = s_tgt;
    g.cap = c.softcap;
    g.group_m = 16;
    NC_CUDA(cudaMemsetAsync(s_tgt, 0, (size_t)M * 4, ctx.stream));
    NC_RUN("lm.logits_gemm", run_gemm(bf, g, &L, ws, ctx));
    NC_RUN("lm.ce_rows", ce_rows_from_partials(g.part, L.n_part, lse, M, ctx));
  } else {
    NC_RUN("lm.logits_gemm", run_gemm(bf, gemm_args(GEMM_NT, EPI_STORE, M, V, d, xf, d, w_lm, d, logits, V), &L,
                     ws, ctx));
    NC_RUN("lm.softcap_rows", softcap_rows_f32(static_cast<float*>(logits), targets, lse, s_tgt, M, V, c.softcap,
                             ctx));
  }
  return NC_OK;
}

nc_status lmhead_impl(const nc_config& c, int B, int T, const float* x_L, const void* w_lm,
                      const int32_t* targets, float* loss, float* dx_L, float* dw_lm,
                      int accumulate, void* ws, const Layout& L, const Ctx& ctx) {
  const bool bf = c.dtype == NC_BF16;
  const int M = L.M, d = c.d_model, V = c.vocab;
  void* xf = at(ws, L.xf);
  float* rstdf = at<float>(ws, L.rstdf);
  void* logits = at(ws, L.big);
  float* lse = at<float>(ws, L.lse_row);
  float* s_tgt = at<float>(ws, L.s_tgt);
  float* inv_n = at<float>(ws, L.loss_misc);
  (void)B;
  (void)T;
  nc_status st = lm_fwd_impl(c, x_L, w_lm, targets, ws, L, ctx);
  if (st != NC_OK) return st;
  NC_RUN("lm.loss", ce_loss(lse, s_tgt, targets, M, V, loss, inv_n, ctx));
  NC_RUN("lm.dlogits", ce_dlogits(bf, logits, lse, targets, inv_n, M, V, c.softcap, ctx));
  // dW_lm = G^T xf ; dxf = G W_lm
  GemmArgs gw = gemm_args(GEMM_TN, EPI_STORE_F32, V, d, M, logits, V, xf, d, dw_lm, d);
  gw.accumulate = accumulate;
  NC_RUN("lm.dw_gemm", run_gemm(bf, gw, &L, ws, ctx));
  void* dxf = at(ws, L.dxn);
  NC_RUN("lm.dx_gemm", run_gemm(bf, gemm_args(GEMM_NN, EPI_STORE, M, d, V, logits, V, w_lm, d, dxf, d), &L, ws,
                   ctx));
  NC_RUN("lm.norm_bwd", rmsnorm_bwd(bf, dxf, xf, rstdf, dx_L, at(ws, L.dx_act), 0, M, d, ctx));
  return NC_OK;
}

// dx_act (activation copy of dx) must be current on entry.
nc_status block_bwd_impl(const nc_config& c, int layer, int B, int T, const nc_layer_w& w,
                         float* dx, const nc_layer_g& g, int accumulate, void* ws,
                         const Layout& L, const Ctx& ctx) {
  const bool bf = c.dtype == NC_BF16;
  const int M = L.M, d = c.d_model, H = c.n_head, h = c.head_dim, f = c.d_mlp;
  const int qkvw = (H + 2) * h, Hh = H * h;
  LayerBufs lb = layer_bufs(ws, L, layer);
  void* dxa = at(ws, L.dx_act);
  void* du = at(ws, L.du);
  void* dxn = at(ws, L.dxn);
  void* dact = at(ws, L.dact);
  void* dqkv = at(ws, L.qkv);

  GemmArgs gw = gemm_args(GEMM_TN, EPI_STORE_F32, d, f, M, dxa, d, lb.a, f, g.d_proj, f);
  gw.accumulate = accumulate;
  NC_RUN("bwd.proj_dw_gemm", run_gemm(bf, gw, &L, ws, ctx));
  GemmArgs gd = gemm_args(GEMM_NN, EPI_RELU2_BWD, M, f, d, dxa, d, w.w_proj, f, du, f);
  gd.aux = lb.a;
  NC_RUN("bwd.proj_dx_gemm", run_gemm(bf, gd, &L, ws, ctx));
  gw = gemm_args(GEMM_TN, EPI_STORE_F32, f, d, M, du, f, lb.xn2, d, g.d_fc, d);
  gw.accumulate = accumulate;
  NC_RUN("bwd.fc_dw_gemm", run_gemm(bf, gw, &L, ws, ctx));
  NC_RUN("bwd.fc_dx_gemm", run_gemm(bf, gemm_args(GEMM_NN, EPI_STORE, M, d, f, du, f, w.w_fc, d, dxn, d), &L, ws,
                   ctx));
  NC_RUN("bwd.norm2_bwd", rmsnorm_bwd(bf, dxn, lb.xn2, lb.rstd2, dx, dxa, 1, M, d, ctx));

  gw = gemm_args(GEMM_TN, EPI_STORE_F32, d, Hh, M, dxa, d, lb.o, Hh, g.d_o, Hh);
  gw.accumulate = accumulate;
  NC_RUN("bwd.out_dw_gemm", run_gemm(bf, gw, &L, ws, ctx));
  NC_RUN("bwd.out_dx_gemm", run_gemm(bf, gemm_args(GEMM_NN, EPI_STORE, M, Hh, d, dxa, d, w.w_o, Hh, dact, Hh), &L,
                   ws, ctx));
  uint8_t* dq = static_cast<uint8_t*>(dqkv);
  const size_t es = bf ? 2 : 4;
  NC_RUN("bwd.attention", attention_bwd(bf, B, T, H, h, lb.q, lb.k, lb.v, lb.o, lb.lse, dact, dq, qkvw,
                        dq + (size_t)Hh * es, qkvw, dq + (size_t)(Hh + h) * es, qkvw,
                        at<float>(ws, L.delta), ctx));
  NC_RUN("bwd.qknorm_rope", qknorm_rope_bwd(bf, dqkv, lb.q, lb.k, lb.rstd_qk, at<float2>(ws, L.rope), B, T, H, h,
                          ctx));
  gw = gemm_args(GEMM_TN, EPI_STORE_F32, qkvw, d, M, dqkv, qkvw, lb.xn, d, g.d_qkv, d);
  gw.accumulate = accumulate;
  NC_RUN("bwd.qkv_dw_gemm", run_gemm(bf, gw, &L, ws, ctx));
  NC_RUN("bwd.qkv_dx_gemm", run_gemm(bf, gemm_args(GEMM_NN, EPI_STORE, M, d, qkvw, dqkv, qkvw, w.w_qkv, d, dxn, d),
                   &L, ws, ctx));
  NC_RUN("bwd.norm1_bwd", rmsnorm_bwd(bf, dxn, lb.xn, lb.rstd1, dx, dxa, 1, M, d, ctx));
  return NC_OK;
}

nc_status embed_bwd_impl(const nc_config& c, int B, int T, const int32_t* ids, const void* wte,
                         const float* dx, float* dwte, int accumulate, void* ws, const Layout& L,
                         const Ctx& ctx) {
  NC_RUN("embed_bwd", embed_norm_bwd(c.dtype == NC_BF16, ids, wte, at<float>(ws, L.rstd0), dx, dwte,
                         accumulate, L.M, c.d_model, c.vocab, at(ws, L.big), ctx));
  return NC_OK;
}

nc_status check_ws(const nc_config* cfg, int B, int T, void* ws, size_t ws_bytes, Layout* L) {
  nc_status s = check_cfg(cfg, B, T);
  if (s != NC_OK) return s;
  if (!ws) return fail(NC_ERR_INVALID_ARG, "workspace is null");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(NC_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  *L = make_layout(*cfg, B, T);
  if (ws_bytes < L->total)
    return fail(NC_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, L->total);
  return NC_OK;
}

__global__ void selftest_wait_kernel(int* err, long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, &abort_flag, err, 900, timeout_ns);
}

}  // namespace

std::atomic<long long> g_launches{0};
void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

cudaError_t selftest_wait(long long timeout_ns, const Ctx& ctx) {
  selftest_wait_kernel<<<1, 32, 0, ctx.stream>>>(ctx.err, timeout_ns);
  return launched(1);
}

}  // namespace nc

using namespace nc;

extern "C" {

size_t nc_workspace_bytes(const nc_config* cfg, int B, int T) {
  if (check_cfg(cfg, B, T) != NC_OK) return 0;
  return make_layout(*cfg, B, T).total;
}

nc_status nc_embed_norm(const nc_config* cfg, int B, int T, const int32_t* ids, const void* wte,
                        float* x, void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  nc_status s = check_ws(cfg, B, T, ws, ws_bytes, &L);
  if (s == NC_OK) s = check_ptrs({ids, wte, x});
  if (s != NC_OK) return s;
  return embed_fwd_impl(*cfg, B, T, ids, wte, x, ws, L, make_ctx(ws, stream));
}

nc_status nc_block_fwd(const nc_config* cfg, int layer, int B, int T, const nc_layer_w* w,
                       float* x, void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  nc_status s = check_ws(cfg, B, T, ws, ws_bytes, &L);
  if (s != NC_OK) return s;
  if (!w) return fail(NC_ERR_INVALID_ARG, "layer weights are null");
  if (layer < 0 || layer >= cfg->depth)
    return fail(NC_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, cfg->depth);
  if ((s = check_ptrs({w->w_qkv, w->w_o, w->w_fc, w->w_proj, x})) != NC_OK) return s;
  return block_fwd_impl(*cfg, layer, B, T, *w, x, ws, L, make_ctx(ws, stream));
}

nc_status nc_lmhead_softcap_ce_fwd_bwd(const nc_config* cfg, int B, int T, const float* x_L,
                                       const void* w_lm, const int32_t* targets, float* loss,
                                       float* dx_L, float* dw_lm, int accumulate, void* ws,
                                       size_t ws_bytes, void* stream) {
  Layout L;
  nc_status s = check_ws(cfg, B, T, ws, ws_bytes, &L);
  if (s == NC_OK) s = check_ptrs({x_L, w_lm, targets, dx_L, dw_lm});
  if (s != NC_OK) return s;
  if (!loss || (reinterpret_cast<uintptr_t>(loss) & 3u))
    return fail(NC_ERR_INVALID_ARG, "loss pointer is null or misaligned");
  return lmhead_impl(*cfg, B, T, x_L, w_lm, targets, loss, dx_L, dw_lm, accumulate != 0, ws, L,
                     make_ctx(ws, stream));
}

nc_status nc_block_bwd(const nc_config* cfg, int layer, int B, int T, const nc_layer_w* w,
                       float* dx, const nc_layer_g* g, int accumulate, void* ws, size_t ws_bytes,
                       void* stream) {
  Layout L;
  nc_status s = check_ws(cfg, B, T, ws, ws_bytes, &L);
  if (s != NC_OK) return s;
  if (!w || !g) return fail(NC_ERR_INVALID_ARG, "layer weights or gradients are null");
  if (layer < 0 || layer >= cfg->depth)
    return fail(NC_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, cfg->depth);
  if ((s = check_ptrs({w->w_qkv, w->w_o, w->w_fc, w->w_proj, dx, g->d_qkv, g->d_o, g->d_fc,
                       g->d_proj})) != NC_OK)
    return s;
  Ctx ctx = make_ctx(ws, stream);
  const bool bf = cfg->dtype == NC_BF16;
  NC_CUDA(cast_f32_to_act(bf, dx, at(ws, L.dx_act), (long)L.M * cfg->d_model, ctx));
  return block_bwd_impl(*cfg, layer, B, T, *w, dx, *g, accumulate != 0, ws, L, ctx);
}

nc_status nc_embed_norm_bwd(const nc_config* cfg, int B, int T, const int32_t* ids,
                            const void* wte, const float* dx, float* dwte, int accumulate,
                            void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  nc_status s = check_ws(cfg, B, T, ws, ws_bytes, &L);
  if (s == NC_OK) s = check_ptrs({ids, wte, dx, dwte});
  if (s != NC_OK) return s;
  return embed_bwd_impl(*cfg, B, T, ids, wte, dx, dwte, accumulate != 0, ws, L,
                        make_ctx(ws, stream));
}

nc_status nc_step(const nc_config* cfg, int B, int T, const int32_t* ids, const int32_t* targets,
                  const void* wte, const nc_layer_w* layers, const void* w_lm, float* loss,
                  float* dwte, const nc_layer_g* grads, float* dw_lm, int accumulate, void* ws,
                  size_t ws_bytes, void* stream) {
  Layout L;
  nc_status s = check_ws(cfg, B, T, ws, ws_bytes, &L);
  if (s == NC_OK) s = check_ptrs({ids, targets, wte, w_lm, dwte, dw_lm});
  if (s != NC_OK) return s;
  if (!layers || !grads) return fail(NC_ERR_INVALID_ARG, "layers or grads array is null");
  if (!loss || (reinterpret_cast<uintptr_t>(loss) & 3u))
    return fail(NC_ERR_INVALID_ARG, "loss pointer is null or misaligned");
  for (int l = 0; l < cfg->depth; ++l) {
    if ((s = check_ptrs({layers[l].w_qkv, layers[l].w_o, layers[l].w_fc, layers[l].w_proj,
                         grads[l].d_qkv, grads[l].d_o, grads[l].d_fc, grads[l].d_proj})) != NC_OK)
      return fail(s, "layer %d: %s", l, g_last_error.c_str());
  }
  const Ctx ctx = make_ctx(ws, stream);
  float* x = at<float>(ws, L.x);
  float* dx = at<float>(ws, L.dx);
  accumulate = accumulate != 0;
  if ((s = embed_fwd_impl(*cfg, B, T, ids, wte, x, ws, L, ctx)) != NC_OK) return s;
  for (int l = 0; l < cfg->depth; ++l)
    if ((s = block_fwd_impl(*cfg, l, B, T, layers[l], x, ws, L, ctx)) != NC_OK) return s;
  if ((s = lmhead_impl(*cfg, B, T, x, w_lm, targets, loss, dx, dw_lm, accumulate, ws, L, ctx)) !=
      NC_OK)
    return s;
  for (int l = cfg->depth - 1; l >= 0; --l)
    if ((s = block_bwd_impl(*cfg, l, B, T, layers[l], dx, grads[l], accumulate, ws, L, ctx)) !=
        NC_OK)
      return s;
  return embed_bwd_impl(*cfg, B, T, ids, wte, dx, dwte, accumulate, ws, L, ctx);
}

nc_status nc_eval(const nc_config* cfg, int B, int T, const int32_t* ids, const int32_t* targets,
                  const int32_t* token_bytes, const void* wte, const nc_layer_w* layers,
                  const void* w_lm, float* out, void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  nc_status s = check_ws(cfg, B, T, ws, ws_bytes, &L);
  if (s == NC_OK) s = check_ptrs({ids, targets, wte, w_lm});
  if (s != NC_OK) return s;
  if (!layers) return fail(NC_ERR_INVALID_ARG, "layers array is null");
  if (!out || (reinterpret_cast<uintptr_t>(out) & 7u))
    return fail(NC_ERR_INVALID_ARG, "out pointer is null or not 8-byte aligned");
  if (token_bytes && (reinterpret_cast<uintptr_t>(token_bytes) & 3u))
    return fail(NC_ERR_INVALID_ARG, "token_bytes is misaligned");
  for (int l = 0; l < cfg->depth; ++l) {
    if ((s = check_ptrs({layers[l].w_qkv, layers[l].w_o, layers[l].w_fc, layers[l].w_proj})) !=
        NC_OK)
      return fail(s, "layer %d: %s", l, g_last_error.c_str());
  }
  const Ctx ctx = make_ctx(ws, stream);
  float* x = at<float>(ws, L.x);
  if ((s = embed_fwd_impl(*cfg, B, T, ids, wte, x, ws, L, ctx)) != NC_OK) return s;
  for (int l = 0; l < cfg->depth; ++l)
    if ((s = block_fwd_impl(*cfg, l, B, T, layers[l], x, ws, L, ctx)) != NC_OK) return s;
  if ((s = lm_fwd_impl(*cfg, x, w_lm, targets, ws, L, ctx)) != NC_OK) return s;
  NC_RUN("eval.loss", eval_loss(at<float>(ws, L.lse_row), at<float>(ws, L.s_tgt), targets,
                                token_bytes, L.M, cfg->vocab, out, ctx));
  return NC_OK;
}

nc_status nc_get_device_status(void* ws, void* stream) {
  if (!ws) return fail(NC_ERR_INVALID_ARG, "workspace is null");
  int word[4] = {0, 0, 0, 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  NC_CUDA(cudaStreamSynchronize(st));
  NC_CUDA(cudaMemcpy(word, ws, 16, cudaMemcpyDeviceToHost));
  NC_CUDA(cudaMemset(ws, 0, 16));
  if (word[0] == NC_OK) return NC_OK;
  return fail(static_cast<nc_status>(word[0]), "device reported %s at site %d (detail %d)",
              nc_status_string(static_cast<nc_status>(word[0])), word[1], word[2]);
}

const char* nc_status_string(nc_status s) {
  switch (s) {
    case NC_OK: return "NC_OK";
    case NC_ERR_INVALID_ARG: return "NC_ERR_INVALID_ARG";
    case NC_ERR_UNSUPPORTED_SHAPE: return "NC_ERR_UNSUPPORTED_SHAPE";
    case NC_ERR_WORKSPACE: return "NC_ERR_WORKSPACE";
    case NC_ERR_CUDA: return "NC_ERR_CUDA";
    case NC_ERR_TIMEOUT: return "NC_ERR_TIMEOUT";
    case NC_ERR_TOKEN_RANGE: return "NC_ERR_TOKEN_RANGE";
  }
  return "NC_ERR_UNKNOWN";
}

const char* nc_last_error_message(void) { return g_last_error.c_str(); }

size_t nc_gemm_workspace_bytes(int dtype, int layout, int M, int N, int K) {
  if (dtype != NC_BF16) return 256;
  return 256 + al(gemm_bf16_split_elems(layout, EPI_STORE_F32, M, N, K) * 4);
}

nc_status nc_gemm(int dtype, int layout, int epilogue, int M, int N, int K, const void* A, int lda,
                  const void* Bm, int ldb, void* C, int ldc, const void* aux, int accumulate,
                  void* ws, size_t ws_bytes, void* stream) {
  if (dtype != NC_BF16 && dtype != NC_F32) return fail(NC_ERR_INVALID_ARG, "bad dtype %d", dtype);
  if (layout < NC_GEMM_NT || layout > NC_GEMM_TN)
    return fail(NC_ERR_INVALID_ARG, "bad layout %d", layout);
  if (epilogue < NC_EPI_STORE || epilogue > NC_EPI_RELU2_BWD)
    return fail(NC_ERR_INVALID_ARG, "bad epilogue %d", epilogue);
  if (M < 1 || N < 1 || K < 1 || N % 32)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "M=%d N=%d K=%d: need >= 1 and N %% 32 == 0", M, N, K);
  if (lda % 8 || ldb % 8 || ldc % 8)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "leading dimensions must be multiples of 8");
  const long a_min = layout == NC_GEMM_TN ? M : K;
  const long b_min = layout == NC_GEMM_NT ? K : N;
  if (lda < a_min || ldb < b_min || ldc < N)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "leading dimension smaller than the row length");
  nc_status s = check_ptrs({A, Bm, C, ws});
  if (s != NC_OK) return s;
  if (epilogue == NC_EPI_RELU2_BWD && ((s = check_ptrs({aux})) != NC_OK)) return s;
  if (ws_bytes < nc_gemm_workspace_bytes(dtype, layout, M, N, K))
    return fail(NC_ERR_WORKSPACE, "gemm workspace too small");
  if (epilogue == NC_EPI_STORE_F32 && dtype == NC_BF16 &&
      gemm_bf16_split_elems(layout, EPI_STORE_F32, M, N, K) > 0 && ldc != N)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "split-K fp32 output needs ldc == N");
  GemmArgs g = gemm_args(layout, epilogue, M, N, K, A, lda, Bm, ldb, C, ldc);
  g.aux = aux;
  g.accumulate = accumulate != 0;
  g.split_buf = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  g.split_buf_elems = (ws_bytes - 256) / 4;
  const Ctx ctx = make_ctx(ws, stream);
  cudaError_t e = dtype == NC_BF16 ? gemm_bf16(g, ctx) : gemm_f32(g, ctx);
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
  return NC_OK;
}

nc_status nc_gemm_fp8(int M, int N, int K, const void* A, int lda, const void* Bm, int ldb,
                      int out_dtype, void* C, int ldc, float scale, void* ws, size_t ws_bytes,
                      void* stream) {
  if (out_dtype != NC_BF16 && out_dtype != NC_F32)
    return fail(NC_ERR_INVALID_ARG, "bad output dtype %d", out_dtype);
  if (M < 1 || N < 1 || K < 1 || N % 32 || K % 16)
    return fail(NC_ERR_UNSUPPORTED_SHAPE,
                "M=%d N=%d K=%d: need >= 1, N %% 32 == 0 and K %% 16 == 0", M, N, K);
  if (lda % 16 || ldb % 16 || ldc % 8)
    return fail(NC_ERR_UNSUPPORTED_SHAPE,
                "lda, ldb must be multiples of 16 and ldc a multiple of 8");
  if (lda < K || ldb < K || ldc < N)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "leading dimension smaller than the row length");
  if (!std::isfinite(scale)) return fail(NC_ERR_INVALID_ARG, "scale must be finite");
  nc_status s = check_ptrs({A, Bm, C, ws});
  if (s != NC_OK) return s;
  if (ws_bytes < 256) return fail(NC_ERR_WORKSPACE, "gemm workspace too small");
  GemmArgs g = gemm_args(NC_GEMM_NT, NC_EPI_STORE, M, N, K, A, lda, Bm, ldb, C, ldc);
  const Ctx ctx = make_ctx(ws, stream);
  cudaError_t e = gemm_fp8(g, out_dtype == NC_F32, scale, ctx);
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "fp8 gemm launch: %s", cudaGetErrorString(e));
  return NC_OK;
}

nc_status nc_gemm_batched(int dtype, int layout, int epilogue, int batch, int M, int N, int K,
                          const void* A, int lda, long a_bstride, const void* Bm, int ldb,
                          long b_bstride, void* C, int ldc, long c_bstride, const void* aux,
                          float alpha, float beta, void* ws, size_t ws_bytes, void* stream) {
  if (dtype != NC_BF16 && dtype != NC_F32) return fail(NC_ERR_INVALID_ARG, "bad dtype %d", dtype);
  if (layout < NC_GEMM_NT || layout > NC_GEMM_TN)
    return fail(NC_ERR_INVALID_ARG, "bad layout %d", layout);
  if (epilogue != NC_EPI_STORE && epilogue != NC_EPI_AXPBY)
    return fail(NC_ERR_INVALID_ARG, "batched epilogue %d is not STORE or AXPBY", epilogue);
  if (batch < 1 || M < 1 || N < 1 || K < 1 || N % 32)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "batch=%d M=%d N=%d K=%d: need >= 1 and N %% 32 == 0",
                batch, M, N, K);
  if (lda % 8 || ldb % 8 || ldc % 8 || a_bstride % 8 || b_bstride % 8 || c_bstride % 8)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "leading dimensions and batch strides must be multiples of 8");
  const long a_min = layout == NC_GEMM_TN ? M : K;
  const long b_min = layout == NC_GEMM_NT ? K : N;
  if (lda < a_min || ldb < b_min || ldc < N)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "leading dimension smaller than the row length");
  const long a_rows = layout == NC_GEMM_TN ? K : M, b_rows = layout == NC_GEMM_NT ? N : K;
  if (batch > 1 && (a_bstride < a_rows * lda || b_bstride < b_rows * ldb || c_bstride < (long)M * ldc))
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "batch entries overlap (stride smaller than a matrix)");
  nc_status s = check_ptrs({A, Bm, C, ws});
  if (s != NC_OK) return s;
  if (epilogue == NC_EPI_AXPBY && ((s = check_ptrs({aux})) != NC_OK)) return s;
  if (ws_bytes < 256) return fail(NC_ERR_WORKSPACE, "gemm workspace too small");
  GemmArgs g = gemm_args(layout, epilogue, M, N, K, A, lda, Bm, ldb, C, ldc);
  g.aux = aux;
  g.batch = batch;
  g.a_bstride = a_bstride;
  g.b_bstride = b_bstride;
  g.c_bstride = c_bstride;
  g.alpha = alpha;
  g.beta = beta;
  const Ctx ctx = make_ctx(ws, stream);
  cudaError_t e = dtype == NC_BF16 ? gemm_bf16(g, ctx) : gemm_f32(g, ctx);
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
  return NC_OK;
}

size_t nc_optimizer_workspace_bytes(const nc_config* cfg) {
  if (!cfg || check_cfg(cfg, 1, 1) != NC_OK) return 0;
  return optimizer_ws_bytes(*cfg);
}

nc_status nc_optimizer_step(const nc_config* cfg, const nc_opt_config* oc, int t, float lrm,
                            float* wte, float* w_lm, const nc_layer_f* layers, void* wte_c,
                            void* w_lm_c, const nc_layer_wc* layers_c, const float* dwte,
                            const float* dw_lm, const nc_layer_g* grads, float* m_wte,
                            float* v_wte, float* m_lm, float* v_lm,
                            const nc_layer_f* momentum_bufs, void* ws, size_t ws_bytes,
                            void* stream) {
  nc_status s = check_cfg(cfg, 1, 1);
  if (s != NC_OK) return s;
  if (!oc || !layers || !layers_c || !grads || !momentum_bufs)
    return fail(NC_ERR_INVALID_ARG, "null optimizer config or per-layer array");
  if (t < 1) return fail(NC_ERR_INVALID_ARG, "optimizer step t=%d must be >= 1", t);
  if (oc->ns_steps < 0 || oc->ns_steps > 64)
    return fail(NC_ERR_INVALID_ARG, "ns_steps %d outside [0, 64]", oc->ns_steps);
  if (!(oc->beta1 >= 0.f && oc->beta1 < 1.f) || !(oc->beta2 >= 0.f && oc->beta2 < 1.f) ||
      !(oc->eps > 0.f))
    return fail(NC_ERR_INVALID_ARG, "AdamW betas must lie in [0, 1) and eps > 0");
  if ((s = check_ptrs({wte, w_lm, wte_c, w_lm_c, dwte, dw_lm, m_wte, v_wte, m_lm, v_lm, ws})) !=
      NC_OK)
    return s;
  for (int l = 0; l < cfg->depth; ++l) {
    const nc_layer_f& p = layers[l];
    const nc_layer_wc& c = layers_c[l];
    const nc_layer_g& g = grads[l];
    const nc_layer_f& m = momentum_bufs[l];
    if ((s = check_ptrs({p.w_qkv, p.w_o, p.w_fc, p.w_proj, c.w_qkv, c.w_o, c.w_fc, c.w_proj,
                         g.d_qkv, g.d_o, g.d_fc, g.d_proj, m.w_qkv, m.w_o, m.w_fc, m.w_proj})) !=
        NC_OK) {
      const std::string why = nc_last_error_message();
      return fail(s, "layer %d: %s", l, why.c_str());
    }
  }
  if (ws_bytes < optimizer_ws_bytes(*cfg)) return fail(NC_ERR_WORKSPACE, "optimizer workspace too small");
  OptTensors w;
  w.wte = wte;
  w.w_lm = w_lm;
  w.layers = layers;
  w.wte_c = wte_c;
  w.w_lm_c = w_lm_c;
  w.layers_c = layers_c;
  w.dwte = dwte;
  w.dw_lm = dw_lm;
  w.grads = grads;
  w.m_wte = m_wte;
  w.v_wte = v_wte;
  w.m_lm = m_lm;
  w.v_lm = v_lm;
  w.mom = momentum_bufs;
  const Ctx ctx = make_ctx(ws, stream);
  cudaError_t e = optimizer_step(*cfg, *oc, t, lrm, w, ws, ctx);
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "optimizer launch: %s", cudaGetErrorString(e));
  return NC_OK;
}

long long nc_launch_count(void) { return g_launches.load(); }

nc_status nc_profile_start(int max_records) {
  if (max_records < 1 || max_records > (1 << 20))
    return fail(NC_ERR_INVALID_ARG, "max_records %d outside [1, 2^20]", max_records);
  for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
  g_prof.pool.clear();
  g_prof.recs.clear();
  g_prof.used = 0;
  for (int i = 0; i < 2 * max_records; ++i) {
    cudaEvent_t e;
    NC_CUDA(cudaEventCreate(&e));
    g_prof.pool.push_back(e);
  }
  g_prof.on = true;
  return NC_OK;
}

int nc_profile_stop(void) {
  g_prof.on = false;
  return (int)g_prof.recs.size();
}

nc_status nc_profile_record(int i, const char** name, float* ms) {
  if (i < 0 || i >= (int)g_prof.recs.size() || !name || !ms)
    return fail(NC_ERR_INVALID_ARG, "record %d out of range", i);
  const ProfRec& r = g_prof.recs[i];
  NC_CUDA(cudaEventSynchronize(r.b));
  NC_CUDA(cudaEventElapsedTime(ms, r.a, r.b));
  *name = r.name;
  return NC_OK;
}

size_t nc_attention_workspace_bytes(int B, int T, int H) {
  return 256 + al(attention_scratch_bytes(B, T, H));
}

static nc_status check_attn(int dtype, int B, int T, int H, int h) {
  if (dtype != NC_BF16 && dtype != NC_F32) return fail(NC_ERR_INVALID_ARG, "bad dtype %d", dtype);
  if (B < 1 || T < 1 || H < 1 || (long)B * T * H > (1L << 28))
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "bad B/T/H");
  if ((long)T * H > kMaxAttnRowsPerSeq)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "T*H = %ld exceeds %ld query rows per sequence",
                (long)T * H, kMaxAttnRowsPerSeq);
  if (h != 128 && !(dtype == NC_F32 && h == 64))
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "head_dim %d unsupported for this dtype", h);
  return NC_OK;
}

nc_status nc_attention_fwd(int dtype, int B, int T, int H, int h, const void* q, const void* k,
                           const void* v, void* o, float* lse, void* ws, size_t ws_bytes,
                           void* stream) {
  nc_status s = check_attn(dtype, B, T, H, h);
  if (s == NC_OK) s = check_ptrs({q, k, v, o, lse, ws});
  if (s != NC_OK) return s;
  if (ws_bytes < nc_attention_workspace_bytes(B, T, H))
    return fail(NC_ERR_WORKSPACE, "attention workspace too small");
  cudaError_t e = attention_fwd(dtype == NC_BF16, B, T, H, h, q, k, v, o, lse, make_ctx(ws, stream));
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "attention fwd: %s", cudaGetErrorString(e));
  return NC_OK;
}

nc_status nc_attention_bwd(int dtype, int B, int T, int H, int h, const void* q, const void* k,
                           const void* v, const void* o, const float* lse, const void* dout,
                           void* dq, int ldq, void* dk, int ldk, void* dv, int ldv, void* ws,
                           size_t ws_bytes, void* stream) {
  nc_status s = check_attn(dtype, B, T, H, h);
  if (s == NC_OK) s = check_ptrs({q, k, v, o, lse, dout, dq, dk, dv, ws});
  if (s != NC_OK) return s;
  if (ldq < H * h || ldk < h || ldv < h || ldq % 8 || ldk % 8 || ldv % 8)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "bad gradient row strides");
  if (ws_bytes < nc_attention_workspace_bytes(B, T, H))
    return fail(NC_ERR_WORKSPACE, "attention workspace too small");
  float* delta = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  cudaError_t e = attention_bwd(dtype == NC_BF16, B, T, H, h, q, k, v, o, lse, dout, dq, ldq, dk,
                                ldk, dv, ldv, delta, make_ctx(ws, stream));
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "attention bwd: %s", cudaGetErrorString(e));
  return NC_OK;
}

nc_status nc_attention_bwd_noalloc(int dtype, int B, int T, int H, int h, const void* q,
                                   const void* k, const void* v, const void* o, const float* lse,
                                   const void* dout, void* dq, int ldq, void* dk, int ldk,
                                   void* dv, int ldv, void* stream) {
  nc_status s = check_attn(dtype, B, T, H, h);
  if (s == NC_OK) s = check_ptrs({q, k, v, o, lse, dout, dq, dk, dv});
  if (s != NC_OK) return s;
  if (ldq < H * h || ldk < h || ldv < h || ldq % 8 || ldk % 8 || ldv % 8)
    return fail(NC_ERR_UNSUPPORTED_SHAPE, "bad gradient row strides");
  if ((long)B * T * H > kNoAllocAttnMaxRows)
    return fail(NC_ERR_UNSUPPORTED_SHAPE,
                "B*T*H = %ld query rows exceeds the fixed scratch of this entry point (%ld rows); "
                "use nc_attention_bwd with a workspace",
                (long)B * T * H, kNoAllocAttnMaxRows);
  Ctx ctx;
  ctx.stream = static_cast<cudaStream_t>(stream);
  ctx.err = nullptr;  // replaced by the library's own error word of the no-alloc calls
  ctx.timeout_ns = kWaitTimeoutNs;
  ctx.num_sms = sm_count();
  cudaError_t e = attention_bwd_noalloc(dtype == NC_BF16, B, T, H, h, q, k, v, o, lse, dout, dq,
                                        ldq, dk, ldk, dv, ldv, ctx);
  if (e != cudaSuccess)
    return fail(NC_ERR_CUDA, "attention bwd (no-alloc): %s", cudaGetErrorString(e));
  return NC_OK;
}

nc_status nc_attention_bwd_noalloc_status(void* stream) {
  int word[4] = {0, 0, 0, 0};
  cudaError_t e = noalloc_read_status(static_cast<cudaStream_t>(stream), word);
  if (e != cudaSuccess)
    return fail(NC_ERR_CUDA, "reading the no-alloc error word: %s", cudaGetErrorString(e));
  if (word[0] == NC_OK) return NC_OK;
  return fail(static_cast<nc_status>(word[0]), "device reported %s at site %d (detail %d)",
              nc_status_string(static_cast<nc_status>(word[0])), word[1], word[2]);
}

nc_status nc_selftest_wait_timeout(int timeout_us, void* ws, size_t ws_bytes, void* stream) {
  if ((ws && ws_bytes < 16) || timeout_us < 1 || timeout_us > 10000000)
    return fail(NC_ERR_INVALID_ARG, "bad selftest arguments");
  Ctx ctx = make_ctx(ws, stream, (long long)timeout_us * 1000);
  if (!ws) {
    cudaError_t e = noalloc_error_word(&ctx.err);
    if (e != cudaSuccess) return fail(NC_ERR_CUDA, "no-alloc error word: %s", cudaGetErrorString(e));
  }
  cudaError_t e = selftest_wait(ctx.timeout_ns, ctx);
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
  return NC_OK;
}

}  // extern "C"
