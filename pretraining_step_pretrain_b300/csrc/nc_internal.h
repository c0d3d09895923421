// Internal launcher interface between the C-ABI host code and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "nc.h"

namespace nc {

struct Ctx {
  cudaStream_t stream;
  int* err;               // device error word (start of the workspace)
  long long timeout_ns;   // limit of every device spin-wait
  int num_sms;
};

// Host-side count of kernel launches issued by the library (nc_launch_count).
void note_launch(int n);
inline cudaError_t launched(int n) {
  note_launch(n);
  return cudaGetLastError();
}

// Query rows (tokens x heads) of one sequence that the attention kernels
// accept: their 128-row tiles are indexed by the grid's y dimension (at most
// 65535, and the forward launches whole CTA pairs).
constexpr long kMaxAttnRowsPerSeq = 65534L * 128;

enum GemmLayout { GEMM_NT = 0, GEMM_NN = 1, GEMM_TN = 2 };
enum GemmEpi { EPI_STORE = 0, EPI_STORE_F32 = 1, EPI_ADD_F32 = 2, EPI_RELU2 = 3,
               EPI_RELU2_BWD = 4, EPI_SOFTCAP_CE = 5, EPI_AXPBY = 6, EPI_QKNORM_ROPE = 7 };

struct GemmArgs {
  int layout, epi;
  int M, N, K;
  const void* A; long lda;
  const void* B; long ldb;
  void* C; long ldc;
  const void* aux;        // RELU2_BWD: saved relu(u)^2, same layout as C
  int accumulate;         // STORE_F32: add into C
  // SOFTCAP_CE (tensor-core path only)
  float* part; int n_part; const int* targets; float* s_tgt; float cap;
  // STORE_F32 split-K slabs (tensor-core path); may be null when not needed
  float* split_buf; size_t split_buf_elems;
  int group_m;            // m-tiles per raster group (0 = default)
  // Batched GEMM: `batch` independent products (0 or 1 = one); entry z uses
  // A + z a_bstride, B + z b_bstride, C + z c_bstride, aux + z c_bstride
  // (element strides).  Not combined with split-K.
  int batch;
  long a_bstride, b_bstride, c_bstride;
  float alpha, beta;      // AXPBY: C = alpha * aux + beta * acc
  // QKNORM_ROPE (tensor-core path, head_dim 128): the QKV product's heads go
  // normalised and rotated to q (M, H 128), k, v (M, 128); rstd_qk (M, H + 1)
  void *qk_q, *qk_k, *qk_v;
  float* qk_rstd;
  const void* qk_tab;     // fp16 pairs (T, 64): cos, sin
  int qk_T, qk_H;
  float qk_eps;
};

// bf16 tensor map with 128-byte swizzle and zero fill out of range.  dims[0]
// is the contiguous extent; strides_bytes has rank - 1 entries.
bool make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

// Tensor-core (bf16) path.
constexpr int kTileN = 256;            // n-tile width (per-row CE partials)
size_t gemm_bf16_split_elems(int layout, int epi, int M, int N, int K);
cudaError_t gemm_bf16(const GemmArgs& g, const Ctx& ctx);
// E4M3 operands (layout NT, K-major raw bytes), C = scale * A B^T, bf16 or fp32 out.
cudaError_t gemm_fp8(const GemmArgs& g, bool out_f32, float scale, const Ctx& ctx);
// fp32 SIMT path (debug / parity mode).
cudaError_t gemm_f32(const GemmArgs& g, const Ctx& ctx);

// ---- memory-bound kernels (act = bf16 or float) ----
// Each takes `bf16` to pick the activation type.
// cos, sin of t theta_i for t < T, i < h/2: float2 (T, h/2) in `tab`, and the
// same as fp16 pairs in `tab16` (may be null) for the QKV epilogue.
cudaError_t rope_table(float2* tab, void* tab16, int T, int h, float base, const Ctx& ctx);
cudaError_t embed_norm_fwd(bool bf16, const int* ids, const void* wte, float* x, float* rstd,
                           int M, int d, int V, float eps, const Ctx& ctx);
cudaError_t rmsnorm_fwd(bool bf16, const float* x, void* y, float* rstd, int M, int d, float eps,
                        const Ctx& ctx);
cudaError_t rmsnorm_bwd(bool bf16, const void* dy, const void* y, const float* rstd, float* dx,
                        void* dx_act, int add, int M, int d, const Ctx& ctx);
cudaError_t cast_f32_to_act(bool bf16, const float* x, void* y, long n, const Ctx& ctx);
cudaError_t qknorm_rope_fwd(bool bf16, const void* qkv, const float2* tab, void* q, void* k,
                            void* v, float* rstd_qk, int B, int T, int H, int h, float eps,
                            const Ctx& ctx);
cudaError_t qknorm_rope_bwd(bool bf16, void* dqkv, const void* q, const void* k,
                            const float* rstd_qk, const float2* tab, int B, int T, int H, int h,
                            const Ctx& ctx);
cudaError_t splitk_reduce(float* c, const float* slabs, int splits, long n, int accumulate,
                          const Ctx& ctx);

// ---- attention ----
size_t attention_scratch_bytes(int B, int T, int H);
cudaError_t attention_fwd(bool bf16, int B, int T, int H, int h, const void* q, const void* k,
                          const void* v, void* o, float* lse, const Ctx& ctx);
cudaError_t attention_bwd(bool bf16, int B, int T, int H, int h, const void* q, const void* k,
                          const void* v, const void* o, const float* lse, const void* dout,
                          void* dq, long ldq, void* dk, long ldk, void* dv, long ldv,
                          float* delta_scratch, const Ctx& ctx);

// tcgen05 kernels behind the bf16 path (attention_tc.cu), head dim 128.
cudaError_t attention_fwd_tc(int B, int T, int H, const void* q, const void* k, const void* v,
                             void* o, float* lse, const Ctx& ctx);
cudaError_t attention_bwd_tc(int B, int T, int H, const void* q, const void* k, const void* v,
                             const void* o, const float* lse, const void* dout, void* dq,
                             long ldq, void* dk, long ldk, void* dv, long ldv, float* delta,
                             const Ctx& ctx);
// Allocation-free variant: delta lives in a fixed device array of the library
// (at most kNoAllocAttnMaxRows = B*T*H rows); see attention.cu.
constexpr long kNoAllocAttnMaxRows = 1L << 21;
cudaError_t attention_bwd_noalloc(bool bf16, int B, int T, int H, int h, const void* q,
                                  const void* k, const void* v, const void* o, const float* lse,
                                  const void* dout, void* dq, long ldq, void* dk, long ldk,
                                  void* dv, long ldv, const Ctx& ctx);
// The allocation-free calls' device error word (a fixed device array of the
// library, like their scratch): its address on the current device, and a
// synchronising read that clears it.
cudaError_t noalloc_error_word(int** err);
cudaError_t noalloc_read_status(cudaStream_t stream, int word[4]);

// ---- loss ----
cudaError_t softcap_rows_f32(float* s, const int* targets, float* lse, float* s_tgt, int M,
                             int V, float cap, const Ctx& ctx);
cudaError_t ce_rows_from_partials(const float* part, int n_part, float* lse, int M,
                                  const Ctx& ctx);
cudaError_t ce_loss(const float* lse, const float* s_tgt, const int* targets, int M, int V,
                    float* loss, float* inv_n, const Ctx& ctx);
cudaError_t eval_loss(const float* lse, const float* s_tgt, const int* targets,
                      const int* token_bytes, int M, int V, float* out, const Ctx& ctx);
cudaError_t ce_dlogits(bool bf16, void* s, const float* lse, const int* targets,
                       const float* inv_n, int M, int V, float cap, const Ctx& ctx);

// ---- embedding backward ----
size_t embed_bwd_scratch_bytes(int M, int d);
cudaError_t embed_norm_bwd(bool bf16, const int* ids, const void* wte, const float* rstd0,
                           const float* dx, float* dwte, int accumulate, int M, int d, int V,
                           void* scratch, const Ctx& ctx);

// Test hook: a CTA waiting on an mbarrier nothing completes (bounded).
cudaError_t selftest_wait(long long timeout_ns, const Ctx& ctx);

// ---- optimizer (optimizer.cu) ------------------------------------------
struct AdamWArgs {
  float lr, beta1, beta2, eps, wd, inv_bc1, inv_bc2;
};
cudaError_t adamw_step(bool bf16_copy, float* p, const float* g, float* m, float* v, void* pc,
                       long n, const AdamWArgs& a, const Ctx& ctx);
cudaError_t muon_momentum(const float* g, float* b, long n, float mu, float* partial,
                          const Ctx& ctx);
cudaError_t muon_prepare(bool bf16, const float* g, const float* b, float mu,
                         const float* partial, int r, int c, bool transpose, void* x,
                         const Ctx& ctx);
cudaError_t muon_update(bool bf16, float* p, const void* x, int r, int c, bool transpose,
                        float step, void* pc, const Ctx& ctx);
int muon_partials();

// Host side of the optimizer step (optimizer.cu), on the C-ABI types.
struct OptTensors {
  float *wte, *w_lm;
  const nc_layer_f* layers;
  void *wte_c, *w_lm_c;
  const nc_layer_wc* layers_c;
  const float *dwte, *dw_lm;
  const nc_layer_g* grads;
  float *m_wte, *v_wte, *m_lm, *v_lm;
  const nc_layer_f* mom;
};
size_t optimizer_ws_bytes(const nc_config& c);
cudaError_t optimizer_step(const nc_config& c, const nc_opt_config& oc, int t, float lrm,
                           const OptTensors& w, void* ws, const Ctx& ctx);
}  // namespace nc
