/*
 * nc.h -- C ABI of the B300 (sm_103a) nanochat-style pretraining step.
 *
 * What is computed.  One forward + backward pass of a dense decoder stack as
 * listed in the launch article's Q&A (vpshk.cn, "安德烈·卡帕西推出nanochat…",
 * section "卡帕西亲自揭秘背后技术", architecture list): token embedding
 * followed by a parameter-free RMSNorm; L pre-norm blocks with bias-free
 * linear maps, QK-norm, rotary embeddings (no learned positions), causal
 * multi-query attention (H query heads, one K/V head) and a ReLU^2 MLP, each
 * sublayer added to the residual stream; a final RMSNorm; an untied LM head
 * whose logits pass a tanh softcap; next-token cross-entropy (imeisheng.com
 * walkthrough "100美元成本、8000行代码纯手搓克隆ChatGPT", section "预训练":
 * B rows x T tokens per forward/backward).  Readings the pages leave open
 * (eps, softcap 15, RoPE base 10000 and half-split pairing, 1/sqrt(h) scale,
 * mean loss over targets >= 0) are fixed by nc_config and stated per call.
 *
 * Conventions (all calls).
 *  - Every pointer is a DEVICE pointer unless stated otherwise; the caller
 *    owns and allocates every buffer (weights, gradients, ids, workspace).
 *    The library never allocates or frees device memory.
 *  - Matrices are row-major.  Weights use the (out, in) layout: y = x W^T.
 *      w_qkv (H+2)h x d : rows [0,Hh) query heads (h rows each), then the
 *                         key head (h rows), then the value head (h rows)
 *      w_o   d x Hh, w_fc f x d, w_proj d x f, wte V x d, w_lm V x d
 *  - Weight and activation element type: bfloat16 when cfg->dtype == NC_BF16
 *    (fp32 tensor-core accumulation), float when cfg->dtype == NC_F32 (the
 *    fp32 debug/parity mode).  The residual stream x, its gradient dx, the
 *    loss and every weight gradient are always float32.
 *  - M = B*T tokens; ids/targets are int32 (B, T).  targets < 0 are ignored.
 *  - `stream` is a cudaStream_t passed as void*.  Calls are asynchronous and
 *    stream-ordered; they return after enqueueing work.
 *  - One GPU per process: the library opts its kernels into large shared
 *    memory once, on the device current at the first call (data-parallel
 *    use runs one process per GPU).
 *  - Workspace: `ws` of at least nc_workspace_bytes(cfg, B, T) bytes, 256-byte
 *    aligned.  It carries state between the calls of one step: nc_embed_norm
 *    writes the RoPE table and embedding statistics, nc_block_fwd(l) saves
 *    layer l's activations, nc_lmhead_softcap_ce_fwd_bwd holds the logits,
 *    nc_block_bwd(l) reads layer l's saved activations.  One step's calls must
 *    use the same workspace, cfg, B and T.  Two steps in flight at once need
 *    two workspaces.
 *  - accumulate = 0 overwrites gradient buffers; 1 adds into them.
 *
 * Errors.  Arguments are validated on the host before anything is launched:
 * a bad shape, null or misaligned pointer (16 B) or a short workspace returns
 * an error and enqueues nothing.  A launch failure returns NC_ERR_CUDA.
 * Conditions only the device can see (token id outside [0, V), a bounded
 * wait that ran out) set an error word in the workspace and the kernel
 * returns without faulting; nc_get_device_status() reports and clears it.
 * nc_last_error_message() gives a one-line reason for the calling thread's
 * last non-OK status.
 *
 * Shape limits: d_model % 64 == 0, head_dim in {64, 128} (128 only in
 * NC_BF16 mode), n_head >= 1, d_mlp % 64 == 0, vocab % 64 == 0,
 * vocab <= 2^24, B >= 1, T >= 1, B*T <= 2^24, T*n_head <= 65534*128.
 */
#ifndef NC_H
#define NC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NC_OK = 0,
  NC_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad enum, bad layer index */
  NC_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the limits above */
  NC_ERR_WORKSPACE = 3,          /* workspace smaller than nc_workspace_bytes() */
  NC_ERR_CUDA = 4,               /* a CUDA launch or runtime call failed */
  NC_ERR_TIMEOUT = 5,            /* device: a bounded wait ran out (kernel returned early) */
  NC_ERR_TOKEN_RANGE = 6         /* device: a token id outside [0, vocab) (row zeroed) */
} nc_status;

typedef enum { NC_BF16 = 0, NC_F32 = 1 } nc_dtype;

typedef struct {
  int depth;       /* L */
  int d_model;     /* d */
  int n_head;      /* H query heads; one shared K/V head */
  int head_dim;    /* h */
  int d_mlp;       /* f (4d in the reference shapes) */
  int vocab;       /* V */
  float softcap;   /* c in s = c tanh(z / c); 15 */
  float rope_base; /* theta_i = base^(-2i/h); 10000 */
  float eps;       /* RMSNorm: x / sqrt(mean(x^2) + eps); 1e-6 */
  int dtype;       /* nc_dtype */
} nc_config;

typedef struct { const void *w_qkv, *w_o, *w_fc, *w_proj; } nc_layer_w;
typedef struct { float *d_qkv, *d_o, *d_fc, *d_proj; } nc_layer_g;

/* Bytes of workspace one step needs (saved activations of every layer,
 * logits, scratch, error word).  0 if cfg/B/T are invalid. */
size_t nc_workspace_bytes(const nc_config* cfg, int B, int T);

/* Embedding lookup then the post-embedding RMSNorm (architecture list: norm
 * right after the token embedding; untied embedding).
 *   ids  int32 (B, T)      wte  (V, d) act type
 *   x    out float32 (M, d): x[t] = wte[ids[t]] / rms(wte[ids[t]])
 * Also writes the RoPE cos/sin table and per-token norm statistics into ws.
 * An id outside [0, V) zeroes its row and sets NC_ERR_TOKEN_RANGE. */
nc_status nc_embed_norm(const nc_config* cfg, int B, int T, const int32_t* ids,
                        const void* wte, float* x, void* ws, size_t ws_bytes,
                        void* stream);

/* One transformer block forward, in place on the float32 residual x (M, d):
 *   x += attn(norm(x)) Wo^T ;  x += relu(norm(x) Wfc^T)^2 Wproj^T
 * attn: q,k,v = split(norm(x) Wqkv^T); q_h <- RoPE(norm(q_h)); k <- RoPE(norm(k));
 * o_h[i] = sum_{j<=i} softmax_j(q_h[i].k[j]/sqrt(h)) v[j]  (MQA, causal).
 * Saves this layer's activations in ws for nc_block_bwd.  0 <= layer < depth. */
nc_status nc_block_fwd(const nc_config* cfg, int layer, int B, int T,
                       const nc_layer_w* w, float* x, void* ws, size_t ws_bytes,
                       void* stream);

/* Final RMSNorm, LM head, softcap and mean next-token cross-entropy, with the
 * backward through all of them (architecture list: untied unembedding, logit
 * softcap; walkthrough "预训练": next-token objective).
 *   x_L      float32 (M, d), the residual after the last block
 *   w_lm     (V, d) act type;  targets int32 (B, T)
 *   loss     out: one float32 on the device, mean over targets >= 0
 *   dx_L     out float32 (M, d): d loss / d x_L
 *   dw_lm    float32 (V, d): d loss / d w_lm (overwritten or accumulated)
 * In NC_BF16 mode fp32 logits never reach HBM: the GEMM epilogue applies the
 * softcap, stores fp16 capped logits and per-row partial exp-sums. */
nc_status nc_lmhead_softcap_ce_fwd_bwd(const nc_config* cfg, int B, int T,
                                       const float* x_L, const void* w_lm,
                                       const int32_t* targets, float* loss,
                                       float* dx_L, float* dw_lm, int accumulate,
                                       void* ws, size_t ws_bytes, void* stream);

/* One block backward.  dx float32 (M, d) holds d loss / d(block output) on
 * entry and d loss / d(block input) on return.  Writes the four weight
 * gradients of g (float32, same shapes as the weights).  Needs the
 * activations nc_block_fwd(layer) saved in the same ws. */
nc_status nc_block_bwd(const nc_config* cfg, int layer, int B, int T,
                       const nc_layer_w* w, float* dx, const nc_layer_g* g,
                       int accumulate, void* ws, size_t ws_bytes, void* stream);

/* Backward of nc_embed_norm: dwte[v] = sum over tokens t with ids[t] == v of
 * d loss / d wte-row, through the post-embedding RMSNorm.  dx float32 (M, d)
 * is d loss / d x.  The sum is deterministic (tokens sorted by id, then
 * summed in token order).  dwte float32 (V, d). */
nc_status nc_embed_norm_bwd(const nc_config* cfg, int B, int T, const int32_t* ids,
                            const void* wte, const float* dx, float* dwte,
                            int accumulate, void* ws, size_t ws_bytes, void* stream);

/* The whole step: nc_embed_norm, nc_block_fwd for l = 0..L-1,
 * nc_lmhead_softcap_ce_fwd_bwd, nc_block_bwd for l = L-1..0, nc_embed_norm_bwd.
 * layers[l] / grads[l] are arrays of `depth` entries (host memory). */
nc_status nc_step(const nc_config* cfg, int B, int T, const int32_t* ids,
                  const int32_t* targets, const void* wte, const nc_layer_w* layers,
                  const void* w_lm, float* loss, float* dwte, const nc_layer_g* grads,
                  float* dw_lm, int accumulate, void* ws, size_t ws_bytes, void* stream);

/* Forward-only evaluation (walkthrough, pretraining section: the run
 * reports validation bits per byte -- the next-token loss normalised by the
 * bytes per token, comparable across tokenizers).  Runs the forward pass and
 * the loss without any backward; writes out[0] = mean loss over targets >= 0
 * (nats) and out[1] = sum of the losses of targets whose byte length is > 0,
 * divided by ln 2 times the sum of those byte lengths (bits per byte), or
 * NaN when token_bytes is NULL.  token_bytes: int32 [vocab] byte length of
 * each token id (0 for special tokens, which then count in neither sum).
 * out: device float[2], 8-byte aligned.  Same workspace as nc_step. */
nc_status nc_eval(const nc_config* cfg, int B, int T, const int32_t* ids, const int32_t* targets,
                  const int32_t* token_bytes, const void* wte, const nc_layer_w* layers,
                  const void* w_lm, float* out, void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, reads the device error word of `ws`, clears it and
 * returns NC_OK, NC_ERR_TIMEOUT or NC_ERR_TOKEN_RANGE (or NC_ERR_CUDA). */
nc_status nc_get_device_status(void* ws, void* stream);

const char* nc_status_string(nc_status s);
const char* nc_last_error_message(void);

/* ---- optimizer step ------------------------------------------------------
 * The update that follows a step (architecture list: Muon + AdamW, after
 * modded-nanoGPT; walkthrough, pretraining section: Muon for the matrices,
 * AdamW for the embedding and the unembedding, learning rates scaled by
 * 1/sqrt(dim), lrm falling linearly to 0 at the end of training).
 *
 * Every tensor here is a device pointer the caller owns.  Master weights,
 * gradients and optimizer state are float32 (same shapes as the weights);
 * each updated master is also written to its compute copy (the bf16 or
 * float weights the step reads, per cfg->dtype).
 *   AdamW (wte, w_lm): m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
 *     w <- w - lr wd w - lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps),
 *     lr = lr_embed (wte) or lr_lm (w_lm) times lrm / sqrt(d_model).
 *   Muon (every block matrix, r x c): b <- mu b + g; u = g + mu b;
 *     X = u / (||u||_F + 1e-7) (transposed when r > c), then ns_steps of
 *     X <- a X + (b A + c A A) X with A = X X^T (act-type batched GEMMs, all
 *     layers of one shape at once); w <- w - lr_muon lrm sqrt(max(1, r/c)) X.
 * t counts optimizer steps from 1 (AdamW bias correction).  lrm is the
 * caller's schedule value for this step.  ws: >= nc_optimizer_workspace_bytes
 * (scratch for the Newton-Schulz iterates, and the error word).  The result
 * is a deterministic function of the inputs (fixed-order reductions). */
typedef struct {
  float lr_muon, momentum;                  /* Muon */
  float lr_embed, lr_lm;                    /* AdamW rates before lrm / sqrt(d_model) */
  float beta1, beta2, eps, weight_decay;    /* AdamW */
  float ns_a, ns_b, ns_c;                   /* Newton-Schulz odd polynomial */
  int ns_steps;
} nc_opt_config;
typedef struct { float *w_qkv, *w_o, *w_fc, *w_proj; } nc_layer_f;   /* float32 per-layer */
typedef struct { void *w_qkv, *w_o, *w_fc, *w_proj; } nc_layer_wc;   /* compute copies */
size_t nc_optimizer_workspace_bytes(const nc_config* cfg);
nc_status nc_optimizer_step(const nc_config* cfg, const nc_opt_config* oc, int t, float lrm,
                            float* wte, float* w_lm, const nc_layer_f* layers,
                            void* wte_c, void* w_lm_c, const nc_layer_wc* layers_c,
                            const float* dwte, const float* dw_lm, const nc_layer_g* grads,
                            float* m_wte, float* v_wte, float* m_lm, float* v_lm,
                            const nc_layer_f* momentum_bufs, void* ws, size_t ws_bytes,
                            void* stream);

/* ---- building blocks (the same kernels the step uses), for tests -------- */

/* Bias-free linear layer contraction on the step's GEMM kernels
 * (architecture list: bias-free linear layers).  dtype selects the kernel:
 * NC_BF16 -> tcgen05/TMEM tensor-core kernel fed by TMA (A, B bfloat16),
 * NC_F32 -> fp32 SIMT kernel (A, B float).
 *   layout NC_GEMM_NT: C(M,N) = A(M,K) . B(N,K)^T     (forward: x W^T)
 *          NC_GEMM_NN: C(M,N) = A(M,K) . B(K,N)       (dX = dY W)
 *          NC_GEMM_TN: C(M,N) = A(K,M)^T . B(K,N)     (dW = dY^T X)
 *   epilogue NC_EPI_STORE      C act type  = acc
 *            NC_EPI_STORE_F32  C float32   = acc  (+ C if accumulate)
 *            NC_EPI_ADD_F32    C float32  += acc  (residual add)
 *            NC_EPI_RELU2      C act type  = max(acc, 0)^2
 *            NC_EPI_RELU2_BWD  C act type  = acc * 2 sqrt(aux), aux (M,N) act
 *                              type holding relu(u)^2 (so 2 sqrt(aux) = 2 relu(u))
 * lda/ldb/ldc are row strides in elements (multiples of 8, so every row
 * starts 16-byte aligned).  M, N, K >= 1, N % 32 == 0; M and K may be ragged.
 * ws: >= nc_gemm_workspace_bytes(...). */
typedef enum { NC_GEMM_NT = 0, NC_GEMM_NN = 1, NC_GEMM_TN = 2 } nc_gemm_layout;
typedef enum {
  NC_EPI_STORE = 0, NC_EPI_STORE_F32 = 1, NC_EPI_ADD_F32 = 2,
  NC_EPI_RELU2 = 3, NC_EPI_RELU2_BWD = 4
} nc_epilogue;
size_t nc_gemm_workspace_bytes(int dtype, int layout, int M, int N, int K);
nc_status nc_gemm(int dtype, int layout, int epilogue, int M, int N, int K,
                  const void* A, int lda, const void* Bm, int ldb, void* C, int ldc,
                  const void* aux, int accumulate, void* ws, size_t ws_bytes,
                  void* stream);

/* Batched contraction on the same kernels: `batch` independent products
 * C_z = op(A_z, B_z), z = 0..batch-1, with A_z = A + z a_bstride,
 * B_z = Bm + z b_bstride, C_z = C + z c_bstride (element strides, multiples
 * of 8).  epilogue NC_EPI_STORE (C act type = acc) or NC_EPI_AXPBY (C act type
 * = alpha aux_z + beta acc, aux_z = aux + z c_bstride, same layout as C).
 * The Muon update's Newton-Schulz steps are built from it.  Same shape rules
 * as nc_gemm; batch >= 1; no workspace beyond the error word (ws >= 256 B). */
enum { NC_EPI_AXPBY = 6 };
nc_status nc_gemm_batched(int dtype, int layout, int epilogue, int batch, int M, int N, int K,
                          const void* A, int lda, long a_bstride, const void* Bm, int ldb,
                          long b_bstride, void* C, int ldc, long c_bstride, const void* aux,
                          float alpha, float beta, void* ws, size_t ws_bytes, void* stream);

/* 8-bit floating-point contraction on the same tensor-core kernel (the FP8
 * mixed-precision training of the latest version: nanochat hub page, core
 * technical highlights.  The pages name no format; this is OCP FP8 E4M3 --
 * 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * S.1111.111 is NaN, largest finite 448):
 *   C(M,N) = scale * A(M,K) . B(N,K)^T
 * A, B: E4M3 codes as raw bytes, row-major, both K-major (layout NT only),
 * leading dimensions lda, ldb in elements (= bytes), multiples of 16;
 * products are exact and accumulate in fp32; scale (finite) is applied to the
 * fp32 sum, e.g. the product of the operands' per-tensor dequantisation
 * scales.  out_dtype NC_BF16 or NC_F32 selects C's type; ldc in elements, a
 * multiple of 8.  M, N, K >= 1, N % 32 == 0, K % 16 == 0 (M ragged).  No
 * workspace beyond the error word (ws >= 256 B); pointers 16-byte aligned.
 * The step itself stays bf16. */
nc_status nc_gemm_fp8(int M, int N, int K, const void* A, int lda, const void* Bm, int ldb,
                      int out_dtype, void* C, int ldc, float scale, void* ws, size_t ws_bytes,
                      void* stream);

/* Causal multi-query attention alone (architecture list: MQA; causal from the
 * next-token objective).  q (B, T, H, h), k and v (B, T, h), o (B, T, H, h),
 * act type; lse float32 (B, T, H): natural-log sum of exp of the scaled
 * scores of each query row.  Scale 1/sqrt(h); key j visible to query i iff
 * j <= i.  Backward: dq like q; dk, dv like k (summed over the H heads).
 * dq/dk/dv rows are written with row strides ldq/ldk/ldv elements (per token),
 * so they can land inside a (M, (H+2)h) gradient buffer.  ws: scratch of at
 * least nc_attention_workspace_bytes(B, T, H). */
size_t nc_attention_workspace_bytes(int B, int T, int H);
nc_status nc_attention_fwd(int dtype, int B, int T, int H, int h, const void* q,
                           const void* k, const void* v, void* o, float* lse,
                           void* ws, size_t ws_bytes, void* stream);
nc_status nc_attention_bwd(int dtype, int B, int T, int H, int h, const void* q,
                           const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, void* dq, int ldq,
                           void* dk, int ldk, void* dv, int ldv, void* ws,
                           size_t ws_bytes, void* stream);

/* Attention backward that allocates nothing and needs no workspace.  The
 * pages have no counterpart: this is a convenience of this library for
 * callers that cannot hand it device memory at this point -- for example an
 * operator running inside another framework's runtime (a plugin or custom
 * call) that owns all device memory and gives this op no scratch, or a hot
 * loop that must not call cudaMalloc, which can synchronise the device.
 * Arguments and results are those of nc_attention_bwd.  The per-row scratch
 * (delta = rowsum(dO * O)) lives in one fixed device array built into the
 * library (8 MB, held on every GPU that loads the library until the process
 * exits), so B*T*H must be <= 2^21 query rows; larger shapes return
 * NC_ERR_UNSUPPORTED_SHAPE without launching.  The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress, with the
 * device current) and caches it; make that first call before any stream
 * capture.  Every call shares the array: calls that overlap on the GPU race,
 * so order them (one stream, or events).  Each call rewrites every scratch
 * entry it reads, so no clearing is needed between calls.  Like the rest of
 * the library it assumes one GPU per process (the kernels' shared-memory
 * opt-in is made once, on the first device used).
 * Device-side conditions: the kernels bound every wait; a wait that runs out
 * makes its CTA stop early, so dq/dk/dv of that call are incomplete, and
 * records NC_ERR_TIMEOUT in a second fixed device word of the library (there
 * is no workspace to hold it).  nc_attention_bwd_noalloc_status() reads it. */
nc_status nc_attention_bwd_noalloc(int dtype, int B, int T, int H, int h, const void* q,
                                   const void* k, const void* v, const void* o,
                                   const float* lse, const void* dout, void* dq, int ldq,
                                   void* dk, int ldk, void* dv, int ldv, void* stream);

/* Status of the allocation-free calls on the current device: synchronises
 * `stream`, reads the device error word they share, clears it and returns
 * NC_OK, NC_ERR_TIMEOUT (some call since the last read stopped early and left
 * its gradients incomplete) or NC_ERR_CUDA.  Allocates nothing. */
nc_status nc_attention_bwd_noalloc_status(void* stream);

/* ---- measurement ----------------------------------------------------------
 * Support for the throughput and roofline measurements of the step (the
 * walkthrough's "预训练" section reports model-FLOP utilisation; these calls
 * let a caller attribute the step's time to its kernels).  Not thread-safe:
 * use from one host thread.
 *   nc_launch_count    kernels launched by the library so far (host counter)
 *   nc_profile_start   from now on, bracket every named launch group of the
 *                      step with CUDA events on its stream (host-side event
 *                      objects, 2 per record, created here; no device memory)
 *   nc_profile_stop    stop recording; returns the number of records
 *   nc_profile_record  name (static string) and elapsed ms of record i;
 *                      waits for that record's end event */
long long nc_launch_count(void);
nc_status nc_profile_start(int max_records);
int nc_profile_stop(void);
nc_status nc_profile_record(int i, const char** name, float* ms);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nothing will complete, for at most `timeout_us` microseconds, then
 * records NC_ERR_TIMEOUT in ws's error word and returns.  Never hangs.  With
 * ws == NULL it records into the allocation-free calls' error word instead
 * (read by nc_attention_bwd_noalloc_status). */
nc_status nc_selftest_wait_timeout(int timeout_us, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NC_H */
