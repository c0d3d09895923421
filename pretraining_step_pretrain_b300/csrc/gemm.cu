// GEMM launchers: the tcgen05 bf16 kernel (gemm_tc.cuh) and the fp32 SIMT
// kernel used by the fp32 debug/parity mode, with the epilogue selection and
// the deterministic split-K reduction for weight gradients.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>
#include <mutex>

#include "epilogue.cuh"
#include "gemm_tc.cuh"
#include "nc_internal.h"

namespace nc {

// ===================================================================
// fp32 SIMT GEMM (debug mode): 64 x 64 tile, 256 threads x (4 x 4) outputs.
// ===================================================================
template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(256) gemm_f32_simt_kernel(const float* __restrict__ A, long lda,
                                                            const float* __restrict__ B, long ldb,
                                                            int M, int N, int K, Epi epi) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 1024; i += 256) {
      int mm, kk;
      if (A_MN) { mm = i & 63; kk = i >> 6; } else { kk = i & 15; mm = i >> 4; }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < M && gk < K) v = A_MN ? A[(long)gk * lda + gm] : A[(long)gm * lda + gk];
      As[kk][mm] = v;
    }
    for (int i = threadIdx.x; i < 1024; i += 256) {
      int nn, kk;
      if (B_MN) { nn = i & 63; kk = i >> 6; } else { kk = i & 15; nn = i >> 4; }
      const int gn = n0 + nn, gk = k0 + kk;
      float v = 0.f;
      if (gn < N && gk < K) v = B_MN ? B[(long)gk * ldb + gn] : B[(long)gn * ldb + gk];
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i, col = n0 + tx * 4;
    if (row < M && col < N) {
      float v[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
      epi.template apply<4>(row, col, v, 0);
    }
  }
}

template <bool A_MN, bool B_MN, class Epi>
static cudaError_t launch_f32(const GemmArgs& g, const Epi& epi, const Ctx& ctx) {
  dim3 grid((g.N + 63) / 64, (g.M + 63) / 64);
  gemm_f32_simt_kernel<A_MN, B_MN, Epi><<<grid, 256, 0, ctx.stream>>>(
      static_cast<const float*>(g.A), g.lda, static_cast<const float*>(g.B), g.ldb, g.M, g.N, g.K,
      epi);
  return launched(1);
}

template <class Epi>
static cudaError_t dispatch_f32(const GemmArgs& g, const Epi& epi, const Ctx& ctx) {
  switch (g.layout) {
    case GEMM_NT: return launch_f32<false, false>(g, epi, ctx);
    case GEMM_NN: return launch_f32<false, true>(g, epi, ctx);
    case GEMM_TN: return launch_f32<true, true>(g, epi, ctx);
  }
  return cudaErrorInvalidValue;
}

cudaError_t gemm_f32_one(const GemmArgs& g, const Ctx& ctx) {
  switch (g.epi) {
    case EPI_STORE: return dispatch_f32(g, EpiStore<float>{static_cast<float*>(g.C), g.ldc}, ctx);
    case EPI_STORE_F32:
      return dispatch_f32(g, EpiStoreF32{static_cast<float*>(g.C), g.ldc, 0, g.accumulate}, ctx);
    case EPI_ADD_F32: return dispatch_f32(g, EpiAddF32{static_cast<float*>(g.C), g.ldc}, ctx);
    case EPI_RELU2: return dispatch_f32(g, EpiRelu2<float>{static_cast<float*>(g.C), g.ldc}, ctx);
    case EPI_RELU2_BWD:
      return dispatch_f32(g,
                          EpiRelu2Bwd<float>{static_cast<float*>(g.C),
                                             static_cast<const float*>(g.aux), g.ldc},
                          ctx);
    case EPI_AXPBY:
      return dispatch_f32(g,
                          EpiAxpby<float>{static_cast<float*>(g.C),
                                          static_cast<const float*>(g.aux), g.ldc, 0, g.alpha,
                                          g.beta},
                          ctx);
  }
  return cudaErrorInvalidValue;
}

// The fp32 SIMT path runs a batched product as one launch per entry.
cudaError_t gemm_f32(const GemmArgs& g, const Ctx& ctx) {
  const int nb = g.batch > 1 ? g.batch : 1;
  for (int z = 0; z < nb; ++z) {
    GemmArgs e = g;
    e.A = static_cast<const float*>(g.A) + z * g.a_bstride;
    e.B = static_cast<const float*>(g.B) + z * g.b_bstride;
    e.C = static_cast<float*>(g.C) + z * g.c_bstride;
    if (g.aux) e.aux = static_cast<const float*>(g.aux) + z * g.c_bstride;
    cudaError_t r = gemm_f32_one(e, ctx);
    if (r != cudaSuccess) return r;
  }
  return cudaSuccess;
}

// ===================================================================
// tcgen05 bf16 GEMM
// ===================================================================
namespace {

// Work-unit count the split heuristic aims at (B300: 148 SMs = 74 CTA pairs).
// The launch itself uses the real SM count.
constexpr int kSplitUnits = 74;

struct Plan {
  tc::Sched sch;
};

Plan make_plan(int layout, int epi, int M, int N, int K, int group_m, int batch = 1) {
  Plan p;
  tc::Sched& s = p.sch;
  s.batches = batch > 1 ? batch : 1;
  s.m_tiles = (M + tc::BM - 1) / tc::BM;
  s.n_tiles = (N + tc::BN - 1) / tc::BN;
  s.k_blocks = (K + tc::BK - 1) / tc::BK;
  s.splits = 1;
  s.kb_per_split = s.k_blocks;
  const int tiles = s.m_tiles * s.n_tiles;
  if (epi == EPI_STORE_F32 && s.batches == 1 && tiles < 2 * kSplitUnits && s.k_blocks >= 32) {
    // Split the reduction so that the units fill the SMs; cost proxy =
    // waves x k-blocks per unit, plus one k-block per split for the slab pass.
    long best = -1;
    for (int sp = 1; sp <= 16; ++sp) {
      const int kbp = (s.k_blocks + sp - 1) / sp;
      if (kbp < 8) break;
      const int eff_splits = (s.k_blocks + kbp - 1) / kbp;
      const int units = tiles * eff_splits;
      const long waves = (units + kSplitUnits - 1) / kSplitUnits;
      const long cost = waves * kbp + (eff_splits > 1 ? eff_splits : 0);
      if (best < 0 || cost < best) {
        best = cost;
        s.splits = eff_splits;
        s.kb_per_split = kbp;
      }
    }
  }
  s.group_m = group_m > 0 ? group_m : 8;
  s.units = tiles * s.splits * s.batches;
  (void)layout;
  return p;
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor map over `nb` row-major (outer x inner) matrices with row
// stride `ld` and matrix stride `bstride` elements (dims {inner, outer, nb});
// 128-byte swizzle; out-of-range elements read as zero.
bool make_tmap(CUtensorMap* m, const void* base, long inner, long outer, long ld, int box_inner,
               int box_outer, long nb = 1, long bstride = 0, bool bytes = false) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  if (nb < 1) nb = 1;
  if (bstride <= 0) bstride = outer * ld;
  const long es = bytes ? 1 : 2;  // 8-bit (E4M3 as raw bytes) or bf16 elements
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)nb};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * es), (cuuint64_t)(bstride * es)};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Destination map for the epilogue's bulk stores: dims {N, M, Z} (Z split-K
// slabs or batch entries, else 1), row stride `ld` elements, slab stride
// `zstride` elements (0: M * ld), box {128 bytes, 128 rows, 1}.
template <typename Out>
bool make_tmap_out(CUtensorMap* m, void* base, long N, long M, long ld, long Z,
                   long zstride = 0) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  const CUtensorMapDataType dt =
      sizeof(Out) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                       : (std::is_same<Out, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  const long es = sizeof(Out);
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)Z};
  if (zstride <= 0) zstride = M * ld;
  cuuint64_t strides[2] = {(cuuint64_t)(ld * es), (cuuint64_t)(zstride * es)};
  cuuint32_t box[3] = {(cuuint32_t)(128 / es), (cuuint32_t)tc::HALF_ROWS, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_tc(const GemmArgs& g, const Plan& p, const Epi& epi, void* out, long ldo,
                      long zslabs, const Ctx& ctx) {
  CUtensorMap ta, tb, tcm;
  const long nb = p.sch.batches;
  bool ok = A_MN ? make_tmap(&ta, g.A, g.M, g.K, g.lda, 64, 64, nb, g.a_bstride)
                 : make_tmap(&ta, g.A, g.K, g.M, g.lda, 64, tc::HALF_ROWS, nb, g.a_bstride);
  ok = ok && (B_MN ? make_tmap(&tb, g.B, g.N, g.K, g.ldb, 64, 64, nb, g.b_bstride)
                   : make_tmap(&tb, g.B, g.K, g.N, g.ldb, 64, tc::HALF_ROWS, nb, g.b_bstride));
  ok = ok && make_tmap_out<typename Epi::Out>(&tcm, out, g.N, g.M, ldo, zslabs * nb,
                                              nb > 1 ? g.c_bstride : 0);
  // Auxiliary operand (same layout as C) for the epilogues that read one;
  // the others get C's map, unused.
  constexpr bool kAux = tc::HasAuxTma<Epi>::value;
  constexpr bool kHeads = tc::HasHeadPairs<Epi>::value;
  CUtensorMap tax = tcm;
  if constexpr (kAux)
    ok = ok && make_tmap_out<typename Epi::Out>(&tax, const_cast<void*>(g.aux), g.N, g.M, ldo,
                                                nb, nb > 1 ? g.c_bstride : 0);
  if constexpr (kHeads)  // the (T, 128) fp16 table, [128 rows][64 values] boxes
    ok = ok && make_tmap_out<__half>(&tax, const_cast<__half2*>(epi.tab), 128, epi.T, 128, 1);
  if (!ok) return cudaErrorInvalidValue;
  auto kern = tc::gemm_bf16_tc_kernel<A_MN, B_MN, Epi>;
  constexpr int smem_bytes = tc::SmemPlan<kAux || kHeads>::BYTES;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // One CTA pair (a 2-CTA cluster) per unit, at most one CTA per SM.
  const int grid = 2 * std::max(1, std::min(p.sch.units, ctx.num_sms / 2));
  kern<<<grid, tc::NUM_THREADS, smem_bytes, ctx.stream>>>(ta, tb, tcm, tax, p.sch, g.M, g.N, epi,
                                                          ctx.err, ctx.timeout_ns);
  return launched(1);
}

// C(M,N) = scale * A(M,K) . B(N,K)^T with E4M3 operands (both K-major, as
// raw bytes), fp32 accumulation, bf16 or fp32 output.
template <class Epi>
cudaError_t launch_tc_fp8(const GemmArgs& g, const Epi& epi, const Ctx& ctx) {
  // A k-block is 128 bytes of a row (128 values); the planner counts k-blocks
  // of 64 elements, so it gets K / 2 (K is a multiple of 16).
  const Plan p = make_plan(GEMM_NT, EPI_STORE, g.M, g.N, g.K / 2, g.group_m);
  CUtensorMap ta, tb, tcm;
  bool ok = make_tmap(&ta, g.A, g.K, g.M, g.lda, 128, tc::HALF_ROWS, 1, 0, true) &&
            make_tmap(&tb, g.B, g.K, g.N, g.ldb, 128, tc::HALF_ROWS, 1, 0, true) &&
            make_tmap_out<typename Epi::Out>(&tcm, g.C, g.N, g.M, g.ldc, 1, 0);
  if (!ok) return cudaErrorInvalidValue;
  auto kern = tc::gemm_bf16_tc_kernel<false, false, Epi, true>;
  constexpr int smem_bytes = tc::SmemPlan<false>::BYTES;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = 2 * std::max(1, std::min(p.sch.units, ctx.num_sms / 2));
  kern<<<grid, tc::NUM_THREADS, smem_bytes, ctx.stream>>>(ta, tb, tcm, tcm, p.sch, g.M, g.N, epi,
                                                          ctx.err, ctx.timeout_ns);
  return launched(1);
}

template <class Epi>
cudaError_t dispatch_tc(const GemmArgs& g, const Plan& p, const Epi& epi, void* out, long ldo,
                        long zslabs, const Ctx& ctx) {
  switch (g.layout) {
    case GEMM_NT: return launch_tc<false, false>(g, p, epi, out, ldo, zslabs, ctx);
    case GEMM_NN: return launch_tc<false, true>(g, p, epi, out, ldo, zslabs, ctx);
    case GEMM_TN: return launch_tc<true, true>(g, p, epi, out, ldo, zslabs, ctx);
  }
  return cudaErrorInvalidValue;
}

__global__ void splitk_reduce_kernel(float4* __restrict__ c, const float4* __restrict__ slabs,
                                     int splits, long n4, long slab4, int accumulate) {
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4;
       i += (long)gridDim.x * blockDim.x) {
    float4 s = accumulate ? c[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < splits; ++k) {
      const float4 t = slabs[k * slab4 + i];
      s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
    }
    c[i] = s;
  }
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
  auto enc = tmap_encoder();
  if (!enc || rank < 2 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, b, e,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t splitk_reduce(float* c, const float* slabs, int splits, long n, int accumulate,
                          const Ctx& ctx) {
  const long n4 = n / 4;
  const int blocks = (int)std::min<long>((n4 + 255) / 256, (long)ctx.num_sms * 8);
  splitk_reduce_kernel<<<std::max(blocks, 1), 256, 0, ctx.stream>>>(
      reinterpret_cast<float4*>(c), reinterpret_cast<const float4*>(slabs), splits, n4, n4,
      accumulate);
  return launched(1);
}

size_t gemm_bf16_split_elems(int layout, int epi, int M, int N, int K) {
  Plan p = make_plan(layout, epi, M, N, K, 0);
  return p.sch.splits > 1 ? (size_t)p.sch.splits * M * N : 0;
}

cudaError_t gemm_fp8(const GemmArgs& g, bool out_f32, float scale, const Ctx& ctx) {
  if (out_f32)
    return launch_tc_fp8(g, EpiScaleStore<float>{static_cast<float*>(g.C), g.ldc, scale}, ctx);
  return launch_tc_fp8(g, EpiScaleStore<bf16>{static_cast<bf16*>(g.C), g.ldc, scale}, ctx);
}

cudaError_t gemm_bf16(const GemmArgs& g, const Ctx& ctx) {
  const Plan p = make_plan(g.layout, g.epi, g.M, g.N, g.K, g.group_m, g.batch);
  const bf16* aux = static_cast<const bf16*>(g.aux);
  switch (g.epi) {
    case EPI_STORE:
      return dispatch_tc(g, p, EpiStore<bf16>{static_cast<bf16*>(g.C), g.ldc}, g.C, g.ldc, 1,
                         ctx);
    case EPI_STORE_F32: {
      if (p.sch.splits == 1)
        return dispatch_tc(g, p, EpiStoreF32{static_cast<float*>(g.C), g.ldc, 0, g.accumulate},
                           g.C, g.ldc, 1, ctx);
      const size_t need = (size_t)p.sch.splits * g.M * g.N;
      if (!g.split_buf || g.split_buf_elems < need || g.ldc != g.N) return cudaErrorInvalidValue;
      cudaError_t e = dispatch_tc(g, p, EpiStoreF32{g.split_buf, (long)g.N, (long)g.M * g.N, 0},
                                  g.split_buf, g.N, p.sch.splits, ctx);
      if (e != cudaSuccess) return e;
      return splitk_reduce(static_cast<float*>(g.C), g.split_buf, p.sch.splits, (long)g.M * g.N,
                           g.accumulate, ctx);
    }
    case EPI_ADD_F32:
      return dispatch_tc(g, p, EpiAddF32{static_cast<float*>(g.C), g.ldc}, g.C, g.ldc, 1, ctx);
    case EPI_RELU2:
      return dispatch_tc(g, p, EpiRelu2<bf16>{static_cast<bf16*>(g.C), g.ldc}, g.C, g.ldc, 1,
                         ctx);
    case EPI_RELU2_BWD:
      return dispatch_tc(g, p, EpiRelu2Bwd<bf16>{static_cast<bf16*>(g.C), aux, g.ldc}, g.C,
                         g.ldc, 1, ctx);
    case EPI_SOFTCAP_CE: {
      EpiSoftcapCE e{static_cast<__half*>(g.C), g.ldc, g.part, g.n_part, tc::BN, g.targets,
                     g.s_tgt, g.cap, 1.f / g.cap};
      return dispatch_tc(g, p, e, g.C, g.ldc, 1, ctx);
    }
    case EPI_AXPBY: {
      EpiAxpby<bf16> e{static_cast<bf16*>(g.C), aux, g.ldc, g.batch > 1 ? g.c_bstride : 0,
                       g.alpha, g.beta};
      return dispatch_tc(g, p, e, g.C, g.ldc, 1, ctx);
    }
    case EPI_QKNORM_ROPE: {
      // NT only; C (the (M, (H + 2) 128) product) is only the kernel's unused
      // default map: the heads go to q, k, v through the epilogue's maps.
      const long Hh = (long)g.qk_H * 128;
      if (g.layout != GEMM_NT || g.N != (g.qk_H + 2) * 128 || g.batch > 1 || !g.qk_q ||
          !g.qk_k || !g.qk_v || !g.qk_rstd || !g.qk_tab || g.qk_T < 1 || g.qk_T % 128 != 0)
        return cudaErrorInvalidValue;
      EpiQkNormRope e;
      if (!make_tmap_out<bf16>(&e.mq, g.qk_q, Hh, g.M, Hh, 1) ||
          !make_tmap_out<bf16>(&e.mk, g.qk_k, 128, g.M, 128, 1) ||
          !make_tmap_out<bf16>(&e.mv, g.qk_v, 128, g.M, 128, 1))
        return cudaErrorInvalidValue;
      e.tab = static_cast<const __half2*>(g.qk_tab);
      e.rstd_qk = g.qk_rstd;
      e.T = g.qk_T;
      e.H = g.qk_H;
      e.eps = g.qk_eps;
      return launch_tc<false, false>(g, p, e, g.C, g.ldc, 1, ctx);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace nc
