// Persistent bf16 GEMM on the 5th-generation tensor cores (sm_100 family,
// built for sm_103a): TMA -> 128B-swizzled shared memory -> tcgen05.mma ->
// fp32 accumulator in tensor memory -> tcgen05.ld -> fused epilogue.
//
//   C[m][n] = sum_k A(m, k) B(n, k)
//   A(m, k) = A[m * lda + k] (K-major)  or  A[k * lda + m] (A_MN: M-major)
//   B(n, k) = B[n * ldb + k] (K-major)  or  B[k * ldb + n] (B_MN: N-major)
//
// Two CTAs of a cluster (a CTA pair on two SMs) compute one 256 x 256 output
// tile with cta_group::2 MMAs: each CTA loads 128 rows of the A tile and 128
// rows of the B tile (64 K-columns a stage, 32 KB, 6 stages), the even CTA
// issues the MMAs, and each CTA's tensor memory holds its 128 output rows x
// 256 columns (two accumulators, so the epilogue of one tile overlaps the
// main loop of the next).  Per FLOP this moves 1.5x fewer operand bytes from
// L2 into shared memory than one CTA working a 128 x 256 tile alone.  Each
// pair walks work units (m-tile, n-tile, k-split) with a grid stride; m-tiles
// are visited in groups so that concurrently running pairs share tiles in L2.
//
// Warp roles (256 threads per CTA): warp 0 lane 0 issues TMA (both CTAs;
// completion is counted on the even CTA's barrier), warp 1 lane 0 of the
// even CTA issues tcgen05.mma, warp 2 owns the TMEM allocation, warps 4..7
// run the epilogue (warp 4 + i reads TMEM lanes 32i..32i+31).  Every wait is
// bounded: on timeout the CTA records DEV_TIMEOUT, its roles stop, in-flight
// work is drained (bounded) and TMEM is released before the pair exits.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "epilogue.cuh"
#include "nc_common.cuh"
#include "tc_common.cuh"

namespace nc {
namespace tc {

constexpr int BM = 256;              // output rows per CTA pair
constexpr int BN = 256;              // output columns
constexpr int BK = 64;
constexpr int HALF_ROWS = 128;       // rows of the A and of the B tile each CTA loads
constexpr int STAGES = 6;
constexpr int A_BYTES = HALF_ROWS * BK * 2;  // 16 KB
constexpr int B_BYTES = HALF_ROWS * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 256;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align slack*/ + 256 /*barriers*/;
// Swizzle-128B atom: 8 rows of 128 bytes.  An MN-major operand half-tile is
// stored as 128/64 = 2 column blocks of 64 elements, each BK rows of 128 B.
constexpr int MN_BLOCK_BYTES = BK * 128;  // 8 KB

struct Sched {
  int m_tiles, n_tiles, splits, k_blocks, kb_per_split, group_m, units;

  __device__ __forceinline__ void decode(int u, int& mt, int& nt, int& split, int& kb0,
                                         int& kb1) const {
    const int per_split = m_tiles * n_tiles;
    split = u / per_split;
    const int r = u - split * per_split;
    const int group_size = group_m * n_tiles;
    const int group = r / group_size;
    const int first_m = group * group_m;
    const int gm = min(group_m, m_tiles - first_m);
    const int in = r - group * group_size;
    mt = first_m + in % gm;
    nt = in / gm;
    kb0 = split * kb_per_split;
    kb1 = min(k_blocks, kb0 + kb_per_split);
  }
};

// K-major tile (rows of 64 K-elements = 128 B, 8-row swizzle atoms 1 KB apart):
// LBO unused for swizzled K-major, SBO = 1 KB.  MMA step k (16 elements) starts
// 32 B further inside the atom.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int k) {
  return sdesc_sw128(tile + k * 32, 16, 1024);
}
// MN-major tile (column blocks of 64 MN-elements, BK rows of 128 B each):
// LBO = distance between 64-wide MN blocks, SBO = distance between 8-row
// K groups.  MMA step k covers K rows 16k..16k+15 = 2 K groups.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int k) {
  return sdesc_sw128(tile + k * 2048, MN_BLOCK_BYTES, 1024);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, M = 256 (pair), N = 256.
__host__ __device__ constexpr uint32_t idesc_bf16(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// Epilogues that declare kPrefetch load their per-row operand for the whole
// tile before waiting for the accumulator.
template <class E, class = void>
struct HasPrefetch {
  static constexpr bool value = false;
};
template <class E>
struct HasPrefetch<E, std::void_t<decltype(E::kPrefetch)>> {
  static constexpr bool value = E::kPrefetch;
};
struct NoPre {};
template <class E, bool kPre>
struct PreOf {
  using type = NoPre;
};
template <class E>
struct PreOf<E, true> {
  using type = typename E::Pre;
};

enum WaitSite : int {
  SITE_PROD_EMPTY = 101, SITE_MMA_ACC_EMPTY = 102, SITE_MMA_FULL = 103,
  SITE_EPI_ACC_FULL = 104, SITE_DRAIN = 105
};

template <bool A_MN, bool B_MN, class Epi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const Sched sch, const int M,
                        const int N, const Epi epi, int* err, const long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs, 1: its peer
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // used on the even CTA: both CTAs' bytes
      mbar_init(&empty[s], 1);  // one multicast commit per phase, in each CTA
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // used on the even CTA: 4 epilogue warps x 2 CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    int stage = 0;
    uint32_t phase = 0;
    int armed_phase[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) armed_phase[s] = -1;
    bool ok = true;
    for (int u = pair; u < sch.units && ok; u += npairs) {
      int mt, nt, split, kb0, kb1;
      sch.decode(u, mt, nt, split, kb0, kb1);
      const int row_a = mt * BM + (int)rank * HALF_ROWS;
      const int row_b = nt * BN + (int)rank * HALF_ROWS;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_flag, err, SITE_PROD_EMPTY,
                               timeout_ns)) {
          ok = false;
          break;
        }
        if (rank == 0) {
          mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          armed_phase[stage] = (int)phase;
        }
        const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
        uint8_t* a = sA + stage * A_BYTES;
        uint8_t* b = sB + stage * B_BYTES;
        const int k0 = kb * BK;
        if (!A_MN) {
          tma_load_2d_pair(a, &tmA, bar, k0, row_a);
        } else {
#pragma unroll
          for (int j = 0; j < HALF_ROWS / 64; ++j)
            tma_load_2d_pair(a + j * MN_BLOCK_BYTES, &tmA, bar, row_a + 64 * j, k0);
        }
        if (!B_MN) {
          tma_load_2d_pair(b, &tmB, bar, k0, row_b);
        } else {
#pragma unroll
          for (int j = 0; j < HALF_ROWS / 64; ++j)
            tma_load_2d_pair(b + j * MN_BLOCK_BYTES, &tmB, bar, row_b + 64 * j, k0);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if ((!ok || *abort_flag) && rank == 0) {
      // Drain: the copies of both CTAs that this barrier counted land before
      // the pair exits.  (The peer's own waits give up only after the limit,
      // long after any copy it issued has landed.)
      int dummy_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if (armed_phase[s] >= 0)
          mbar_wait_cluster(&full[s], (uint32_t)armed_phase[s], &dummy_abort, err, SITE_DRAIN,
                            timeout_ns / 8);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (even CTA) ----------------
    constexpr uint32_t idesc = idesc_bf16(A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true, issued = false;
    for (int u = pair; u < sch.units && ok; u += npairs) {
      int mt, nt, split, kb0, kb1;
      sch.decode(u, mt, nt, split, kb0, kb1);
      if (!mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1u, abort_flag, err,
                             SITE_MMA_ACC_EMPTY, timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_cluster(&full[stage], phase, abort_flag, err, SITE_MMA_FULL,
                               timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
        const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t ad = A_MN ? desc_mnmajor(a_addr, k) : desc_kmajor(a_addr, k);
          const uint64_t bd = B_MN ? desc_mnmajor(b_addr, k) : desc_kmajor(b_addr, k);
          umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        }
        issued = true;
        umma_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit_pair(&acc_full[acc], 0x3);  // both halves of the tile are ready
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if ((!ok || *abort_flag) && issued) {
      // Drain: wait until every MMA issued so far has completed.
      int dummy_abort = 0;
      umma_commit_pair(drain, 0x1);
      mbar_wait_cluster(drain, 0, &dummy_abort, err, SITE_DRAIN, timeout_ns / 8);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs, 128 rows each) ----------------
    const int quarter = warp & 3;
    const uint32_t acc_empty_leader0 = mapa_shared(smem_u32(&acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = mapa_shared(smem_u32(&acc_empty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = pair; u < sch.units; u += npairs) {
      int mt, nt, split, kb0, kb1;
      sch.decode(u, mt, nt, split, kb0, kb1);
      const int row = mt * BM + (int)rank * HALF_ROWS + quarter * 32 + lane;
      constexpr bool kPre = HasPrefetch<Epi>::value;
      using Pre = typename std::conditional<kPre, typename PreOf<Epi, kPre>::type, NoPre>::type;
      Pre pre[kPre ? BN / 32 : 1];
      if constexpr (kPre) {
        if (row < M) {
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            if (nt * BN + c * 32 < N) epi.prefetch(row, nt * BN + c * 32, pre[c]);
        }
      }
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_cluster(&acc_full[acc], acc_phase, abort_flag, err, SITE_EPI_ACC_FULL,
                               timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      float row_acc = 0.f;
      if constexpr (kPre) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld_32cols(taddr + c * 32, v);
          const int col = nt * BN + c * 32;
          if (row < M && col < N) row_acc += epi.apply_pre(row, col, v, split, pre[c]);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld_32cols(taddr + c * 32, v);
          const int col = nt * BN + c * 32;
          if (row < M && col < N) row_acc += epi.template apply<32>(row, col, v, split);
        }
      }
      if (Epi::kRowReduce && row < M) epi.row_end(row, nt * BN, row_acc);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? acc_empty_leader1 : acc_empty_leader0);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still touch it
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace tc
}  // namespace nc
