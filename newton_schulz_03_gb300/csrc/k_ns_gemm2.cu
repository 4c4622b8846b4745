// k_ns_gemm2.cu -- the Newton-Schulz products on CTA pairs (tcgen05
// cta_group::2), 256 x 256 output tiles per pair.
//
// Same three products as k_ns_gemm.cu (Gram A = alpha X X^T, square
// B' = a I + b A + c A A, update X' = alpha B' X; "Frontier Pre-training at
// Microsoft AI", Method details §5, resharding step 3), scheduled on
// clusters of two CTAs on two SMs:
//   * each CTA stages its own 128-row half of the A-side operand and its own
//     128-column half of the B-side operand (TMA, no multicast), so a pair
//     streams one 256 x 64 A tile and one 64 x 256 B tile per stage while
//     each SM reads only 32 KB of shared memory per stage;
//   * the TMA completions of both CTAs are counted on the even CTA's "full"
//     barrier; one thread of the even CTA issues tcgen05.mma.cta_group::2
//     (M = 256, N = 256, K = 16) and its commits arrive on both CTAs'
//     barriers (multicast);
//   * each CTA's TMEM holds its 128 rows x 256 columns of the accumulator
//     (two accumulators, 512 columns); both CTAs run the epilogue on their
//     own rows and report back to the even CTA's "tmem empty" barrier.  The
//     epilogue writes 32 x 32 BF16 chunks through (64-byte swizzled) shared
//     memory with TMA stores;
//   * set-up (barriers, TMEM, tensor-map prefetch) runs before
//     griddepcontrol.wait, so under programmatic dependent launch it
//     overlaps the previous kernel's tail.
// Symmetric products compute AND store only the pair tiles (i, j) with
// i <= j over 256-blocks (diagonal tiles in full).  Their consumers read a
// block left of the diagonal, (I, K) with K < I, as the transpose of the
// stored block (K, I): the producer loads it as an MN-major tile and the
// MMA takes it through the operand-major bit of the instruction
// descriptor, chosen per 64-wide K block.  Nothing is stored twice.
// MN-major tiles (these transposed blocks and the X operand of the update)
// are fetched with one copy through a 4-D view of the matrix (64 columns,
// rows, 64-column chunks, matrix) when the column count is a multiple of
// 64; otherwise as one 64 x 64 box per chunk.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "launch.cuh"
#include "ns_common.cuh"
#include "sm103_ptx.cuh"

namespace muon {
namespace {

using namespace nsk;

constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kPairM = 256;                     // pair tile rows
constexpr int kPairN = 256;                     // pair tile columns
constexpr int kHalf = 128;                      // rows / columns staged per CTA
constexpr int kABytes = kHalf * kBK * 2;        // 16 KB
constexpr int kBBytes = kHalf * kBK * 2;        // 16 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB per CTA
constexpr uint32_t kPairTxBytes = 2u * kStageBytes;
constexpr int kStages = 6;
constexpr int kTmemCols = 2 * kPairN;           // two 256-column accumulators
// After the operand ring: the epilogue's staging buffers (4 warps x 2 x
// 2 KB, for TMA stores), inside a 32 KB region.
constexpr int kTailPad = 32 * 1024;
constexpr int kStageOutBytes = 4096;   // per epilogue warp
constexpr int kSmemBytes = kStages * kStageBytes + kTailPad + 1024 + 256;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    ns_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_at,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_bt,
                        const __grid_constant__ CUtensorMap tmap_out, const NsArgs p) {
  // A-side operand: rows of X (GRAM), of A (POLY) or of B (UPDATE); A and B
  // are stored as upper 256-block triangles.  B-side operand: rows of X
  // (GRAM), of A (POLY), or X as an MN-major operand (UPDATE).
  // tmap_a / tmap_b: K-major boxes (64 x 128); tmap_at / tmap_bt: 64 x 64
  // boxes of the same tensors, for blocks read transposed.
  constexpr bool kSymA = (MODE != kGram);   // A-side source is upper-stored
  constexpr bool kSymB = (MODE == kPoly);   // B-side source is upper-stored
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kTailPad);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], 2 * kEpiWarps * 32);  // both CTAs' epilogues
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmap_a);
    ptx::tma_prefetch_desc(&tmap_b);
    if (kSymA) ptx::tma_prefetch_desc(&tmap_at);
    if (kSymB) ptx::tma_prefetch_desc(&tmap_bt);
    ptx::tma_prefetch_desc(&tmap_out);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // barriers of both CTAs initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Set-up above overlaps the previous kernel's tail; its outputs are read
  // only from here on.
  grid_dep_wait();
  grid_dep_launch();
  const int num_kb = (p.K + kBK - 1) / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int t = pair; t < p.total_tiles && ok; t += npairs) {
        int mat, ti, tj;
        decode_tile_banded(p, MODE, t, mat, ti, tj);
        const int rowA = ti * kPairM + static_cast<int>(rank) * kHalf;
        const int colB = tj * kPairN + static_cast<int>(rank) * kHalf;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = ptx::mapa_shared(ptx::smem_addr(&full[stage]), 0);
          if (leader) ptx::mbar_arrive_expect_tx(&full[stage], kPairTxBytes);
          uint8_t* sa = smem + stage * kStageBytes;
          uint8_t* sb = sa + kABytes;
          const int kblk = (kb * kBK) / kPairM;   // 256-block of this K slice
          if (kSymA && kblk < ti) {
            // Left of the diagonal: the transpose of stored block (kblk, ti).
            if (p.mn4d) {
              ptx::tma_load_4d_pair(sa, &tmap_at, full_leader, 0, kb * kBK, rowA / 64, mat);
            } else {
#pragma unroll
              for (int q = 0; q < kHalf / 64; ++q)
                ptx::tma_load_3d_pair(sa + q * (kBK * 128), &tmap_at, full_leader, rowA + q * 64,
                                      kb * kBK, mat);
            }
          } else {
            ptx::tma_load_3d_pair(sa, &tmap_a, full_leader, kb * kBK, rowA, mat);
          }
          if (MODE == kUpdate || (kSymB && kblk < tj)) {
            // X as the MN-major operand, or the transpose of a stored block.
            const CUtensorMap* mb = (MODE == kUpdate) ? &tmap_b : &tmap_bt;
            if (p.mn4d) {
              ptx::tma_load_4d_pair(sb, mb, full_leader, 0, kb * kBK, colB / 64, mat);
            } else {
#pragma unroll
              for (int q = 0; q < kHalf / 64; ++q)
                ptx::tma_load_3d_pair(sb + q * (kBK * 128), mb, full_leader, colB + q * 64,
                                      kb * kBK, mat);
            }
          } else {
            ptx::tma_load_3d_pair(sb, &tmap_b, full_leader, kb * kBK, colB, mat);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
      // Drain: a stage is free again once the MMAs that read it completed
      // (their commit arrives on this CTA's empty barrier); wait (bounded)
      // for the last stages this CTA filled.
      const int pending = issued < kStages ? issued : kStages;
      for (int j = 0; j < pending; ++j) {
        if (stage == 0) {
          stage = kStages;
          phase ^= 1u;
        }
        --stage;
        ptx::mbar_wait_cluster(&empty[stage], phase, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = pair; t < p.total_tiles && ok; t += npairs) {
        if (!ptx::mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        int mat, ti, tj;
        decode_tile_banded(p, MODE, t, mat, ti, tj);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kPairN);
        for (int kb = 0; kb < num_kb; ++kb) {
          const int kblk = (kb * kBK) / kPairM;
          const uint32_t a_mn = (kSymA && kblk < ti) ? 1u : 0u;
          const uint32_t b_mn = (MODE == kUpdate || (kSymB && kblk < tj)) ? 1u : 0u;
          const uint32_t idesc = ptx::idesc_bf16_f32(kPairM, kPairN, a_mn, b_mn);
          if (!ptx::mbar_wait_cluster(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // K-major: a K step of 16 is +32 bytes inside the swizzle row.
            // MN-major: 64-wide chunks kBK*128 bytes apart, a K step of 16
            // rows is +2048 bytes.
            const uint64_t adesc = a_mn ? ptx::smem_desc_sw128(sa + k * 16 * 128, kBK * 128, 1024)
                                        : ptx::smem_desc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bdesc = b_mn ? ptx::smem_desc_sw128(sb + k * 16 * 128, kBK * 128, 1024)
                                        : ptx::smem_desc_sw128(sb + k * 32, 16, 1024);
            ptx::tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          ptx::tc_commit_pair_multicast(&empty[stage], 0x3);  // frees the stage in both CTAs
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit_pair_multicast(&tmem_full[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
      ptx::tc_commit_pair(drain);
      ptx::mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;
    const int r_tile = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t empty_leader0 = ptx::mapa_shared(ptx::smem_addr(&tmem_empty[0]), 0);
    const uint32_t empty_leader1 = ptx::mapa_shared(ptx::smem_addr(&tmem_empty[1]), 0);
    uint8_t* stage_out = smem + kStages * kStageBytes + (warp - 2) * kStageOutBytes;
    int issued = 0;
    for (int t = pair; t < p.total_tiles; t += npairs) {
      int mat, ti, tj;
      decode_tile_banded(p, MODE, t, mat, ti, tj);
      const int rb = ti * (kPairM / kBM) + static_cast<int>(rank);  // 128-row block index
      EpiAux<MODE, kPairN, false> aux;
      aux.start(p, mat, rb * kBM + r_tile, rb, tj * kPairN);   // loads overlap the MMAs
      const bool got = ptx::mbar_wait_cluster(&tmem_full[acc], acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicOr(p.err, kDevErrTimeout);
        }
        break;
      }
      ptx::tc_fence_after();
      float alpha = 1.f;
      if (p.inv_norm != nullptr) {
        const float s = p.inv_norm[mat];
        alpha = (MODE == kGram) ? s * s : s;
      }
      epilogue_tile_tma<MODE, kPairN>(
          p, &tmap_out,
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * kPairN),
          mat, rb * kBM + r_tile, rb * kBM + quad * 32, aux, alpha, stage_out, issued, lane);
      ptx::tc_fence_before();
      ptx::mbar_arrive_cluster(acc ? empty_leader1 : empty_leader0);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // All TMA stores of this warp complete before the CTA can exit.
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still touch it
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Row tiles per band of the tile order: the band's 256-row blocks of the
// left operand (K elements each) should take about kBandBytes, so that
// they stay in L2 while the band's columns go by; bands are then evened
// out over the matrix's row tiles.
constexpr double kBandBytes = 40.0 * (1 << 20);

int band_rows(int tiles_m, int K) {
  int g = static_cast<int>(kBandBytes / (double(kPairM) * K * 2.0));
  if (g < 1) g = 1;
  if (g > tiles_m) g = tiles_m;
  const int bands = (tiles_m + g - 1) / g;
  return (tiles_m + bands - 1) / bands;
}

template <int MODE>
cudaError_t pair_attr() {
  return cudaFuncSetAttribute(ns_gemm_pair_kernel<MODE>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

// Pairs that can be resident at once (clusters must fit a GPC).
template <int MODE>
int max_pairs() {
  static int cached = -1;
  if (cached < 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, ns_gemm_pair_kernel<MODE>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    cached = n;
  }
  return cached;
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tat, const CUtensorMap& tb,
                        const CUtensorMap& tbt, const CUtensorMap& tout, const NsArgs& p,
                        int grid_cap, cudaStream_t stream) {
  if (p.total_tiles <= 0) return cudaSuccess;
  int pairs = max_pairs<MODE>();
  if (pairs > grid_cap / 2) pairs = grid_cap / 2;
  if (pairs > p.total_tiles) pairs = p.total_tiles;
  if (pairs < 1) pairs = 1;
  return launch_pdl(ns_gemm_pair_kernel<MODE>, dim3(2 * pairs), dim3(kThreads), kSmemBytes, stream,
                    ta, tat, tb, tbt, tout, p);
}

}  // namespace

cudaError_t ns_pair_init() {
  cudaError_t e;
  if ((e = pair_attr<kGram>()) != cudaSuccess) return e;
  if ((e = pair_attr<kPoly>()) != cudaSuccess) return e;
  if ((e = pair_attr<kUpdate>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t ns_pair_gram(const CUtensorMap& tx, const CUtensorMap& tout, int m, int n, int count,
                         BatchView A_out,
                         const float* inv_norm, int* err, int grid_cap, cudaStream_t stream) {
  NsArgs p{};
  p.m = m;
  p.n = n;
  p.K = n;
  p.tiles_m = (m + kPairM - 1) / kPairM;
  p.tiles_n = p.tiles_m;
  p.tiles_per_matrix = p.tiles_m * (p.tiles_m + 1) / 2;
  p.total_tiles = p.tiles_per_matrix * count;
  p.group_rows = band_rows(p.tiles_m, p.K);
  p.out_cols = m;
  p.out = static_cast<__nv_bfloat16*>(const_cast<void*>(A_out.ptr));
  p.out_ld = A_out.ld;
  p.out_ms = A_out.ms;
  p.inv_norm = inv_norm;
  p.err = err;
  return launch_pair<kGram>(tx, tx, tx, tx, tout, p, grid_cap, stream);
}

cudaError_t ns_pair_poly(const CUtensorMap& ta, const CUtensorMap& ta_t, const CUtensorMap& tout,
                         int m, int count, BatchView A, BatchView B_out, float a, float b, float c,
                         int* err, int grid_cap, cudaStream_t stream, int mn4d) {
  NsArgs p{};
  p.mn4d = mn4d;
  p.m = m;
  p.n = m;
  p.K = m;
  p.tiles_m = (m + kPairM - 1) / kPairM;
  p.tiles_n = p.tiles_m;
  p.tiles_per_matrix = p.tiles_m * (p.tiles_m + 1) / 2;
  p.total_tiles = p.tiles_per_matrix * count;
  p.group_rows = band_rows(p.tiles_m, p.K);
  p.out_cols = m;
  p.out = static_cast<__nv_bfloat16*>(const_cast<void*>(B_out.ptr));
  p.out_ld = B_out.ld;
  p.out_ms = B_out.ms;
  p.aux = static_cast<const __nv_bfloat16*>(A.ptr);
  p.aux_ld = A.ld;
  p.aux_ms = A.ms;
  p.c0 = b;
  p.c1 = c;
  p.c2 = a;
  p.err = err;
  return launch_pair<kPoly>(ta, ta_t, ta, ta_t, tout, p, grid_cap, stream);
}

cudaError_t ns_pair_update(const CUtensorMap& tb, const CUtensorMap& tb_t, const CUtensorMap& tx,
                           const CUtensorMap& tout, int m, int n, int count, BatchView X_out,
                           const float* inv_norm, int* err, int grid_cap, cudaStream_t stream,
                           int mn4d) {
  NsArgs p{};
  p.mn4d = mn4d;
  p.m = m;
  p.n = n;
  p.K = m;
  p.tiles_m = (m + kPairM - 1) / kPairM;
  p.tiles_n = (n + kPairN - 1) / kPairN;
  p.tiles_per_matrix = p.tiles_m * p.tiles_n;
  p.total_tiles = p.tiles_per_matrix * count;
  p.group_rows = band_rows(p.tiles_m, p.K);
  p.out_cols = n;
  p.out = static_cast<__nv_bfloat16*>(const_cast<void*>(X_out.ptr));
  p.out_ld = X_out.ld;
  p.out_ms = X_out.ms;
  p.inv_norm = inv_norm;
  p.err = err;
  return launch_pair<kUpdate>(tb, tb_t, tx, tx, tout, p, grid_cap, stream);
}

}  // namespace muon
