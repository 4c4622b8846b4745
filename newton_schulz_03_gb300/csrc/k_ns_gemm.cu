// k_ns_gemm.cu -- batched symmetric Newton-Schulz products on tcgen05.
//
// The pages orthogonalise each whole momentum matrix "with a Newton-Schulz
// operator customised for symmetric matrices" (Frontier Pre-training at
// Microsoft AI, Method details §5, resharding step 3; "symmetry-aware
// Newton-Schulz kernels" in "Microsoft Reveals MAI-Base-2 Training Recipe",
// section "How to Make Parameter Updates Faster and More Stable?").  One
// quintic iteration on a wide BF16 matrix X (m x n, m <= n) is three
// products, each one launch of the kernel below over a whole batch of
// same-shape matrices:
//
//   GRAM    A  = alpha X X^T          K = n   symmetric
//   POLY    B' = a I + b A + c A A    K = m   symmetric
//   UPDATE  X' = alpha B' X           K = m   all tiles
// (the linear term a X of the quintic is folded into the diagonal of B').
//
// alpha folds the Frobenius pre-normalisation into the first iteration
// (alpha = 1/s^2 for the Gram product and 1/s for the update).
//
// Kernel shape (one CTA per SM, persistent over a static tile list):
//   warp 0      TMA producer: 128-byte-swizzled operand tiles into a
//               multi-stage shared-memory ring (mbarrier full/empty).
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer:
//               128 x BN x 16 BF16 MMAs accumulate in FP32 in TMEM; two
//               accumulators so the epilogue of tile i overlaps tile i+1.
//   warps 2..5  epilogue: tcgen05.ld TMEM -> registers, fused polynomial
//               combine, BF16 round, global store (and mirrored store for
//               the symmetric products).
// Operands: A-side tiles are K-major (rows of X, A or B); the UPDATE
// B-side operand X is MN-major (n contiguous) and is read through the
// transposed-operand mode of the MMA, so X is never transposed in memory.
// Matrix edges: the tensor maps are 3-D (cols, rows, matrix), so loads past
// a matrix edge read zeros, which leaves the products exact; stores are
// bounds-checked.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "kernels.h"
#include "launch.cuh"
#include "ns_common.cuh"
#include "sm103_ptx.cuh"

namespace muon {
namespace {

using namespace nsk;

constexpr int kThreads = 192; // 6 warps
constexpr int kEpiWarps = 4;

template <int BN>
struct TileCfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + kBarrierBytes;
  static_assert(kTmemCols <= 512, "two accumulators must fit TMEM");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    ns_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const NsArgs p) {
  using Cfg = TileCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kStages * Cfg::kStageBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* tmem_full = empty + Cfg::kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], kEpiWarps * 32);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmap_a);
    ptx::tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, Cfg::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Set-up above overlaps the previous kernel's tail; its outputs are read
  // only from here on.
  grid_dep_wait();
  grid_dep_launch();

  const int num_kb = (p.K + kBK - 1) / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        int mat, ti, tj;
        decode_tile(p, MODE, kBM, BN, t, mat, ti, tj);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * Cfg::kStageBytes;
          uint8_t* sb = sa + Cfg::kABytes;
          ptx::mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
          ptx::tma_load_3d(sa, &tmap_a, &full[stage], kb * kBK, ti * kBM, mat);
          if (MODE == kUpdate) {
#pragma unroll
            for (int q = 0; q < BN / 64; ++q)
              ptx::tma_load_3d(sb + q * (kBK * 128), &tmap_b, &full[stage], tj * BN + q * 64,
                               kb * kBK, mat);
          } else {
            ptx::tma_load_3d(sb, &tmap_b, &full[stage], kb * kBK, tj * BN, mat);
          }
          ++issued;
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
      // Drain: wait (bounded) until the last loads issued have landed, so
      // no copy is still writing shared memory when the CTA exits.
      const int pending = issued < Cfg::kStages ? issued : Cfg::kStages;
      for (int j = 0; j < pending; ++j) {
        if (stage == 0) {
          stage = Cfg::kStages;
          phase ^= 1u;
        }
        --stage;
        ptx::mbar_wait(&full[stage], phase, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, BN, 0, MODE == kUpdate ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        if (!ptx::mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(smem + stage * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // K-major, 128-byte swizzle: a K step of 16 BF16 is +32 bytes
            // inside the swizzle row; 8-row groups are 1024 bytes apart.
            const uint64_t adesc = ptx::smem_desc_sw128(sa + k * 32, 16, 1024);
            uint64_t bdesc;
            if (MODE == kUpdate) {
              // MN-major, 128-byte swizzle: 64-column chunks kBK*128 bytes
              // apart (leading), 8-row K groups 1024 bytes apart (stride);
              // a K step of 16 rows is +2048 bytes.
              bdesc = ptx::smem_desc_sw128(sb + k * 16 * 128, kBK * 128, 1024);
            } else {
              bdesc = ptx::smem_desc_sw128(sb + k * 32, 16, 1024);
            }
            ptx::tc_mma_bf16(d_tmem, adesc, bdesc, kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          ptx::tc_commit(&empty[stage]);  // frees the stage when the MMAs finish
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit(&tmem_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, kDevErrTimeout);
      }
      // Drain: all MMAs of this thread complete before TMEM is released.
      ptx::tc_commit(drain);
      ptx::mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;             // TMEM lane quadrant of this warp
    const int r_tile = quad * 32 + lane;   // accumulator row of this thread
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      int mat, ti, tj;
      decode_tile(p, MODE, kBM, BN, t, mat, ti, tj);
      EpiAux<MODE, BN, true> aux;
      aux.start(p, mat, ti * kBM + r_tile, ti, tj * BN);   // loads overlap the MMAs
      const bool got = ptx::mbar_wait(&tmem_full[acc], acc_phase, abort_flag);
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
      epilogue_tile<MODE, BN>(
          p, tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN),
          mat, ti * kBM + r_tile, aux, alpha);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tmem_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();  // dealloc is warp-collective
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

thread_local char g_encode_err[256] = "";

EncodeFn get_encode_fn() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  }
  return fn;
}

// 3-D BF16 map over a batch: (cols, rows, count), 128-byte swizzle,
// box (64, box_rows, 1), zero fill outside the matrix.
cudaError_t make_map(CUtensorMap* map, BatchView v, int cols, int rows, int count, int box_rows) {
  EncodeFn enc = get_encode_fn();
  if (enc == nullptr) {
    snprintf(g_encode_err, sizeof(g_encode_err), "cuTensorMapEncodeTiled unavailable");
    return cudaErrorNotSupported;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(count)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(v.ld) * 2,
                                 static_cast<cuuint64_t>(v.ms) * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v.ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_encode_err, sizeof(g_encode_err),
             "cuTensorMapEncodeTiled failed (%d): cols=%d rows=%d count=%d ld=%lld ms=%lld box=%d",
             static_cast<int>(r), cols, rows, count, static_cast<long long>(v.ld),
             static_cast<long long>(v.ms), box_rows);
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// Output map for the TMA-store epilogue: 32 x 32 boxes with the 64-byte
// swizzle (the staging buffer holds the 32 rows x 64 bytes in that
// pattern, so a quarter-warp's row writes hit distinct banks).
cudaError_t make_map_out(CUtensorMap* map, BatchView v, int cols, int rows, int count) {
  EncodeFn enc = get_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(count)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(v.ld) * 2,
                                 static_cast<cuuint64_t>(v.ms) * 2};
  const cuuint32_t box[3] = {32u, 32u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v.ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_encode_err, sizeof(g_encode_err), "output map encode failed (%d)",
             static_cast<int>(r));
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// 4-D view of a batch for MN-major operand tiles: (64 columns, rows,
// 64-column chunks, matrix).  A box (64, 64, chunks, 1) lands in shared
// memory as `chunks` consecutive 64 x 64 swizzled blocks -- the layout the
// MN-major descriptor expects -- in one copy.  Needs cols % 64 == 0.
cudaError_t make_map_mn4d(CUtensorMap* map, BatchView v, int cols, int rows, int count,
                          int chunks) {
  EncodeFn enc = get_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64),
                              static_cast<cuuint64_t>(count)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(v.ld) * 2, 128u,
                                 static_cast<cuuint64_t>(v.ms) * 2};
  const cuuint32_t box[4] = {64u, 64u, static_cast<cuuint32_t>(chunks), 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v.ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_encode_err, sizeof(g_encode_err), "4-D map encode failed (%d)", static_cast<int>(r));
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <int MODE, int BN>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const NsArgs& p, int grid_cap,
                   cudaStream_t stream) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int grid = p.total_tiles < grid_cap ? p.total_tiles : grid_cap;
  return launch_pdl(ns_gemm_kernel<MODE, BN>, dim3(grid), dim3(kThreads), TileCfg<BN>::kSmemBytes,
                    stream, ta, tb, p);
}

template <int MODE, int BN>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(ns_gemm_kernel<MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TileCfg<BN>::kSmemBytes);
}

constexpr int kSymBN = 256;   // symmetric products: 128 x 256 tiles (triangular list)
constexpr int kUpdBN = 256;   // update product: 128 x 256 tiles

int sym_tiles_per_matrix(int tiles_m, int tiles_n) {
  const int ratio = kSymBN / kBM;
  int total = 0;
  for (int i = 0; i < tiles_m; ++i) total += tiles_n - i / ratio;
  return total;
}

}  // namespace

const char* ns_last_encode_error() { return g_encode_err; }

// Matrices with more than 128 rows (after the transpose to wide) run on CTA
// pairs; MUON_NS_PAIR=0 in the environment keeps every product on single
// CTAs (for comparisons).
bool use_pairs(int m) {
  static int enabled = -1;
  if (enabled < 0) {
    const char* v = getenv("MUON_NS_PAIR");
    enabled = (v != nullptr && v[0] == '0') ? 0 : 1;
  }
  return enabled == 1 && m > kBM;
}

cudaError_t ns_gemm_init() {
  cudaError_t e;
  if ((e = ns_pair_init()) != cudaSuccess) return e;
  if ((e = set_attr<kGram, kSymBN>()) != cudaSuccess) return e;
  if ((e = set_attr<kPoly, kSymBN>()) != cudaSuccess) return e;
  if ((e = set_attr<kUpdate, kUpdBN>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t ns_launch_gram(int m, int n, int count, BatchView X, BatchView A_out,
                           const float* inv_norm, int* err, int grid_cap, cudaStream_t stream) {
  if (use_pairs(m)) {
    CUtensorMap t128, tout;
    cudaError_t e = make_map(&t128, X, n, m, count, kBM);
    if (e == cudaSuccess) e = make_map_out(&tout, A_out, m, m, count);
    if (e != cudaSuccess) return e;
    return ns_pair_gram(t128, tout, m, n, count, A_out, inv_norm, err, grid_cap, stream);
  }
  // A-side rows in boxes of kBM, B-side rows in boxes of kSymBN.
  CUtensorMap tx, txb;
  cudaError_t e = make_map(&tx, X, n, m, count, kBM);
  if (e == cudaSuccess) e = make_map(&txb, X, n, m, count, kSymBN);
  if (e != cudaSuccess) return e;
  NsArgs p{};
  p.m = m;
  p.n = n;
  p.K = n;
  p.tiles_m = (m + kBM - 1) / kBM;
  p.tiles_n = (m + kSymBN - 1) / kSymBN;
  p.tiles_per_matrix = sym_tiles_per_matrix(p.tiles_m, p.tiles_n);
  p.total_tiles = p.tiles_per_matrix * count;
  p.out_cols = m;
  p.out = static_cast<__nv_bfloat16*>(const_cast<void*>(A_out.ptr));
  p.out_ld = A_out.ld;
  p.out_ms = A_out.ms;
  p.aux = nullptr;
  p.inv_norm = inv_norm;
  p.err = err;
  return launch<kGram, kSymBN>(tx, txb, p, grid_cap, stream);
}

cudaError_t ns_launch_poly(int m, int count, BatchView A, BatchView B_out, float a, float b,
                           float c, int* err, int grid_cap, cudaStream_t stream) {
  if (use_pairs(m)) {
    CUtensorMap t128, t64, tout;
    const int mn4d = (m % 64 == 0) ? 1 : 0;
    cudaError_t e = make_map(&t128, A, m, m, count, kBM);
    if (e == cudaSuccess)
      e = mn4d ? make_map_mn4d(&t64, A, m, m, count, 2) : make_map(&t64, A, m, m, count, kBK);
    if (e == cudaSuccess) e = make_map_out(&tout, B_out, m, m, count);
    if (e != cudaSuccess) return e;
    return ns_pair_poly(t128, t64, tout, m, count, A, B_out, a, b, c, err, grid_cap, stream,
                        mn4d);
  }
  CUtensorMap ta, tab;
  cudaError_t e = make_map(&ta, A, m, m, count, kBM);
  if (e == cudaSuccess) e = make_map(&tab, A, m, m, count, kSymBN);
  if (e != cudaSuccess) return e;
  NsArgs p{};
  p.m = m;
  p.n = m;
  p.K = m;
  p.tiles_m = (m + kBM - 1) / kBM;
  p.tiles_n = (m + kSymBN - 1) / kSymBN;
  p.tiles_per_matrix = sym_tiles_per_matrix(p.tiles_m, p.tiles_n);
  p.total_tiles = p.tiles_per_matrix * count;
  p.out_cols = m;
  p.out = static_cast<__nv_bfloat16*>(const_cast<void*>(B_out.ptr));
  p.out_ld = B_out.ld;
  p.out_ms = B_out.ms;
  p.aux = static_cast<const __nv_bfloat16*>(A.ptr);
  p.aux_ld = A.ld;
  p.aux_ms = A.ms;
  p.inv_norm = nullptr;
  p.c0 = b;
  p.c1 = c;
  p.c2 = a;
  p.err = err;
  return launch<kPoly, kSymBN>(ta, tab, p, grid_cap, stream);
}

cudaError_t ns_launch_update(int m, int n, int count, BatchView B, BatchView X, BatchView X_out,
                             const float* inv_norm, int* err, int grid_cap, cudaStream_t stream) {
  CUtensorMap tb, tx;
  cudaError_t e = make_map(&tb, B, m, m, count, kBM);
  if (e != cudaSuccess) return e;
  // X as the MN-major operand: boxes of 64 columns x 64 K-rows.
  e = make_map(&tx, X, n, m, count, kBK);
  if (e != cudaSuccess) return e;
  if (use_pairs(m)) {
    CUtensorMap tb64, tx4, tout;
    const int mn4d = (m % 64 == 0 && n % 64 == 0) ? 1 : 0;
    if (mn4d) {
      e = make_map_mn4d(&tb64, B, m, m, count, 2);
      if (e == cudaSuccess) e = make_map_mn4d(&tx4, X, n, m, count, 2);
    } else {
      e = make_map(&tb64, B, m, m, count, kBK);
      tx4 = tx;
    }
    if (e == cudaSuccess) e = make_map_out(&tout, X_out, n, m, count);
    if (e != cudaSuccess) return e;
    return ns_pair_update(tb, tb64, tx4, tout, m, n, count, X_out, inv_norm, err, grid_cap, stream,
                          mn4d);
  }
  NsArgs p{};
  p.m = m;
  p.n = n;
  p.K = m;
  p.tiles_m = (m + kBM - 1) / kBM;
  p.tiles_n = (n + kUpdBN - 1) / kUpdBN;
  p.tiles_per_matrix = p.tiles_m * p.tiles_n;
  p.total_tiles = p.tiles_per_matrix * count;
  p.out_cols = n;
  p.out = static_cast<__nv_bfloat16*>(const_cast<void*>(X_out.ptr));
  p.out_ld = X_out.ld;
  p.out_ms = X_out.ms;
  p.inv_norm = inv_norm;
  p.err = err;
  return launch<kUpdate, kUpdBN>(tb, tx, p, grid_cap, stream);
}

}  // namespace muon
