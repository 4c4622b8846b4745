// ns_common.cuh -- pieces shared by the Newton-Schulz product kernels:
// argument block, tile decoding, and the fused epilogues (TMEM -> registers
// -> polynomial combine -> BF16 -> global): direct stores, mirrored for the
// symmetric products, in the single-CTA kernels; TMA stores of the upper
// 256-block triangle in the CTA-pair kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace muon {
namespace nsk {

enum NsMode : int { kGram = 0, kPoly = 1, kUpdate = 2 };

constexpr int kBM = 128;   // accumulator rows per CTA (TMEM lanes)
constexpr int kBK = 64;    // K per pipeline stage: one 128-byte swizzle row of BF16

struct NsArgs {
  int32_t m, n;               // X is m x n; A, B are m x m
  int32_t K;                  // reduction length
  int32_t tiles_m;            // row tiles per matrix (tile rows = rows per tile)
  int32_t tiles_n;            // column tiles per matrix
  int32_t tiles_per_matrix;
  int32_t total_tiles;
  int32_t out_cols;           // columns of the output matrix
  __nv_bfloat16* out;
  int64_t out_ld, out_ms;
  const __nv_bfloat16* aux;   // POLY: A (the only product with an auxiliary operand)
  int64_t aux_ld, aux_ms;
  const float* inv_norm;      // alpha source (NULL: alpha = 1)
  float c0, c1, c2;           // POLY: (b, c, a): B' = a I + b A + c A A
  int* err;
  int32_t mn4d;               // MN-major operand maps are 4-D chunk views (one copy per operand)
  int32_t group_rows;         // pair kernels: row tiles per band of the tile order (>= 1)
};

// Tile t -> (matrix, row tile, column tile).  Symmetric products list, per
// row tile i, the column tiles j >= floor(i * tile_rows / tile_cols) (the
// first holds the diagonal); the update product lists every tile.
__device__ __forceinline__ void decode_tile(const NsArgs& p, int mode, int tile_rows,
                                            int tile_cols, int t, int& mat, int& ti, int& tj) {
  mat = t / p.tiles_per_matrix;
  int l = t - mat * p.tiles_per_matrix;
  if (mode == kUpdate) {
    ti = l / p.tiles_n;
    tj = l - ti * p.tiles_n;
  } else {
    int i = 0;
    while (l >= p.tiles_n - (i * tile_rows) / tile_cols) {
      l -= p.tiles_n - (i * tile_rows) / tile_cols;
      ++i;
    }
    ti = i;
    tj = (i * tile_rows) / tile_cols + l;
  }
}

// Tile order of the CTA-pair kernels (square 256 x 256 tiles): a matrix's
// tiles go band by band, a band being `group_rows` consecutive row tiles,
// and inside a band column by column (each column's rows in order).  The
// pairs running at one time then share a few row blocks of the left
// operand and a few column blocks of the right one, a working set that L2
// holds, instead of sweeping a whole row of tiles -- and so the whole right
// operand -- per row block.  Symmetric products list only the tiles
// (i, j) with i <= j: column j of a band holds its rows up to j.
__device__ __forceinline__ void decode_tile_banded(const NsArgs& p, int mode, int t, int& mat,
                                                   int& ti, int& tj) {
  mat = t / p.tiles_per_matrix;
  int l = t - mat * p.tiles_per_matrix;
  const int T = p.tiles_m, G = p.group_rows;
  if (mode == kUpdate) {
    const int band = l / (G * p.tiles_n);
    const int r0 = band * G;
    const int rows = min(G, T - r0);
    l -= r0 * p.tiles_n;
    tj = l / rows;
    ti = r0 + (l - tj * rows);
    return;
  }
  int r0 = 0;
  for (;;) {
    const int r1 = min(r0 + G, T);
    const int k = r1 - r0;
    const int tri = k * (k + 1) / 2;          // columns r0 .. r1-1: 1, 2, .., k rows
    const int cnt = tri + (T - r1) * k;       // columns r1 .. T-1: k rows each
    if (l < cnt) {
      if (l < tri) {
        int c = 1;
        while (l >= c) {
          l -= c;
          ++c;
        }
        tj = r0 + c - 1;
        ti = r0 + l;
      } else {
        l -= tri;
        tj = r1 + l / k;
        ti = r0 + (l - (l / k) * k);
      }
      return;
    }
    l -= cnt;
    r0 = r1;
  }
}

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Epilogue of one accumulator: this thread owns output row `grow` and the
// BN columns col0 .. col0+BN-1, read from TMEM at `taddr` (lane and column
// already set).  `rb` is the kBM-row block index of the row (symmetric
// products: a 128-column sub-block left of it is skipped, right of it is
// also stored mirrored).
//
// With MIRROR the symmetric result is stored in full (sub-blocks left of
// the diagonal skipped, right of it stored twice); without it only the
// tile as computed is stored (upper-triangle storage).
//
// The auxiliary operand (A, read by POLY only) does not depend on the
// accumulator, so its first kPrefetch chunks are loaded before the wait
// for the accumulator (EpiAux::start) and the rest kPrefetch chunks ahead.
template <int MODE, int BN, bool MIRROR>
struct EpiAux {
  static constexpr int kChunks = BN / 32;
  static constexpr int kPrefetch = (kChunks < 4) ? kChunks : 4;
  uint4 pre[kPrefetch][4];
  const __nv_bfloat16* row;   // aux row of this thread (POLY only)
  int col0, rb;
  bool row_ok;
  int out_cols;

  __device__ __forceinline__ bool live(int cb) const {
    const int g0 = col0 + cb * 32;
    const bool below = MIRROR && (MODE != kUpdate) && (g0 / kBM < rb);
    return row_ok && g0 < out_cols && !below;
  }
  __device__ __forceinline__ bool full(int cb) const { return col0 + cb * 32 + 32 <= out_cols; }
  __device__ __forceinline__ void load(int cb) {
    if (MODE == kPoly && cb < kChunks && live(cb) && full(cb)) {
      const uint4* src = reinterpret_cast<const uint4*>(row + col0 + cb * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) pre[cb % kPrefetch][q] = __ldg(src + q);
    }
  }
  __device__ __forceinline__ void start(const NsArgs& p, int mat, int grow, int rb_, int col0_) {
    col0 = col0_;
    rb = rb_;
    row_ok = grow < p.m;
    out_cols = p.out_cols;
    row = (MODE != kPoly) ? nullptr
                          : p.aux + static_cast<int64_t>(mat) * p.aux_ms +
                                static_cast<int64_t>(grow) * p.aux_ld;
#pragma unroll
    for (int cb = 0; cb < kPrefetch; ++cb) load(cb);
  }
};

template <int MODE, int BN, bool MIRROR>
__device__ __forceinline__ void epilogue_tile(const NsArgs& p, uint32_t taddr, int mat, int grow,
                                              EpiAux<MODE, BN, MIRROR>& aux, float alpha) {
  constexpr int kChunks = BN / 32;
  constexpr int kPre = EpiAux<MODE, BN, MIRROR>::kPrefetch;
  __nv_bfloat16* out_m = p.out + static_cast<int64_t>(mat) * p.out_ms;

#pragma unroll
  for (int cb = 0; cb < kChunks; ++cb) {
    uint32_t v[32];
    __syncwarp();  // tcgen05.ld is warp-collective: keep the warp converged
    ptx::tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(cb * 32), v);
    ptx::tmem_ld_wait();
    const int gcol0 = aux.col0 + cb * 32;
    if (aux.live(cb)) {
      const bool full_chunk = aux.full(cb);
      const bool mirror = MIRROR && (MODE != kUpdate) && (gcol0 / kBM > aux.rb);
      float f[32];
      if (MODE != kPoly) {
        // Gram: alpha X X^T.  Update: alpha (a I + b A + c A^2) X, the a X
        // term being folded into the square product's diagonal.
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = alpha * __uint_as_float(v[e]);
      } else {
        float x[32];
        if (full_chunk) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 u = aux.pre[cb % kPre][q];
            x[q * 8 + 0] = bf16lo(u.x); x[q * 8 + 1] = bf16hi(u.x);
            x[q * 8 + 2] = bf16lo(u.y); x[q * 8 + 3] = bf16hi(u.y);
            x[q * 8 + 4] = bf16lo(u.z); x[q * 8 + 5] = bf16hi(u.z);
            x[q * 8 + 6] = bf16lo(u.w); x[q * 8 + 7] = bf16hi(u.w);
          }
        } else {
          const uint16_t* a16 = reinterpret_cast<const uint16_t*>(aux.row + gcol0);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            x[e] = (gcol0 + e < p.out_cols) ? __uint_as_float(static_cast<uint32_t>(a16[e]) << 16)
                                            : 0.f;
        }
        // B' = b A + c A^2, plus a on the diagonal (only in the chunk
        // holding column `grow`).
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = fmaf(p.c1, __uint_as_float(v[e]), p.c0 * x[e]);
        const int dg = grow - gcol0;
        if (dg >= 0 && dg < 32) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e == dg) f[e] = fmaf(p.c1, __uint_as_float(v[e]), fmaf(p.c0, x[e], p.c2));
        }
      }
      __nv_bfloat16* orow = out_m + static_cast<int64_t>(grow) * p.out_ld + gcol0;
      if (full_chunk) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          u.x = pack_bf16(f[q * 8 + 0], f[q * 8 + 1]);
          u.y = pack_bf16(f[q * 8 + 2], f[q * 8 + 3]);
          u.z = pack_bf16(f[q * 8 + 4], f[q * 8 + 5]);
          u.w = pack_bf16(f[q * 8 + 6], f[q * 8 + 7]);
          reinterpret_cast<uint4*>(orow)[q] = u;
        }
      } else {
        uint16_t* o16 = reinterpret_cast<uint16_t*>(orow);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (gcol0 + e < p.out_cols) o16[e] = to_bf16_bits(f[e]);
      }
      if (mirror) {
        // Element (grow, gcol) above the diagonal is also element (gcol, grow).
        uint16_t* o16 = reinterpret_cast<uint16_t*>(out_m);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (gcol0 + e < p.out_cols)
            o16[static_cast<int64_t>(gcol0 + e) * p.out_ld + grow] = to_bf16_bits(f[e]);
      }
    }
    aux.load(cb + kPre);
  }
  __syncwarp();
}

// Epilogue through shared memory and TMA stores (upper-triangle storage,
// no mirror): each 32 x 32 chunk of this warp's rows is packed to BF16 in
// a 2 KB staging buffer of the warp (two per warp, alternating) and
// written by one TMA store, which also clips rows and columns past the
// matrix.  `stage` is the warp's 4 KB staging area, `issued` its running
// count of stores (for buffer reuse).  row0 is the warp's first row.
template <int MODE, int BN>
__device__ __forceinline__ void epilogue_tile_tma(const NsArgs& p, const CUtensorMap* tmap_out,
                                                  uint32_t taddr, int mat, int grow, int row0,
                                                  EpiAux<MODE, BN, false>& aux, float alpha,
                                                  uint8_t* stage, int& issued, int lane) {
  constexpr int kChunks = BN / 32;
  constexpr int kPre = EpiAux<MODE, BN, false>::kPrefetch;
  const bool warp_rows = row0 < p.m;   // some row of this warp is inside the matrix
#pragma unroll
  for (int cb = 0; cb < kChunks; ++cb) {
    uint32_t v[32];
    __syncwarp();
    ptx::tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(cb * 32), v);
    ptx::tmem_ld_wait();
    const int gcol0 = aux.col0 + cb * 32;
    if (warp_rows && gcol0 < p.out_cols) {
      float f[32];
      if (MODE != kPoly) {
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = alpha * __uint_as_float(v[e]);
      } else {
        float x[32];
        if (aux.live(cb) && aux.full(cb)) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 u = aux.pre[cb % kPre][q];
            x[q * 8 + 0] = bf16lo(u.x); x[q * 8 + 1] = bf16hi(u.x);
            x[q * 8 + 2] = bf16lo(u.y); x[q * 8 + 3] = bf16hi(u.y);
            x[q * 8 + 4] = bf16lo(u.z); x[q * 8 + 5] = bf16hi(u.z);
            x[q * 8 + 6] = bf16lo(u.w); x[q * 8 + 7] = bf16hi(u.w);
          }
        } else {
          const uint16_t* a16 = reinterpret_cast<const uint16_t*>(aux.row + gcol0);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            x[e] = (aux.row_ok && gcol0 + e < p.out_cols)
                       ? __uint_as_float(static_cast<uint32_t>(a16[e]) << 16)
                       : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = fmaf(p.c1, __uint_as_float(v[e]), p.c0 * x[e]);
        // a on the diagonal: only the chunk holding column `grow` has it.
        const int dg = grow - gcol0;
        if (dg >= 0 && dg < 32) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e == dg) f[e] = fmaf(p.c1, __uint_as_float(v[e]), fmaf(p.c0, x[e], p.c2));
        }
      }
      // Reuse a staging buffer only after the store issued from it two
      // stores ago has finished reading shared memory.
      uint8_t* buf = stage + (issued & 1) * 2048;
      if (issued >= 2) {
        if (lane == 0) ptx::bulk_wait_read<1>();
        __syncwarp();
      }
      // The output map uses the 64-byte swizzle: the 16-byte chunk q of row
      // `lane` sits at chunk q ^ ((lane >> 1) & 3) of the row's 64 bytes, so
      // the eight rows a quarter-warp writes fall in distinct banks.
      uint8_t* drow = buf + lane * 64;
      const int sw = (lane >> 1) & 3;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16(f[q * 8 + 0], f[q * 8 + 1]);
        u.y = pack_bf16(f[q * 8 + 2], f[q * 8 + 3]);
        u.z = pack_bf16(f[q * 8 + 4], f[q * 8 + 5]);
        u.w = pack_bf16(f[q * 8 + 6], f[q * 8 + 7]);
        *reinterpret_cast<uint4*>(drow + ((q ^ sw) << 4)) = u;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_3d(tmap_out, buf, gcol0, row0, mat);
        ptx::bulk_commit();
      }
      ++issued;
    }
    aux.load(cb + kPre);
  }
  __syncwarp();
}

}  // namespace nsk
}  // namespace muon
