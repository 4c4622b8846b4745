// k_elementwise.cu -- the HBM-bound steps of the Muon step on sm_103a.
//
//  * momentum_cast: "update the FP32 momentum shard in place, then cast it
//    to BF16" (Frontier Pre-training at Microsoft AI, Method details §5,
//    resharding step 1), fused with the transpose of tall matrices to the
//    wide orientation and with per-tile partial sums of M^2 for the
//    Frobenius pre-normalisation.  Traffic: read M, G; write M, X.
//  * norm_finalize: deterministic per-matrix reduction of the partials.
//  * apply_update: "cast the update back to FP32 and apply it to the
//    weights" (same section, resharding step 5) with decoupled weight decay.
//    Traffic: read W, O; write W.  The contiguous wide case streams both
//    arrays flat; tall matrices (O transposed back through shared memory)
//    run on a resident grid with the next tile's O prefetched; unaligned
//    update pitches fall back to one 64 x 64 tile per block.
//  * scale_bf16: the degenerate zero-iteration case O = X / s.
//
// Except the flat apply, they work on 64 x 64 tiles of the source matrix
// with 256 threads; rows are read as float4 when the pitch allows it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "launch.cuh"

namespace muon {
namespace {

constexpr int T = kEwTile;   // 64
constexpr int kThreads = 256;
constexpr int kPad = 8;      // shared-memory row padding (bf16 elements)
constexpr int64_t kMaxGrid = 0x7fffffff;   // gridDim.x limit

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t u) {
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

template <typename Tv>
__device__ __forceinline__ Tv block_sum(Tv v, Tv* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  Tv s = 0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];  // fixed order
  }
  return s;  // valid in thread 0
}

// grid = (tiles per matrix, count); tile = 64 source rows x 64 source cols.
// With kNesterov the matrix cast (and normed) is U = G + mu * M' instead
// of the updated momentum M' itself.
template <bool kTranspose, bool kNesterov>
__global__ void __launch_bounds__(kThreads) momentum_cast_kernel(
    int rows, int cols, float* __restrict__ M, const float* __restrict__ G, float mu,
    uint16_t* __restrict__ X, int64_t x_ld, int64_t x_ms, float* __restrict__ partials) {
  grid_dep_wait();    // inputs come from the previous kernel of the step
  grid_dep_launch();
  __shared__ __align__(16) uint16_t sT[kTranspose ? T : 1][T + kPad];
  __shared__ float red[kThreads / 32];

  const int tiles_c = (cols + T - 1) / T;
  const int tr = blockIdx.x / tiles_c, tc = blockIdx.x % tiles_c;
  const int64_t mat = blockIdx.y;
  const int64_t base = mat * static_cast<int64_t>(rows) * cols;
  float* Mm = M + base;
  const float* Gm = G + base;
  uint16_t* Xm = X + mat * x_ms;

  const int rr = threadIdx.x >> 4;        // 0..15
  const int cc = (threadIdx.x & 15) * 4;  // 0..60
  const bool vec_ok = (cols & 3) == 0;
  float ss = 0.f;

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int lr_ = rr + 16 * i;
    const int r = tr * T + lr_;
    const int c = tc * T + cc;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < rows) {
      const int64_t off = static_cast<int64_t>(r) * cols + c;
      if (vec_ok && c + 3 < cols) {
        float4 m4 = *reinterpret_cast<const float4*>(Mm + off);
        const float4 g4 = __ldg(reinterpret_cast<const float4*>(Gm + off));
        m4.x = fmaf(mu, m4.x, g4.x);
        m4.y = fmaf(mu, m4.y, g4.y);
        m4.z = fmaf(mu, m4.z, g4.z);
        m4.w = fmaf(mu, m4.w, g4.w);
        *reinterpret_cast<float4*>(Mm + off) = m4;
        if constexpr (kNesterov) {
          v[0] = fmaf(mu, m4.x, g4.x); v[1] = fmaf(mu, m4.y, g4.y);
          v[2] = fmaf(mu, m4.z, g4.z); v[3] = fmaf(mu, m4.w, g4.w);
        } else {
          v[0] = m4.x; v[1] = m4.y; v[2] = m4.z; v[3] = m4.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (c + e < cols) {
            const float gv = Gm[off + e];
            const float mv = fmaf(mu, Mm[off + e], gv);
            Mm[off + e] = mv;
            v[e] = kNesterov ? fmaf(mu, mv, gv) : mv;
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) ss = fmaf(v[e], v[e], ss);
    if constexpr (kTranspose) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sT[cc + e][lr_] = bf16_bits(v[e]);
    } else if (r < rows) {
      uint16_t* xr = Xm + static_cast<int64_t>(r) * x_ld + c;
      if (c + 3 < cols && ((x_ld & 3) == 0)) {
        uint2 p;
        p.x = static_cast<uint32_t>(bf16_bits(v[0])) | (static_cast<uint32_t>(bf16_bits(v[1])) << 16);
        p.y = static_cast<uint32_t>(bf16_bits(v[2])) | (static_cast<uint32_t>(bf16_bits(v[3])) << 16);
        *reinterpret_cast<uint2*>(xr) = p;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + e < cols) xr[e] = bf16_bits(v[e]);
      }
    }
  }

  if constexpr (kTranspose) {
    __syncthreads();
    // X (wide) row = source column, X column = source row.
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = threadIdx.x + kThreads * j;  // 0..511
      const int xrow_l = idx >> 3;                 // source column within tile
      const int seg = (idx & 7) * 8;               // source rows seg..seg+7
      const int xrow = tc * T + xrow_l;
      const int xcol = tr * T + seg;
      if (xrow < cols) {
        uint16_t* dst = Xm + static_cast<int64_t>(xrow) * x_ld + xcol;
        if (xcol + 7 < rows && ((x_ld & 7) == 0)) {
          *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&sT[xrow_l][seg]);
        } else {
          for (int e = 0; e < 8; ++e)
            if (xcol + e < rows) dst[e] = sT[xrow_l][seg + e];
        }
      }
    }
  }

  const float tot = block_sum(ss, red);
  if (threadIdx.x == 0) partials[mat * gridDim.x + blockIdx.x] = tot;
}

// 1/(||U||_F + eps) per matrix, from the cast kernel's partials, summed in
// FP64 in a fixed order (deterministic).  Range: the cast kernel's FP32
// partial sums of squares overflow once entries pass ~1.8e19; such a
// matrix (partials +inf, not NaN) has its norm recomputed here in FP64 from
// its BF16 copy (within 2^-9 of the FP32 norm).  And the Gram product
// accumulates X X^T in FP32 before it applies 1/s^2, so a norm above 2^60
// would overflow its accumulator: such a matrix's BF16 copy is scaled by a
// power of two 2^e (s * 2^e in [1, 2); exact for every entry that stays
// normal) and 1/s by 2^-e, so X * inv_norm -- all the products use -- is
// unchanged.  (Underflowing squares only occur for norms far below eps.)
constexpr double kNormScaleLimit = 1152921504606846976.0;   // 2^60

__global__ void __launch_bounds__(kThreads) norm_finalize_kernel(
    const float* __restrict__ partials, int per_matrix, float eps, float* __restrict__ inv_norm,
    int* __restrict__ err, uint16_t* __restrict__ X, int64_t x_ld, int64_t x_ms, int m, int n) {
  grid_dep_wait();    // inputs come from the previous kernel of the step
  grid_dep_launch();
  __shared__ double red[kThreads / 32];
  __shared__ int recompute, scale_exp;
  const int64_t mat = blockIdx.x;
  const float* p = partials + mat * per_matrix;
  uint16_t* Xm = X != nullptr ? X + mat * x_ms : nullptr;
  const int64_t total = static_cast<int64_t>(m) * n;
  double acc = 0.0;
  for (int i = threadIdx.x; i < per_matrix; i += kThreads) acc += static_cast<double>(p[i]);
  double tot = block_sum(acc, red);   // valid in thread 0
  if (threadIdx.x == 0) recompute = (isinf(tot) && Xm != nullptr) ? 1 : 0;
  __syncthreads();
  if (recompute) {
    double a2 = 0.0;
    for (int64_t i = threadIdx.x; i < total; i += kThreads) {
      const double v = bf16_to_f32(Xm[(i / n) * x_ld + i % n]);
      a2 = fma(v, v, a2);
    }
    tot = block_sum(a2, red);
  }
  if (threadIdx.x == 0) {
    int e = 0;
    if (!isfinite(tot)) {
      atomicOr(err, kDevErrNonFinite);
      inv_norm[mat] = 0.f;
    } else {
      const double s = sqrt(tot);
      if (s > kNormScaleLimit && Xm != nullptr) e = -ilogb(s);
      inv_norm[mat] = static_cast<float>(1.0 / ((s + static_cast<double>(eps)) * ldexp(1.0, e)));
    }
    scale_exp = e;
  }
  __syncthreads();
  const int e = scale_exp;
  if (e != 0) {
    // Two normal factors (2^e alone may be below the FP32 normal range).
    const float f1 = ldexpf(1.0f, e / 2), f2 = ldexpf(1.0f, e - e / 2);
    for (int64_t i = threadIdx.x; i < total; i += kThreads) {
      uint16_t* q = Xm + (i / n) * x_ld + i % n;
      *q = bf16_bits(bf16_to_f32(*q) * f1 * f2);
    }
  }
}

// grid = (tiles per matrix of the weight, count); tile = 64 x 64 of W.
template <bool kTranspose>
__global__ void __launch_bounds__(kThreads) apply_update_kernel(
    int rows, int cols, float* __restrict__ W, const uint16_t* __restrict__ O, int64_t o_ld,
    int64_t o_ms, float lr, float wd, float scale) {
  grid_dep_wait();    // inputs come from the previous kernel of the step
  grid_dep_launch();
  __shared__ __align__(16) uint16_t sO[kTranspose ? T : 1][T + kPad];
  const int tiles_c = (cols + T - 1) / T;
  const int tr = blockIdx.x / tiles_c, tc = blockIdx.x % tiles_c;
  const int64_t mat = blockIdx.y;
  float* Wm = W + mat * static_cast<int64_t>(rows) * cols;
  const uint16_t* Om = O + mat * o_ms;
  const float decay = fmaf(-lr, wd, 1.0f);
  const float step = lr * scale;

  if constexpr (kTranspose) {
    // O (wide) is cols x rows: stage O rows tc*64.. (= W columns) into smem.
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = threadIdx.x + kThreads * j;
      const int orow_l = idx >> 3;
      const int seg = (idx & 7) * 8;
      const int orow = tc * T + orow_l;
      const int ocol = tr * T + seg;
      if (orow < cols) {
        const uint16_t* src = Om + static_cast<int64_t>(orow) * o_ld + ocol;
        if (ocol + 7 < rows && ((o_ld & 7) == 0)) {
          *reinterpret_cast<uint4*>(&sO[orow_l][seg]) = __ldg(reinterpret_cast<const uint4*>(src));
        } else {
          for (int e = 0; e < 8; ++e) sO[orow_l][seg + e] = (ocol + e < rows) ? src[e] : 0;
        }
      }
    }
    __syncthreads();
  }

  const int rr = threadIdx.x >> 4;
  const int cc = (threadIdx.x & 15) * 4;
  const bool vec_ok = (cols & 3) == 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int lr_ = rr + 16 * i;
    const int r = tr * T + lr_;
    const int c = tc * T + cc;
    if (r >= rows) continue;
    float o[4];
    if constexpr (kTranspose) {
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = bf16_to_f32(sO[cc + e][lr_]);
    } else {
      const uint16_t* src = Om + static_cast<int64_t>(r) * o_ld + c;
      if (c + 3 < cols && ((o_ld & 3) == 0)) {
        const uint2 p = __ldg(reinterpret_cast<const uint2*>(src));
        o[0] = bf16_to_f32(p.x & 0xFFFFu); o[1] = bf16_to_f32(p.x >> 16);
        o[2] = bf16_to_f32(p.y & 0xFFFFu); o[3] = bf16_to_f32(p.y >> 16);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = (c + e < cols) ? bf16_to_f32(src[e]) : 0.f;
      }
    }
    const int64_t off = static_cast<int64_t>(r) * cols + c;
    if (vec_ok && c + 3 < cols) {
      float4 w4 = *reinterpret_cast<const float4*>(Wm + off);
      w4.x = fmaf(w4.x, decay, -step * o[0]);
      w4.y = fmaf(w4.y, decay, -step * o[1]);
      w4.z = fmaf(w4.z, decay, -step * o[2]);
      w4.w = fmaf(w4.w, decay, -step * o[3]);
      *reinterpret_cast<float4*>(Wm + off) = w4;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (c + e < cols) Wm[off + e] = fmaf(Wm[off + e], decay, -step * o[e]);
    }
  }
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_prior() {   // all groups but the newest
  asm volatile("cp.async.wait_group 1;\n" ::: "memory");
}

// Apply for a tall batch (rows > cols; O stored wide, cols x rows), on
// tiles of 128 W rows x 64 W columns.  A block copies its tile's O block
// (64 O rows x 256 bytes) into shared memory with cp.async (16 bytes per
// copy, no register staging) and loads its W rows while that copy is in
// flight.  The launch gives every tile its own block (measured 6.95 TB/s
// on 64 x 4096x1536, against 6.32 for a grid of resident blocks walking
// the tiles); a grid capped by the launch limit walks the remaining tiles
// with the next tile's O block prefetched into the other half of a double
// buffer.  The 16-byte chunk q of buffer row j sits at chunk
// q ^ ((j >> 2) & 7): the update reads one O element of each of 16 rows
// j = 4k + e at a time; with 256-byte rows those would all fall in one
// bank, with the swizzle they spread over eight (two-way at most).
// Needs cols % 4 == 0, W 16-byte aligned, O pitches multiples of 8
// elements and O 16-byte aligned.
constexpr int kTallR = 128;   // W rows per tile (= O columns)

__device__ __forceinline__ int tall_chunk(int j, int q) { return q ^ ((j >> 2) & 7); }

__global__ void __launch_bounds__(kThreads) apply_update_tall_kernel(
    int rows, int cols, int count, float* __restrict__ W, const uint16_t* __restrict__ O,
    int64_t o_ld, int64_t o_ms, float lr, float wd, float scale) {
  grid_dep_wait();    // inputs come from the previous kernel of the step
  grid_dep_launch();
  __shared__ __align__(16) uint16_t sO[2][T][kTallR];
  const int tiles_c = (cols + T - 1) / T;
  const int per_matrix = ((rows + kTallR - 1) / kTallR) * tiles_c;
  const int64_t total = static_cast<int64_t>(per_matrix) * count;
  const float decay = fmaf(-lr, wd, 1.0f);
  const float step = lr * scale;

  // O block of tile t: O rows tc*64.. (W columns), O columns tr*128.. (W rows).
  auto stage = [&](int64_t t, int buf) {
    const int64_t mat = t / per_matrix;
    const int l = static_cast<int>(t - mat * per_matrix);
    const int tr = l / tiles_c, tc = l - (l / tiles_c) * tiles_c;
    const uint16_t* Om = O + mat * o_ms;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int idx = threadIdx.x + kThreads * j;   // 0..1023
      const int orow_l = idx >> 4;                  // 0..63
      const int q = idx & 15;                       // 16-byte chunk of the row
      const int orow = tc * T + orow_l;
      const int ocol = tr * kTallR + q * 8;
      if (orow >= cols) continue;
      uint16_t* dst = &sO[buf][orow_l][tall_chunk(orow_l, q) * 8];
      const uint16_t* src = Om + static_cast<int64_t>(orow) * o_ld + ocol;
      if (ocol + 7 < rows) {
        cp_async16(dst, src);
      } else {
        for (int e = 0; e < 8; ++e) dst[e] = (ocol + e < rows) ? src[e] : 0;
      }
    }
  };

  const int rr = threadIdx.x >> 4;        // 0..15
  const int cc = (threadIdx.x & 15) * 4;  // 0..60
  int buf = 0;
  int64_t t = blockIdx.x;
  if (t < total) stage(t, 0);
  cp_async_commit();
  for (; t < total; t += gridDim.x) {
    const int64_t tn = t + gridDim.x;
    if (tn < total) stage(tn, buf ^ 1);
    cp_async_commit();
    const int64_t mat = t / per_matrix;
    const int l = static_cast<int>(t - mat * per_matrix);
    const int tr = l / tiles_c, tc = l - (l / tiles_c) * tiles_c;
    float* Wm = W + mat * static_cast<int64_t>(rows) * cols;
    const int c = tc * T + cc;
    float4 w[kTallR / 16];
#pragma unroll
    for (int i = 0; i < kTallR / 16; ++i) {
      const int r = tr * kTallR + rr + 16 * i;
      if (r < rows && c < cols)
        w[i] = *reinterpret_cast<const float4*>(Wm + static_cast<int64_t>(r) * cols + c);
    }
    cp_async_wait_prior();   // this tile's O block has landed (the next may still fly)
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTallR / 16; ++i) {
      const int lr_ = rr + 16 * i;   // O column within the block
      const int r = tr * kTallR + lr_;
      if (r < rows && c < cols) {
        const int q = lr_ >> 3, e8 = lr_ & 7;
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[e] = bf16_to_f32(sO[buf][cc + e][tall_chunk(cc + e, q) * 8 + e8]);
        float4 v = w[i];
        v.x = fmaf(v.x, decay, -step * o[0]);
        v.y = fmaf(v.y, decay, -step * o[1]);
        v.z = fmaf(v.z, decay, -step * o[2]);
        v.w = fmaf(v.w, decay, -step * o[3]);
        *reinterpret_cast<float4*>(Wm + static_cast<int64_t>(r) * cols + c) = v;
      }
    }
    __syncthreads();   // sO[buf] is refilled by the iteration after next
    buf ^= 1;
  }
}

// Apply for a wide (or square) batch whose update has the weights' own
// pitch: W and O are then flat arrays of the same length, streamed in
// 4-element groups (float4 of W, 8 bytes of O).  The launch gives every
// group its own thread (7.23 TB/s on 96 x 2048^2, against 6.50 for a
// grid-stride loop over 8 blocks per SM); the loop only covers batches
// beyond the launch limit.
__global__ void __launch_bounds__(kThreads) apply_update_flat_kernel(
    int64_t n4, float4* __restrict__ W4, const uint2* __restrict__ O2, float lr, float wd,
    float scale) {
  grid_dep_wait();    // inputs come from the previous kernel of the step
  grid_dep_launch();
  const float decay = fmaf(-lr, wd, 1.0f);
  const float step = lr * scale;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n4;
       i += stride) {
    float4 w = W4[i];
    const uint2 o = __ldg(O2 + i);
    w.x = fmaf(w.x, decay, -step * bf16_to_f32(o.x & 0xFFFFu));
    w.y = fmaf(w.y, decay, -step * bf16_to_f32(o.x >> 16));
    w.z = fmaf(w.z, decay, -step * bf16_to_f32(o.y & 0xFFFFu));
    w.w = fmaf(w.w, decay, -step * bf16_to_f32(o.y >> 16));
    W4[i] = w;
  }
}

__global__ void __launch_bounds__(kThreads) scale_bf16_kernel(
    int m, int n, const uint16_t* __restrict__ x, int64_t x_ld, int64_t x_ms,
    uint16_t* __restrict__ out, int64_t o_ld, int64_t o_ms, const float* __restrict__ inv_norm) {
  grid_dep_wait();    // inputs come from the previous kernel of the step
  grid_dep_launch();
  const int64_t mat = blockIdx.y;
  const float s = inv_norm[mat];
  const int64_t total = static_cast<int64_t>(m) * n;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t r = i / n, c = i % n;
    const float v = bf16_to_f32(x[mat * x_ms + r * x_ld + c]) * s;
    out[mat * o_ms + r * o_ld + c] = bf16_bits(v);
  }
}

}  // namespace

cudaError_t launch_momentum_cast(int rows, int cols, int count, float* M, const float* G,
                                 float mu, uint16_t* X, int64_t x_ld, int64_t x_ms,
                                 float* partials, cudaStream_t stream, bool nesterov) {
  if (count <= 0) return cudaSuccess;
  const dim3 grid(ew_tiles_per_matrix(rows, cols), count);
  const dim3 block(kThreads);
  const bool tr = rows > cols;
  auto kern = tr ? (nesterov ? momentum_cast_kernel<true, true> : momentum_cast_kernel<true, false>)
                 : (nesterov ? momentum_cast_kernel<false, true> : momentum_cast_kernel<false, false>);
  return launch_pdl(kern, grid, block, 0, stream, rows, cols, M, G, mu, X, x_ld, x_ms, partials);
}

cudaError_t launch_norm_finalize(const float* partials, int per_matrix, int count, float eps,
                                 float* inv_norm, int* err, uint16_t* x, int64_t x_ld,
                                 int64_t x_ms, int m, int n, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  return launch_pdl(norm_finalize_kernel, dim3(count), dim3(kThreads), 0, stream, partials,
                    per_matrix, eps, inv_norm, err, x, x_ld, x_ms, m, n);
}

cudaError_t launch_apply_update(int rows, int cols, int count, float* W, const uint16_t* O,
                                int64_t o_ld, int64_t o_ms, float lr, float wd, float scale,
                                cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  if (rows <= cols && o_ld == cols && o_ms == int64_t(rows) * cols && (cols & 3) == 0 &&
      (reinterpret_cast<uintptr_t>(W) & 15) == 0 && (reinterpret_cast<uintptr_t>(O) & 7) == 0) {
    const int64_t n4 = int64_t(count) * rows * cols / 4;
    const int64_t grid = std::min<int64_t>((n4 + kThreads - 1) / kThreads, kMaxGrid);
    return launch_pdl(apply_update_flat_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads),
                      0, stream, n4, reinterpret_cast<float4*>(W),
                      reinterpret_cast<const uint2*>(O), lr, wd, scale);
  }
  if (rows > cols && (cols & 3) == 0 && (o_ld & 7) == 0 && (o_ms & 7) == 0 &&
      (reinterpret_cast<uintptr_t>(W) & 15) == 0 && (reinterpret_cast<uintptr_t>(O) & 15) == 0) {
    const int64_t tiles =
        int64_t((rows + kTallR - 1) / kTallR) * ((cols + T - 1) / T) * count;
    const int64_t grid = std::min<int64_t>(tiles, kMaxGrid);
    return launch_pdl(apply_update_tall_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads),
                      0, stream, rows, cols, count, W, O, o_ld, o_ms, lr, wd, scale);
  }
  const dim3 grid(ew_tiles_per_matrix(rows, cols), count);
  auto kern = rows > cols ? apply_update_kernel<true> : apply_update_kernel<false>;
  return launch_pdl(kern, grid, dim3(kThreads), 0, stream, rows, cols, W, O, o_ld, o_ms, lr, wd,
                    scale);
}

cudaError_t launch_scale_bf16(int m, int n, int count, const uint16_t* x, int64_t x_ld,
                              int64_t x_ms, uint16_t* out, int64_t o_ld, int64_t o_ms,
                              const float* inv_norm, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  const int64_t total = static_cast<int64_t>(m) * n;
  int64_t blocks = (total + kThreads - 1) / kThreads;
  if (blocks > 4096) blocks = 4096;
  const dim3 grid(static_cast<unsigned>(blocks), count);
  return launch_pdl(scale_bf16_kernel, grid, dim3(kThreads), 0, stream, m, n, x, x_ld, x_ms, out,
                    o_ld, o_ms, inv_norm);
}

}  // namespace muon
