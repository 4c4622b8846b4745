// k_shard.cu -- the shard-side kernels of the resharded Muon step.
//
// "Frontier Pre-training at Microsoft AI", Method details §5, resharding
// pipeline: under ZeRO data parallelism each rank holds a flat shard of
// every group's FP32 momentum, gradient and weights.
//  * shard_cast: step 1 on the shard -- M <- mu M + G in place, the BF16
//    cast, and per matrix the sum of squares of the shard's piece of it
//    (the matrix's owner adds the pieces for the Frobenius norm).  Reads
//    M, G; writes M, X: 14 B per element, as the one-GPU cast.
//  * shard_apply: step 5 on the shard -- W <- W (1 - lr wd) - lr s O with
//    O the BF16 update of the shard's elements (same arithmetic as the
//    one-GPU apply).  Reads W, O; writes W: 10 B per element.
//  * transpose_bf16: the owner turns tall matrices wide before the
//    Newton-Schulz products and their updates back afterwards.
// A shard is the element range [begin, end) of a group's flat buffer;
// matrix k of the group is [k E, (k + 1) E), so the shard's piece of
// matrix k is the intersection of the two ranges.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "launch.cuh"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;   // transpose tile (32 x 32), 32 x 8 threads

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t u) {
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// grid = (blocks per piece, pieces); block y covers the shard's piece of
// matrix k0 + y and writes its FP32 sum of squares to partials[y][x].
__global__ void __launch_bounds__(kThreads) shard_cast_kernel(
    int64_t begin, int64_t end, int64_t E, int64_t k0, float* __restrict__ M,
    const float* __restrict__ G, float mu, uint16_t* __restrict__ X,
    float* __restrict__ partials) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float red[kThreads / 32];
  const int64_t k = k0 + blockIdx.y;
  const int64_t lo = max(begin, k * E) - begin;
  const int64_t hi = min(end, (k + 1) * E) - begin;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  float ss = 0.f;
  for (int64_t i = lo + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < hi;
       i += stride) {
    const float v = fmaf(mu, M[i], __ldg(G + i));
    M[i] = v;
    X[i] = bf16_bits(v);
    ss = fmaf(v, v, ss);
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];   // fixed order
    partials[static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x] = s;
  }
}

// One block per piece: FP64 sum of its block partials in a fixed order.
__global__ void __launch_bounds__(kThreads) piece_sum_kernel(const float* __restrict__ partials,
                                                             int per, float* __restrict__ out) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ double red[kThreads / 32];
  const float* p = partials + static_cast<int64_t>(blockIdx.x) * per;
  double acc = 0.0;
  for (int i = threadIdx.x; i < per; i += kThreads) acc += static_cast<double>(p[i]);
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    out[blockIdx.x] = static_cast<float>(s);
  }
}

__global__ void __launch_bounds__(kThreads) shard_apply_kernel(int64_t n, float* __restrict__ W,
                                                               const uint16_t* __restrict__ O,
                                                               float lr, float wd, float scale) {
  grid_dep_wait();
  grid_dep_launch();
  const float decay = fmaf(-lr, wd, 1.0f);
  const float step = lr * scale;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    W[i] = fmaf(W[i], decay, -step * bf16_to_f32(__ldg(O + i)));
}

// grid = (tiles of the source matrix, matrices); dst[k][c][r] = src[k][r][c].
__global__ void __launch_bounds__(kTile * 8) transpose_bf16_kernel(int rows, int cols,
                                                                  const uint16_t* __restrict__ src,
                                                                  uint16_t* __restrict__ dst) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ uint16_t tile[kTile][kTile + 2];
  const int tiles_c = (cols + kTile - 1) / kTile;
  const int tr = blockIdx.x / tiles_c, tc = blockIdx.x % tiles_c;
  const int64_t base = static_cast<int64_t>(blockIdx.y) * rows * cols;
  const uint16_t* s = src + base;
  uint16_t* d = dst + base;
  const int c = tc * kTile + threadIdx.x;
  for (int j = threadIdx.y; j < kTile; j += 8) {
    const int r = tr * kTile + j;
    if (r < rows && c < cols) tile[j][threadIdx.x] = s[static_cast<int64_t>(r) * cols + c];
  }
  __syncthreads();
  const int r = tr * kTile + threadIdx.x;   // source row = destination column
  for (int j = threadIdx.y; j < kTile; j += 8) {
    const int cc = tc * kTile + j;           // source column = destination row
    if (r < rows && cc < cols) d[static_cast<int64_t>(cc) * rows + r] = tile[threadIdx.x][j];
  }
}

}  // namespace

int shard_cast_blocks(int64_t piece_elems) {
  int64_t b = (piece_elems + int64_t(kThreads) * 16 - 1) / (int64_t(kThreads) * 16);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(b, 128)));
}

cudaError_t launch_shard_cast(int64_t begin, int64_t end, int64_t E, float* M, const float* G,
                              float mu, uint16_t* X, float* partials, int blocks, float* sums,
                              cudaStream_t stream) {
  if (end <= begin) return cudaSuccess;
  const int64_t k0 = begin / E, k1 = (end - 1) / E;
  const int64_t pieces = k1 - k0 + 1;
  for (int64_t done = 0; done < pieces; done += kMaxGridY) {
    const int64_t take = std::min<int64_t>(pieces - done, kMaxGridY);
    cudaError_t e = launch_pdl(shard_cast_kernel, dim3(blocks, static_cast<unsigned>(take)),
                               dim3(kThreads), 0, stream, begin, end, E, k0 + done, M, G, mu, X,
                               partials + done * blocks);
    if (e != cudaSuccess) return e;
  }
  for (int64_t done = 0; done < pieces; done += 0x7fffffff) {
    const int64_t take = std::min<int64_t>(pieces - done, 0x7fffffff);
    cudaError_t e = launch_pdl(piece_sum_kernel, dim3(static_cast<unsigned>(take)), dim3(kThreads),
                               0, stream, partials + done * blocks, blocks, sums + done);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_shard_apply(int64_t n, float* W, const uint16_t* O, float lr, float wd,
                               float scale, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t grid = std::min<int64_t>((n + kThreads - 1) / kThreads, 152 * 16);
  return launch_pdl(shard_apply_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0,
                    stream, n, W, O, lr, wd, scale);
}

cudaError_t launch_transpose_bf16(int rows, int cols, int count, const uint16_t* src,
                                  uint16_t* dst, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  const int64_t tiles = int64_t((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
  const int64_t per = int64_t(rows) * cols;
  for (int64_t done = 0; done < count; done += kMaxGridY) {
    const int take = static_cast<int>(std::min<int64_t>(count - done, kMaxGridY));
    cudaError_t e = launch_pdl(transpose_bf16_kernel,
                               dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(take)),
                               dim3(kTile, 8), 0, stream, rows, cols, src + done * per,
                               dst + done * per);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace muon
