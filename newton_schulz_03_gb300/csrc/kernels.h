// kernels.h -- internal launch interface between the host library
// (muon_api.cpp) and the CUDA translation units.  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace muon {

// Device error bits written by kernels into the handle's flag word.
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrNonFinite = 2;

// Limits shared by every entry point: the longest matrix side, the
// iteration count, and the largest grid.y of the elementwise kernels (one
// grid row per matrix).
constexpr int kMaxDim = 1 << 20;
constexpr int kMaxSteps = 64;
constexpr int64_t kMaxGridY = 65535;

// Largest matrix count one Newton-Schulz launch sequence may cover: tile
// indices stay in int32 (the update product has the most tiles,
// ceil(m/128) * ceil(n/256); the Gram product t(t+1)/2 with t = ceil(m/128))
// and the scale kernel of ns_steps == 0 keeps grid.y within its limit.
inline int64_t ns_max_count_per_launch(int m, int n) {
  const int64_t tm = (m + 127) / 128, tn = (n + 255) / 256;
  const int64_t per = (tm * tn > tm * (tm + 1) / 2) ? tm * tn : tm * (tm + 1) / 2;
  int64_t cap = (int64_t(1) << 30) / per;
  if (cap > kMaxGridY) cap = kMaxGridY;
  return cap < 1 ? 1 : cap;
}

// Elementwise kernels work on 64 x 64 tiles of the source matrix.
constexpr int kEwTile = 64;

inline int ew_tiles_per_matrix(int rows, int cols) {
  return ((rows + kEwTile - 1) / kEwTile) * ((cols + kEwTile - 1) / kEwTile);
}

// Step 1: M <- mu*M + G (FP32, in place); U = M (or G + mu*M with
// `nesterov`); X <- bf16_rne(U) in wide layout (transposed when
// rows > cols) with row pitch x_ld and matrix pitch x_ms (elements);
// partials[mat * tiles + tile] <- sum of U^2 over the tile.
cudaError_t launch_momentum_cast(int rows, int cols, int count, float* M, const float* G,
                                 float mu, uint16_t* X, int64_t x_ld, int64_t x_ms,
                                 float* partials, cudaStream_t stream, bool nesterov = false);

// inv_norm[mat] <- 1 / (sqrt(sum of partials of mat) + eps); flags NaN/Inf.
// A matrix whose norm exceeds 2^60 has its BF16 copy x (m x n, pitches in
// elements) scaled by 2^e and inv_norm by 2^-e (see the kernel).
cudaError_t launch_norm_finalize(const float* partials, int per_matrix, int count, float eps,
                                 float* inv_norm, int* err, uint16_t* x, int64_t x_ld,
                                 int64_t x_ms, int m, int n, cudaStream_t stream);

// Step 5: W <- W (1 - lr wd) - lr scale O, O in wide layout (pitches in
// elements), transposed back when rows > cols.
cudaError_t launch_apply_update(int rows, int cols, int count, float* W, const uint16_t* O,
                                int64_t o_ld, int64_t o_ms, float lr, float wd, float scale,
                                cudaStream_t stream);

// ns_steps == 0: out <- bf16(inv_norm[mat] * x), both m x n with pitches.
cudaError_t launch_scale_bf16(int m, int n, int count, const uint16_t* x, int64_t x_ld,
                              int64_t x_ms, uint16_t* out, int64_t o_ld, int64_t o_ms,
                              const float* inv_norm, cudaStream_t stream);

// ------------------------------------------------------------------ shards
// Resharded step, on a rank's flat shard [begin, end) of a group whose
// matrices have E elements: M <- mu M + G (in place), X <- bf16(M) (flat,
// the shard's layout), and sums[y] = sum of M^2 over the shard's piece of
// matrix begin/E + y (two-level: FP32 per block into `partials`, `blocks`
// per piece, then FP64 per piece).
int shard_cast_blocks(int64_t piece_elems);
cudaError_t launch_shard_cast(int64_t begin, int64_t end, int64_t E, float* M, const float* G,
                              float mu, uint16_t* X, float* partials, int blocks, float* sums,
                              cudaStream_t stream);
// W <- W (1 - lr wd) - lr scale O over n flat elements (O BF16).
cudaError_t launch_shard_apply(int64_t n, float* W, const uint16_t* O, float lr, float wd,
                               float scale, cudaStream_t stream);
// dst[k] = src[k]^T for `count` BF16 matrices of rows x cols (contiguous).
cudaError_t launch_transpose_bf16(int rows, int cols, int count, const uint16_t* src,
                                  uint16_t* dst, cudaStream_t stream);

// ------------------------------------------------------------------ NS GEMMs
// A BF16 matrix batch: element pointer, row pitch and matrix pitch (elements).
struct BatchView {
  const void* ptr;
  int64_t ld;
  int64_t ms;
};

// Set up kernel attributes once per process (dynamic shared memory).
cudaError_t ns_gemm_init();

// A = alpha * X X^T, alpha = inv_norm[mat]^2 (or 1 when inv_norm == NULL).
// X: m x n, A: m x m.  m > 128: only the 256-blocks on and above the block
// diagonal are computed and stored; m <= 128: one tile, stored in full.
cudaError_t ns_launch_gram(int m, int n, int count, BatchView X, BatchView A_out,
                           const float* inv_norm, int* err, int grid_cap, cudaStream_t stream);

// B' = a I + b A + c A A (A symmetric m x m): the quintic polynomial with
// the linear term folded in.  Stored like A.
cudaError_t ns_launch_poly(int m, int count, BatchView A, BatchView B_out, float a, float b,
                           float c, int* err, int grid_cap, cudaStream_t stream);

// X' = alpha B' X, alpha = inv_norm[mat] (or 1 when NULL).
cudaError_t ns_launch_update(int m, int n, int count, BatchView B, BatchView X,
                             BatchView X_out, const float* inv_norm, int* err, int grid_cap,
                             cudaStream_t stream);

// ------------------------------------------------------------------ AdamW
constexpr int kAdamwMaxTensors = 40;
// Tensors of one AdamW launch, passed by value in the kernel parameters.
struct AdamwTable {
  float* p[kAdamwMaxTensors];
  const float* g[kAdamwMaxTensors];
  float* m[kAdamwMaxTensors];
  float* v[kAdamwMaxTensors];
  int64_t n[kAdamwMaxTensors];
  int64_t block_start[kAdamwMaxTensors + 1];  // prefix sum of blocks per tensor
  int count;
};
int64_t adamw_blocks(int64_t numel);
cudaError_t launch_adamw(const AdamwTable& table, float lr, float beta1, float beta2, float eps,
                         float wd, int step, cudaStream_t stream);

// One kernel whose barrier wait can never complete: the bounded wait must
// expire after limit_ns and set kDevErrTimeout in *err.
cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t stream);

// Last error text of a tensor-map encode (host, thread-local).
const char* ns_last_encode_error();

// CTA-pair (cta_group::2) variants of the three products, 256 x 256 tiles;
// the tensor maps are built by the ns_launch_* functions above (`_t`
// maps: 64 x 64 boxes of the same tensor, for transposed block reads).
// A and B produced by the pair kernels hold only their upper 256-block
// triangle; the pair kernels read them accordingly.
}  // namespace muon
#include <cuda.h>
namespace muon {
cudaError_t ns_pair_init();
cudaError_t ns_pair_gram(const CUtensorMap& tx, const CUtensorMap& tout, int m, int n, int count,
                         BatchView A_out, const float* inv_norm, int* err, int grid_cap,
                         cudaStream_t stream);
cudaError_t ns_pair_poly(const CUtensorMap& ta, const CUtensorMap& ta_t, const CUtensorMap& tout,
                         int m, int count, BatchView A, BatchView B_out, float a, float b, float c,
                         int* err, int grid_cap, cudaStream_t stream, int mn4d);
cudaError_t ns_pair_update(const CUtensorMap& tb, const CUtensorMap& tb_t, const CUtensorMap& tx,
                           const CUtensorMap& tout, int m, int n, int count, BatchView X_out,
                           const float* inv_norm, int* err, int grid_cap, cudaStream_t stream,
                           int mn4d);

// Record `msg` as the calling thread's last error text and return `status`
// (read back through muon_last_error_message).
int report(int status, const char* msg);

}  // namespace muon
