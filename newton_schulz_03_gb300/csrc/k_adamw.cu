// k_adamw.cu -- AdamW for the parameters Muon does not handle (embeddings,
// norms, scalars): "Microsoft Reveals MAI-Base-2 Training Recipe", section
// "How to Make Parameter Updates Faster and More Stable?" (Muon for 2-D
// non-embedding matrices, AdamW for the rest).  Decoupled decay and bias
// correction, FP32 state:
//   p <- p (1 - lr wd)
//   m <- b1 m + (1 - b1) g            v <- b2 v + (1 - b2) g^2
//   p <- p - (lr / (1 - b1^t)) m / (sqrt(v) / sqrt(1 - b2^t) + eps)
// One launch covers up to kMaxTensors tensors, described in the kernel's
// parameter block (no device-side table to allocate).  HBM-bound: 28 bytes
// per element (read p, g, m, v; write p, m, v).
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;                      // two float4 per thread
constexpr int64_t kBlockElems = int64_t(kThreads) * kPerThread;

struct AdamwScalars {
  float lr, beta1, one_minus_beta1, beta2, one_minus_beta2, eps, decay, step_size, bc2_sqrt;
};

__device__ __forceinline__ void adamw_elem(float& p, float g, float& m, float& v,
                                           const AdamwScalars& s) {
  p *= s.decay;
  m = fmaf(s.beta1, m, s.one_minus_beta1 * g);
  v = fmaf(s.beta2, v, s.one_minus_beta2 * g * g);
  const float denom = sqrtf(v) / s.bc2_sqrt + s.eps;
  p -= s.step_size * (m / denom);
}

__global__ void __launch_bounds__(kThreads) adamw_kernel(const AdamwTable table,
                                                         const AdamwScalars s) {
  // Tensor of this block: last t with block_start[t] <= blockIdx.x.
  int t = 0;
  while (t + 1 < table.count && table.block_start[t + 1] <= blockIdx.x) ++t;
  const int64_t n = table.n[t];
  const int64_t base = (static_cast<int64_t>(blockIdx.x) - table.block_start[t]) * kBlockElems;
  float* __restrict__ P = table.p[t];
  const float* __restrict__ G = table.g[t];
  float* __restrict__ M = table.m[t];
  float* __restrict__ V = table.v[t];
  const bool vec = ((reinterpret_cast<uintptr_t>(P) | reinterpret_cast<uintptr_t>(G) |
                     reinterpret_cast<uintptr_t>(M) | reinterpret_cast<uintptr_t>(V)) & 15u) == 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t i = base + (static_cast<int64_t>(h) * kThreads + threadIdx.x) * 4;
    if (vec && i + 3 < n) {
      float4 p4 = *reinterpret_cast<const float4*>(P + i);
      const float4 g4 = __ldg(reinterpret_cast<const float4*>(G + i));
      float4 m4 = *reinterpret_cast<const float4*>(M + i);
      float4 v4 = *reinterpret_cast<const float4*>(V + i);
      adamw_elem(p4.x, g4.x, m4.x, v4.x, s);
      adamw_elem(p4.y, g4.y, m4.y, v4.y, s);
      adamw_elem(p4.z, g4.z, m4.z, v4.z, s);
      adamw_elem(p4.w, g4.w, m4.w, v4.w, s);
      *reinterpret_cast<float4*>(P + i) = p4;
      *reinterpret_cast<float4*>(M + i) = m4;
      *reinterpret_cast<float4*>(V + i) = v4;
    } else {
      for (int e = 0; e < 4; ++e) {
        if (i + e < n) {
          float p = P[i + e], m = M[i + e], v = V[i + e];
          adamw_elem(p, G[i + e], m, v, s);
          P[i + e] = p;
          M[i + e] = m;
          V[i + e] = v;
        }
      }
    }
  }
}

}  // namespace

int64_t adamw_blocks(int64_t numel) { return (numel + kBlockElems - 1) / kBlockElems; }

cudaError_t launch_adamw(const AdamwTable& table, float lr, float beta1, float beta2, float eps,
                         float wd, int step, cudaStream_t stream) {
  if (table.count <= 0 || table.block_start[table.count] <= 0) return cudaSuccess;
  AdamwScalars s;
  s.lr = lr;
  s.beta1 = beta1;
  s.one_minus_beta1 = 1.0f - beta1;
  s.beta2 = beta2;
  s.one_minus_beta2 = 1.0f - beta2;
  s.eps = eps;
  s.decay = 1.0f - lr * wd;
  // Bias corrections in double on the host, then FP32.
  double p1 = 1.0, p2 = 1.0;
  for (int i = 0; i < step; ++i) {
    p1 *= static_cast<double>(beta1);
    p2 *= static_cast<double>(beta2);
  }
  s.step_size = static_cast<float>(static_cast<double>(lr) / (1.0 - p1));
  s.bc2_sqrt = static_cast<float>(sqrt(1.0 - p2));
  const unsigned grid = static_cast<unsigned>(table.block_start[table.count]);
  adamw_kernel<<<grid, kThreads, 0, stream>>>(table, s);
  return cudaGetLastError();
}

}  // namespace muon
