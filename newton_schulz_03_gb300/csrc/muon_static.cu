// muon_static.cu -- Newton-Schulz entry point that allocates no memory.
//
// Some callers cannot call cudaMalloc at all: code that runs while a CUDA
// graph is being built around it, allocators and runtimes that must not
// re-enter themselves, and deployments that forbid device allocations
// after start-up (fixed memory budgets, pre-planned arenas).  For them the
// library keeps one file-scope scratch array in device memory, loaded with
// the library: every GPU that loads the library holds kStaticScratchBytes
// of it until the process exits.
//
// The entry point below runs the same batched Newton-Schulz kernels as
// muon_newton_schulz_bf16, with the Gram matrix A, the square B and the
// second iterate buffer placed in that array instead of a handle's
// workspace.  It calls no cudaMalloc, cudaFree or allocating library
// routine.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "muon.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = MUON_STATIC_SCRATCH_BYTES;
constexpr size_t kFlagBytes = 256;   // device error word(s) at the front
constexpr size_t kAlignS = 256;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a host-side stand-in: its
// device address comes from cudaGetSymbolAddress at set-up.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Per-device set-up state.  The address is latched only once a set-up
// succeeded: a failed attempt (say, a first call made during a stream
// capture) leaves `ready` unset and the next call tries again.
struct DeviceSetup {
  bool ready = false;
  uint8_t* scratch = nullptr;  // device address of g_static_scratch
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

size_t align_s(size_t v) { return (v + kAlignS - 1) / kAlignS * kAlignS; }

muon_status_t fail_s(muon_status_t st, const char* msg) {
  muon::report(st, msg);
  return st;
}

// Once per device, with that device current: resolve the scratch address
// and set the kernels' shared-memory attribute.
cudaError_t setup_device(int dev, uint8_t** scratch) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& S = g_setup[dev];
  if (!S.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e == cudaSuccess) e = muon::ns_gemm_init();
    if (e != cudaSuccess) {
      cudaGetLastError();  // leave no sticky-looking error behind; retry next call
      *scratch = nullptr;
      return e;
    }
    S.scratch = static_cast<uint8_t*>(p);
    S.ready = true;
  }
  *scratch = S.scratch;
  return cudaSuccess;
}

}  // namespace

extern "C" muon_status_t muon_newton_schulz_bf16_static(int32_t m, int32_t n, int32_t count,
                                                        const uint16_t* x_dev, uint16_t* out_dev,
                                                        const float* inv_norm_dev,
                                                        int32_t ns_steps, const float* coeffs_host,
                                                        int32_t* error_flag_dev, void* stream) {
  if (m < 1 || n < 1 || m > n || m > muon::kMaxDim || n > muon::kMaxDim || count < 0 ||
      (m % 8) != 0 || (n % 8) != 0)
    return fail_s(MUON_ERR_INVALID_ARG,
                  "need 1 <= m <= n <= 2^20, both multiples of 8, and count >= 0");
  if (ns_steps < 0 || ns_steps > muon::kMaxSteps)
    return fail_s(MUON_ERR_INVALID_ARG, "ns_steps out of range");
  float a = MUON_NS_A, b = MUON_NS_B, c = MUON_NS_C;
  if (coeffs_host != nullptr) {
    a = coeffs_host[0];
    b = coeffs_host[1];
    c = coeffs_host[2];
    if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c))
      return fail_s(MUON_ERR_INVALID_ARG, "coefficients not finite");
  }
  // One matrix needs one more iterate (m x n) plus A and B (m x m).
  const size_t per = align_s(size_t(m) * n * 2) + 2 * align_s(size_t(m) * m * 2);
  if (per > kStaticScratchBytes - kFlagBytes)
    return fail_s(MUON_ERR_INVALID_ARG,
                        "one matrix needs more scratch than the fixed static array holds "
                        "(m*n*2 + 2*m*m*2 bytes must fit MUON_STATIC_SCRATCH_BYTES - 256)");
  if (count == 0) return MUON_OK;
  if (x_dev == nullptr || out_dev == nullptr || inv_norm_dev == nullptr)
    return fail_s(MUON_ERR_INVALID_ARG, "NULL buffer");
  if ((reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(out_dev)) & 15u)
    return fail_s(MUON_ERR_INVALID_ARG, "x/out must be 16-byte aligned");
  const size_t xbytes = size_t(count) * m * n * 2;
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x_dev), ob = reinterpret_cast<uintptr_t>(out_dev);
  if (xb < ob + xbytes && ob < xb + xbytes)
    return fail_s(MUON_ERR_INVALID_ARG, "x and out overlap");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail_s(MUON_ERR_CUDA, "no current device");
  uint8_t* scratch = nullptr;
  if (setup_device(dev, &scratch) != cudaSuccess || scratch == nullptr)
    return fail_s(MUON_ERR_CUDA, "static scratch set-up failed (cudaGetSymbolAddress)");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = error_flag_dev != nullptr ? reinterpret_cast<int*>(error_flag_dev)
                                       : reinterpret_cast<int*>(scratch);
  if (error_flag_dev == nullptr && cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess)
    return fail_s(MUON_ERR_CUDA, "clearing the error word failed");

  // Matrices per pass through the scratch; the batch is walked in passes.
  int64_t cap = static_cast<int64_t>((kStaticScratchBytes - kFlagBytes) / per);
  cap = std::min<int64_t>(cap, count);
  cap = std::min<int64_t>(cap, muon::ns_max_count_per_launch(m, n));
  uint8_t* base = scratch + kFlagBytes;
  const size_t xs = align_s(size_t(cap) * m * n * 2), as = align_s(size_t(cap) * m * m * 2);
  uint16_t* other = reinterpret_cast<uint16_t*>(base);
  uint16_t* A = reinterpret_cast<uint16_t*>(base + xs);
  uint16_t* B = reinterpret_cast<uint16_t*>(base + xs + as);
  const int64_t xms = int64_t(m) * n, ams = int64_t(m) * m;

  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail_s(MUON_ERR_CUDA, "cannot read the SM count");
  for (int64_t done = 0; done < count; done += cap) {
    const int take = static_cast<int>(std::min<int64_t>(count - done, cap));
    const muon::BatchView vx{x_dev + done * xms, n, xms}, vo{out_dev + done * xms, n, xms};
    const muon::BatchView vt{other, n, xms}, vA{A, m, ams}, vB{B, m, ams};
    const float* inv = inv_norm_dev + done;
    cudaError_t e = cudaSuccess;
    if (ns_steps == 0) {
      e = muon::launch_scale_bf16(m, n, take, static_cast<const uint16_t*>(vx.ptr), n, xms,
                                  out_dev + done * xms, n, xms, inv, s);
      if (e != cudaSuccess) return fail_s(MUON_ERR_CUDA, "scale kernel launch failed");
      continue;
    }
    muon::BatchView src = vx;
    for (int k = 0; k < ns_steps && e == cudaSuccess; ++k) {
      const muon::BatchView dst = (((ns_steps - 1 - k) % 2) == 0) ? vo : vt;
      const float* alpha = (k == 0) ? inv : nullptr;
      e = muon::ns_launch_gram(m, n, take, src, vA, alpha, err, sms, s);
      if (e == cudaSuccess) e = muon::ns_launch_poly(m, take, vA, vB, a, b, c, err, sms, s);
      if (e == cudaSuccess) e = muon::ns_launch_update(m, n, take, vB, src, dst, alpha, err, sms, s);
      src = dst;
    }
    if (e != cudaSuccess) return fail_s(MUON_ERR_CUDA, "Newton-Schulz launch failed");
  }
  return MUON_OK;
}
