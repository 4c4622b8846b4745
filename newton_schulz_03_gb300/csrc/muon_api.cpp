// muon_api.cpp -- host side of the C ABI declared in include/muon.h.
//
// Responsibilities: argument validation (nothing is launched for an invalid
// call), the shape-group planner ("parameters of identical shape are packed
// into one batch", Frontier Pre-training at Microsoft AI, Method details §5,
// resharding step 2), the device workspace, the launch sequence of one step,
// per-kernel event timing and the device error flag.
//
// Plan: caller groups are keyed by their wide shape (m, n) = (min, max), so a
// tall group joins the batch of its transpose.  A batch is cut into chunks
// that fit the workspace.  Per chunk: momentum_cast for each caller segment,
// one norm finalisation, ns_steps x (gram, poly, update), apply for each
// segment.  The plan of a group list is cached, as the pages cache their
// resharding metadata ("resharding metadata caching").
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "muon.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

muon_status_t fail(muon_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

muon_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MUON_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kDefaultWorkspace = size_t(8) << 30;  // 8 GiB
constexpr size_t kAlign = 256;
using muon::kMaxDim;
using muon::kMaxSteps;
constexpr int64_t kMaxMatrixElems = int64_t(1) << 34;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t pad8(int64_t v) { return (v + 7) / 8 * 8; }

// Workspace layout of one chunk of `cap` matrices of wide shape m x n.
struct ChunkLayout {
  int64_t ldx, ldm;  // row pitches (elements) of X and of A/B
  int tiles;         // elementwise tiles per matrix (norm partials)
  size_t off_x0, off_x1, off_a, off_b, off_part, off_inv, bytes;
};

ChunkLayout chunk_layout(int m, int n, int64_t cap) {
  ChunkLayout L{};
  L.ldx = pad8(n);
  L.ldm = pad8(m);
  L.tiles = muon::ew_tiles_per_matrix(m, n);
  size_t off = 0;
  const size_t xb = align_up(size_t(cap) * m * L.ldx * 2, kAlign);
  const size_t ab = align_up(size_t(cap) * m * L.ldm * 2, kAlign);
  L.off_x0 = off; off += xb;
  L.off_x1 = off; off += xb;
  L.off_a = off; off += ab;
  L.off_b = off; off += ab;
  L.off_part = off; off += align_up(size_t(cap) * L.tiles * 4, kAlign);
  L.off_inv = off; off += align_up(size_t(cap) * 4, kAlign);
  L.bytes = off;
  return L;
}

size_t per_matrix_bytes(int m, int n) {
  const int64_t ldx = pad8(n), ldm = pad8(m);
  return size_t(2) * m * ldx * 2 + size_t(2) * m * ldm * 2 +
         size_t(muon::ew_tiles_per_matrix(m, n)) * 4 + 4;
}

struct Segment {
  int group;        // caller group index
  int64_t first;    // first matrix of the group in this segment
  int count;        // matrices
  int slot;         // first slot in the chunk
};

struct Chunk {
  int m, n;
  int count;
  std::vector<Segment> segs;
};

struct Plan {
  std::vector<Chunk> chunks;
  int n_batches = 0;
  int max_chunk = 0;
  int64_t matrices = 0;
  size_t ws_bytes = 0;
  double flops = 0.0;
  int64_t launches = 0;
};

muon_status_t validate_groups(const muon_group_t* groups, int32_t n_groups) {
  if (n_groups < 0) return fail(MUON_ERR_INVALID_ARG, "n_groups < 0");
  if (n_groups > 0 && groups == nullptr) return fail(MUON_ERR_INVALID_ARG, "groups is NULL");
  for (int g = 0; g < n_groups; ++g) {
    const muon_group_t& G = groups[g];
    if (G.rows < 1 || G.cols < 1 || G.rows > kMaxDim || G.cols > kMaxDim)
      return fail(MUON_ERR_INVALID_ARG, "group %d: rows/cols out of range (%d x %d)", g, G.rows,
                  G.cols);
    if (G.count < 0) return fail(MUON_ERR_INVALID_ARG, "group %d: count < 0", g);
    if (int64_t(G.rows) * G.cols > kMaxMatrixElems)
      return fail(MUON_ERR_INVALID_ARG, "group %d: matrix of %d x %d is too large", g, G.rows,
                  G.cols);
    if (!std::isfinite(G.update_scale))
      return fail(MUON_ERR_INVALID_ARG, "group %d: update_scale not finite", g);
  }
  return MUON_OK;
}

muon_status_t build_plan(const muon_group_t* groups, int32_t n_groups, int32_t ns_steps,
                         size_t ws_cap, Plan* plan) {
  muon_status_t st = validate_groups(groups, n_groups);
  if (st != MUON_OK) return st;
  if (ns_steps < 0 || ns_steps > kMaxSteps)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps out of range (%d)", ns_steps);
  if (ws_cap == 0) ws_cap = kDefaultWorkspace;
  // Batches keyed by wide shape, in order of first appearance.
  std::vector<std::pair<std::pair<int, int>, std::vector<int>>> batches;
  std::map<std::pair<int, int>, size_t> index;
  for (int g = 0; g < n_groups; ++g) {
    if (groups[g].count == 0) continue;
    const std::pair<int, int> key{std::min(groups[g].rows, groups[g].cols),
                                  std::max(groups[g].rows, groups[g].cols)};
    auto it = index.find(key);
    if (it == index.end()) {
      index[key] = batches.size();
      batches.push_back({key, {g}});
    } else {
      batches[it->second].second.push_back(g);
    }
  }
  Plan P;
  P.n_batches = static_cast<int>(batches.size());
  for (auto& b : batches) {
    const int m = b.first.first, n = b.first.second;
    int64_t total = 0;
    for (int g : b.second) total += groups[g].count;
    const size_t pm = per_matrix_bytes(m, n);
    int64_t cap = static_cast<int64_t>((ws_cap > 8 * kAlign ? ws_cap - 8 * kAlign : 0) / pm);
    if (cap < 1) cap = 1;  // a single matrix always gets room
    if (cap > total) cap = total;
    cap = std::min(cap, muon::ns_max_count_per_launch(m, n));  // also the grid.y limit
    P.ws_bytes = std::max(P.ws_bytes, chunk_layout(m, n, cap).bytes);
    P.matrices += total;
    P.flops += double(total) * ns_steps * (3.0 * m * double(m) * n + double(m) * m * m);
    // Cut the batch into chunks of at most `cap` matrices.
    Chunk cur{m, n, 0, {}};
    for (int g : b.second) {
      int64_t done = 0;
      while (done < groups[g].count) {
        const int64_t take = std::min<int64_t>(groups[g].count - done, cap - cur.count);
        cur.segs.push_back({g, done, static_cast<int>(take), cur.count});
        cur.count += static_cast<int>(take);
        done += take;
        if (cur.count == cap) {
          P.chunks.push_back(cur);
          cur = Chunk{m, n, 0, {}};
        }
      }
    }
    if (cur.count > 0) P.chunks.push_back(cur);
  }
  for (const Chunk& c : P.chunks) {
    P.max_chunk = std::max(P.max_chunk, c.count);
    P.launches += 2 * static_cast<int64_t>(c.segs.size()) + 1 + (ns_steps > 0 ? 3 * ns_steps : 1);
  }
  *plan = std::move(P);
  return MUON_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// ---------------------------------------------------------------- the handle
struct muon_handle_s {
  int device = 0;
  int num_sms = 0;
  size_t ws_cap = kDefaultWorkspace;
  void* ws = nullptr;
  size_t ws_size = 0;
  int* dev_err = nullptr;
  // Host-buffer step: device staging ring, copy streams and their events.
  float* staging = nullptr;
  size_t staging_bytes = 0;
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t entry_ev = nullptr;
  cudaEvent_t slot_in[3] = {nullptr, nullptr, nullptr};
  cudaEvent_t slot_comp[3] = {nullptr, nullptr, nullptr};
  cudaEvent_t slot_out[3] = {nullptr, nullptr, nullptr};
  bool timing = false;
  struct Pending {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> free_events;
  muon_kernel_stats_t stats{};
  // Plan cache keyed by the group list and step count.
  std::string plan_key;
  Plan plan;
};

namespace {

cudaEvent_t get_event(muon_handle_t h) {
  if (!h->free_events.empty()) {
    cudaEvent_t e = h->free_events.back();
    h->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Brackets one kernel launch for accounting and (optionally) timing.
struct LaunchScope {
  muon_handle_t h;
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  LaunchScope(muon_handle_t h_, int kind_, cudaStream_t s_) : h(h_), kind(kind_), s(s_) {
    if (h->timing) {
      a = get_event(h);
      cudaEventRecord(a, s);
    }
  }
  ~LaunchScope() {
    h->stats.launches[kind] += 1;
    h->stats.total_launches += 1;
    if (h->timing && a != nullptr) {
      cudaEvent_t b = get_event(h);
      cudaEventRecord(b, s);
      h->pending.push_back({kind, a, b});
    }
  }
};

muon_status_t ensure_workspace(muon_handle_t h, size_t bytes) {
  if (h->ws_size >= bytes) return MUON_OK;
  if (h->ws != nullptr) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    cudaFree(h->ws);
    h->ws = nullptr;
    h->ws_size = 0;
  }
  cudaError_t e = cudaMalloc(&h->ws, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(MUON_ERR_NOMEM, "workspace allocation of %zu bytes failed: %s", bytes,
                cudaGetErrorString(e));
  }
  h->ws_size = bytes;
  return MUON_OK;
}

struct Coeffs {
  float a, b, c;
};

// ns_steps iterations on `count` wide matrices.  Reads x (never written);
// iteration k writes dst[k]; the last one lands in `out`.  A, B: scratch.
// `sched` holds the (a, b, c) of every iteration (at least `steps` entries).
muon_status_t run_newton_schulz(muon_handle_t h, int m, int n, int count, muon::BatchView x,
                                muon::BatchView out, muon::BatchView other, muon::BatchView A,
                                muon::BatchView B, const float* inv_norm, int steps,
                                const Coeffs* sched, cudaStream_t s) {
  if (steps == 0) {
    LaunchScope L(h, MUON_KERNEL_SCALE, s);
    cudaError_t e = muon::launch_scale_bf16(
        m, n, count, static_cast<const uint16_t*>(x.ptr), x.ld, x.ms,
        static_cast<uint16_t*>(const_cast<void*>(out.ptr)), out.ld, out.ms, inv_norm, s);
    if (e != cudaSuccess) return cuda_fail(e, "scale kernel launch");
    return MUON_OK;
  }
  muon::BatchView src = x;
  for (int k = 0; k < steps; ++k) {
    // Alternate so that the final iteration writes `out`.
    const bool to_out = ((steps - 1 - k) % 2) == 0;
    muon::BatchView dst = to_out ? out : other;
    const float* inv = (k == 0) ? inv_norm : nullptr;
    const Coeffs co = sched[k];
    cudaError_t e;
    {
      LaunchScope L(h, MUON_KERNEL_NS_GRAM, s);
      e = muon::ns_launch_gram(m, n, count, src, A, inv, h->dev_err, h->num_sms, s);
    }
    if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "gram launch: %s %s", cudaGetErrorString(e),
                                      muon::ns_last_encode_error());
    {
      LaunchScope L(h, MUON_KERNEL_NS_POLY, s);
      e = muon::ns_launch_poly(m, count, A, B, co.a, co.b, co.c, h->dev_err, h->num_sms, s);
    }
    if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "poly launch: %s %s", cudaGetErrorString(e),
                                      muon::ns_last_encode_error());
    {
      LaunchScope L(h, MUON_KERNEL_NS_UPDATE, s);
      e = muon::ns_launch_update(m, n, count, B, src, dst, inv, h->dev_err, h->num_sms, s);
    }
    if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "update launch: %s %s",
                                      cudaGetErrorString(e), muon::ns_last_encode_error());
    src = dst;
  }
  return MUON_OK;
}

std::string plan_key_of(const muon_group_t* groups, int32_t n, int32_t steps) {
  std::string k;
  k.reserve(16 * n + 8);
  char buf[64];
  snprintf(buf, sizeof(buf), "%d;", steps);
  k += buf;
  for (int i = 0; i < n; ++i) {
    snprintf(buf, sizeof(buf), "%d,%d,%d;", groups[i].rows, groups[i].cols, groups[i].count);
    k += buf;
  }
  return k;
}

muon_status_t check_handle(muon_handle_t h) {
  if (h == nullptr) return fail(MUON_ERR_INVALID_ARG, "handle is NULL");
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != h->device) {
    cudaError_t e = cudaSetDevice(h->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  }
  return MUON_OK;
}

bool finite3(float a, float b, float c) {
  return std::isfinite(a) && std::isfinite(b) && std::isfinite(c);
}

}  // namespace

namespace muon {
int report(int status, const char* msg) {
  g_last_error = msg;
  return status;
}
}  // namespace muon

// ======================================================================== ABI
extern "C" {

const char* muon_status_string(muon_status_t s) {
  switch (s) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG";
    case MUON_ERR_NOMEM: return "MUON_ERR_NOMEM";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA";
    case MUON_ERR_UNSUPPORTED_ARCH: return "MUON_ERR_UNSUPPORTED_ARCH";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT";
    case MUON_ERR_NONFINITE: return "MUON_ERR_NONFINITE";
    case MUON_ERR_NO_DEVICE: return "MUON_ERR_NO_DEVICE";
  }
  return "MUON_ERR_UNKNOWN";
}

const char* muon_last_error_message(void) { return g_last_error.c_str(); }

const char* muon_version(void) { return "muon-gb300 0.1.0 (sm_103a)"; }

muon_status_t muon_create(muon_handle_t* out, int32_t device, size_t workspace_bytes_max) {
  if (out == nullptr) return fail(MUON_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return fail(MUON_ERR_NO_DEVICE, "no CUDA device visible (%s)",
                e == cudaSuccess ? "count 0" : cudaGetErrorString(e));
  }
  if (device < 0) {
    e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  }
  if (device >= ndev) return fail(MUON_ERR_INVALID_ARG, "device %d >= %d devices", device, ndev);
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (major != 10 || minor != 3)
    return fail(MUON_ERR_UNSUPPORTED_ARCH, "device %d is sm_%d%d; this library is built for sm_103a",
                device, major, minor);
  e = cudaSetDevice(device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  e = muon::ns_gemm_init();
  if (e != cudaSuccess) return cuda_fail(e, "kernel attribute setup");
  muon_handle_t h = new muon_handle_s();
  h->device = device;
  h->num_sms = sms;
  h->ws_cap = workspace_bytes_max == 0 ? kDefaultWorkspace : workspace_bytes_max;
  e = cudaMalloc(reinterpret_cast<void**>(&h->dev_err), 256);
  if (e != cudaSuccess) {
    delete h;
    return fail(MUON_ERR_NOMEM, "error-flag allocation failed: %s", cudaGetErrorString(e));
  }
  cudaMemset(h->dev_err, 0, 256);
  cudaDeviceSynchronize();
  *out = h;
  return MUON_OK;
}

muon_status_t muon_destroy(muon_handle_t h) {
  if (h == nullptr) return MUON_OK;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  for (auto& p : h->pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (cudaEvent_t e : h->free_events) cudaEventDestroy(e);
  if (h->ws) cudaFree(h->ws);
  if (h->staging) cudaFree(h->staging);
  if (h->copy_in) cudaStreamDestroy(h->copy_in);
  if (h->copy_out) cudaStreamDestroy(h->copy_out);
  if (h->entry_ev) cudaEventDestroy(h->entry_ev);
  for (int i = 0; i < 3; ++i) {
    if (h->slot_in[i]) cudaEventDestroy(h->slot_in[i]);
    if (h->slot_comp[i]) cudaEventDestroy(h->slot_comp[i]);
    if (h->slot_out[i]) cudaEventDestroy(h->slot_out[i]);
  }
  if (h->dev_err) cudaFree(h->dev_err);
  delete h;
  return MUON_OK;
}

muon_status_t muon_plan_describe(const muon_group_t* groups, int32_t n_groups, int32_t ns_steps,
                                 size_t workspace_bytes_max, muon_plan_info_t* out) {
  if (out == nullptr) return fail(MUON_ERR_INVALID_ARG, "out is NULL");
  Plan P;
  muon_status_t st = build_plan(groups, n_groups, ns_steps, workspace_bytes_max, &P);
  if (st != MUON_OK) return st;
  out->n_batches = P.n_batches;
  out->n_chunks = static_cast<int32_t>(P.chunks.size());
  out->max_chunk_matrices = P.max_chunk;
  out->matrices = P.matrices;
  out->workspace_bytes = P.ws_bytes;
  out->ns_algorithmic_flops = P.flops;
  out->launches_per_step = P.launches;
  return MUON_OK;
}

muon_status_t muon_partition(const muon_group_t* groups, int32_t n_groups, int32_t ns_steps,
                             int32_t world, int64_t* first_out, int32_t* count_out,
                             double* rank_seconds_out) {
  muon_status_t st = validate_groups(groups, n_groups);
  if (st != MUON_OK) return st;
  if (ns_steps < 0 || ns_steps > kMaxSteps)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps out of range (%d)", ns_steps);
  if (world < 1 || world > 65536) return fail(MUON_ERR_INVALID_ARG, "world out of range (%d)", world);
  if (n_groups > 0 && (first_out == nullptr || count_out == nullptr))
    return fail(MUON_ERR_INVALID_ARG, "first_out and count_out must not be NULL");
  // Estimated device seconds of one matrix: its algorithmic Newton-Schulz
  // flops at the tensor rate plus its elementwise bytes (momentum update +
  // cast 14 B, apply 10 B per element) at the HBM rate.
  constexpr double kFlopRate = 1.9e15, kByteRate = 6.8e12;
  std::vector<double> cost(n_groups);
  for (int g = 0; g < n_groups; ++g) {
    const double m = std::min(groups[g].rows, groups[g].cols);
    const double n = std::max(groups[g].rows, groups[g].cols);
    cost[g] = ns_steps * (3.0 * m * m * n + m * m * m) / kFlopRate + 24.0 * m * n / kByteRate;
  }
  // Longest processing time first: matrices in order of decreasing cost
  // (a group's matrices are identical, so a group is one run of the
  // order), each to the rank with the least load so far.
  std::vector<int> order(n_groups);
  for (int g = 0; g < n_groups; ++g) order[g] = g;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  using Load = std::pair<double, int>;  // (seconds, rank): ties go to the lower rank
  std::vector<Load> heap;
  for (int r = 0; r < world; ++r) heap.push_back({0.0, r});
  auto later = [](const Load& a, const Load& b) { return a > b; };
  std::make_heap(heap.begin(), heap.end(), later);
  std::vector<int64_t> per(size_t(n_groups) * world, 0);
  for (int g : order) {
    for (int64_t i = 0; i < groups[g].count; ++i) {
      std::pop_heap(heap.begin(), heap.end(), later);
      Load& least = heap.back();
      least.first += cost[g];
      per[size_t(g) * world + least.second] += 1;
      std::push_heap(heap.begin(), heap.end(), later);
    }
  }
  // A rank's matrices of one group form one contiguous slice (ranks in
  // order), so each rank passes a group as one pointer and count.
  std::vector<double> load(world, 0.0);
  for (int g = 0; g < n_groups; ++g) {
    int64_t first = 0;
    for (int r = 0; r < world; ++r) {
      const int64_t c = per[size_t(g) * world + r];
      first_out[size_t(g) * world + r] = first;
      count_out[size_t(g) * world + r] = static_cast<int32_t>(c);
      load[r] += static_cast<double>(c) * cost[g];
      first += c;
    }
  }
  if (rank_seconds_out != nullptr)
    for (int r = 0; r < world; ++r) rank_seconds_out[r] = load[r];
  return MUON_OK;
}

}  // extern "C"

namespace {

// Everything a step needs beyond the buffers.
struct StepOptions {
  float lr, wd, mu;
  int32_t ns_steps;
  bool nesterov = false;
  std::vector<Coeffs> sched;  // one (a, b, c) per iteration
  int32_t scale_rule = MUON_SCALE_NONE;
  float rms_target = 0.2f;
};

// FP32 shape factor of a rule (sqrt of an FP32 ratio or size).
float rule_scale(int32_t rule, int rows, int cols, float rms_target) {
  switch (rule) {
    case MUON_SCALE_SQRT_ASPECT:
      return sqrtf(fmaxf(1.0f, static_cast<float>(rows) / static_cast<float>(cols)));
    case MUON_SCALE_RMS_MATCH:
      return rms_target * sqrtf(static_cast<float>(std::max(rows, cols)));
    default:
      return 1.0f;
  }
}

muon_status_t step_impl(muon_handle_t h, const muon_group_t* groups, int32_t n_groups,
                        float* const* momentum, const float* const* grad, float* const* weights,
                        const StepOptions& o, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (!finite3(o.lr, o.wd, o.mu)) return fail(MUON_ERR_INVALID_ARG, "lr, wd and mu must be finite");
  st = validate_groups(groups, n_groups);
  if (st != MUON_OK) return st;
  if (n_groups > 0 && (momentum == nullptr || grad == nullptr || weights == nullptr))
    return fail(MUON_ERR_INVALID_ARG, "pointer arrays must not be NULL");
  for (int g = 0; g < n_groups; ++g) {
    if (groups[g].count == 0) continue;
    if (momentum[g] == nullptr || grad[g] == nullptr || weights[g] == nullptr)
      return fail(MUON_ERR_INVALID_ARG, "group %d: NULL buffer", g);
    if (!aligned16(momentum[g]) || !aligned16(grad[g]) || !aligned16(weights[g]))
      return fail(MUON_ERR_INVALID_ARG, "group %d: buffers must be 16-byte aligned", g);
  }
  const int32_t ns_steps = o.ns_steps;
  const std::string key = plan_key_of(groups, n_groups, ns_steps);
  if (key != h->plan_key) {
    Plan P;
    st = build_plan(groups, n_groups, ns_steps, h->ws_cap, &P);
    if (st != MUON_OK) return st;
    h->plan = std::move(P);
    h->plan_key = key;
  }
  const Plan& P = h->plan;
  st = ensure_workspace(h, P.ws_bytes);
  if (st != MUON_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(h->ws);
  for (const Chunk& c : P.chunks) {
    const ChunkLayout L = chunk_layout(c.m, c.n, c.count);
    uint16_t* x0 = reinterpret_cast<uint16_t*>(ws + L.off_x0);
    uint16_t* x1 = reinterpret_cast<uint16_t*>(ws + L.off_x1);
    uint16_t* A = reinterpret_cast<uint16_t*>(ws + L.off_a);
    uint16_t* B = reinterpret_cast<uint16_t*>(ws + L.off_b);
    float* part = reinterpret_cast<float*>(ws + L.off_part);
    float* inv = reinterpret_cast<float*>(ws + L.off_inv);
    const int64_t xms = int64_t(c.m) * L.ldx, ams = int64_t(c.m) * L.ldm;
    for (const Segment& sg : c.segs) {
      const muon_group_t& G = groups[sg.group];
      const int64_t off = sg.first * int64_t(G.rows) * G.cols;
      LaunchScope Ls(h, MUON_KERNEL_MOMENTUM_CAST, s);
      cudaError_t e = muon::launch_momentum_cast(
          G.rows, G.cols, sg.count, momentum[sg.group] + off, grad[sg.group] + off, o.mu,
          x0 + sg.slot * xms, L.ldx, xms, part + int64_t(sg.slot) * L.tiles, s, o.nesterov);
      if (e != cudaSuccess) return cuda_fail(e, "momentum_cast launch");
    }
    {
      LaunchScope Ls(h, MUON_KERNEL_NORM, s);
      cudaError_t e = muon::launch_norm_finalize(part, L.tiles, c.count, MUON_NORM_EPS, inv,
                                                 h->dev_err, x0, L.ldx, xms, c.m, c.n, s);
      if (e != cudaSuccess) return cuda_fail(e, "norm launch");
    }
    // The iterates alternate between x0 and x1, starting from x0; the
    // final one lands in x0 for an even (non-zero) step count, else in x1.
    uint16_t* fin = (ns_steps > 0 && ns_steps % 2 == 0) ? x0 : x1;
    uint16_t* oth = (fin == x0) ? x1 : x0;
    const muon::BatchView vx0{x0, L.ldx, xms}, vfin{fin, L.ldx, xms}, voth{oth, L.ldx, xms};
    const muon::BatchView vA{A, L.ldm, ams}, vB{B, L.ldm, ams};
    st = run_newton_schulz(h, c.m, c.n, c.count, vx0, vfin, voth, vA, vB, inv, ns_steps,
                           o.sched.data(), s);
    if (st != MUON_OK) return st;
    for (const Segment& sg : c.segs) {
      const muon_group_t& G = groups[sg.group];
      const int64_t off = sg.first * int64_t(G.rows) * G.cols;
      const float scale = G.update_scale * rule_scale(o.scale_rule, G.rows, G.cols, o.rms_target);
      LaunchScope Ls(h, MUON_KERNEL_APPLY, s);
      cudaError_t e = muon::launch_apply_update(G.rows, G.cols, sg.count, weights[sg.group] + off,
                                                fin + sg.slot * xms, L.ldx, xms, o.lr, o.wd,
                                                scale, s);
      if (e != cudaSuccess) return cuda_fail(e, "apply launch");
    }
  }
  return MUON_OK;
}

StepOptions default_options(float lr, float wd, float mu, int32_t ns_steps) {
  StepOptions o;
  o.lr = lr;
  o.wd = wd;
  o.mu = mu;
  o.ns_steps = ns_steps;
  o.sched.assign(ns_steps > 0 ? ns_steps : 1, Coeffs{MUON_NS_A, MUON_NS_B, MUON_NS_C});
  return o;
}

}  // namespace

extern "C" {

muon_status_t muon_step(muon_handle_t h, const muon_group_t* groups, int32_t n_groups,
                        float* const* momentum, const float* const* grad, float* const* weights,
                        float lr, float wd, float mu, int32_t ns_steps, void* stream) {
  if (ns_steps < 0 || ns_steps > kMaxSteps)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps out of range (%d)", ns_steps);
  return step_impl(h, groups, n_groups, momentum, grad, weights,
                   default_options(lr, wd, mu, ns_steps), stream);
}

muon_status_t muon_step_ex(muon_handle_t h, const muon_group_t* groups, int32_t n_groups,
                           float* const* momentum, const float* const* grad,
                           float* const* weights, const muon_options_t* opts, void* stream) {
  if (opts == nullptr) return fail(MUON_ERR_INVALID_ARG, "opts is NULL");
  if (opts->ns_steps < 0 || opts->ns_steps > kMaxSteps)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps out of range (%d)", opts->ns_steps);
  if (opts->scale_rule < MUON_SCALE_NONE || opts->scale_rule > MUON_SCALE_RMS_MATCH)
    return fail(MUON_ERR_INVALID_ARG, "unknown scale_rule %d", opts->scale_rule);
  StepOptions o = default_options(opts->lr, opts->wd, opts->mu, opts->ns_steps);
  o.nesterov = opts->nesterov != 0;
  o.scale_rule = opts->scale_rule;
  o.rms_target = opts->rms_target > 0.f ? opts->rms_target : 0.2f;
  if (!std::isfinite(o.rms_target)) return fail(MUON_ERR_INVALID_ARG, "rms_target not finite");
  if (opts->coeffs != nullptr) {
    for (int k = 0; k < opts->ns_steps; ++k) {
      const Coeffs c{opts->coeffs[3 * k], opts->coeffs[3 * k + 1], opts->coeffs[3 * k + 2]};
      if (!finite3(c.a, c.b, c.c)) return fail(MUON_ERR_INVALID_ARG, "coefficient %d not finite", k);
      o.sched[k] = c;
    }
  }
  return step_impl(h, groups, n_groups, momentum, grad, weights, o, stream);
}

muon_status_t muon_step_host(muon_handle_t h, const muon_group_t* groups, int32_t n_groups,
                             float* const* momentum_host, const float* const* grad_host,
                             float* const* weights_host, float lr, float wd, float mu,
                             int32_t ns_steps, void* stream) {
  // Pipeline over pieces of at most kPieceBytes of state: while piece k is
  // stepped on `stream`, piece k+1 is copied in on one copy stream and
  // piece k-1 is copied out on another.  A ring of three device slots holds
  // the pieces' momentum, gradient and weights.
  constexpr size_t kPieceBytes = size_t(384) << 20;
  constexpr int kSlots = 3;
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  st = validate_groups(groups, n_groups);
  if (st != MUON_OK) return st;
  if (!finite3(lr, wd, mu)) return fail(MUON_ERR_INVALID_ARG, "lr, wd and mu must be finite");
  if (ns_steps < 0 || ns_steps > kMaxSteps)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps out of range (%d)", ns_steps);
  if (n_groups > 0 && (momentum_host == nullptr || grad_host == nullptr || weights_host == nullptr))
    return fail(MUON_ERR_INVALID_ARG, "pointer arrays must not be NULL");
  for (int g = 0; g < n_groups; ++g) {
    if (groups[g].count == 0) continue;
    if (momentum_host[g] == nullptr || grad_host[g] == nullptr || weights_host[g] == nullptr)
      return fail(MUON_ERR_INVALID_ARG, "group %d: NULL host buffer", g);
  }

  // Pieces: consecutive runs of matrices of one group.
  struct Piece {
    int group;
    int64_t first;
    int count;
  };
  std::vector<Piece> pieces;
  size_t slot_elems = 64;
  for (int g = 0; g < n_groups; ++g) {
    const int64_t per = int64_t(groups[g].rows) * groups[g].cols;
    int64_t take = std::max<int64_t>(1, static_cast<int64_t>(kPieceBytes / (12 * size_t(per))));
    for (int64_t first = 0; first < groups[g].count; first += take) {
      const int c = static_cast<int>(std::min<int64_t>(take, groups[g].count - first));
      pieces.push_back({g, first, c});
      slot_elems = std::max(slot_elems, align_up(size_t(per) * c, 64));
    }
  }
  if (pieces.empty()) return MUON_OK;
  // Nothing overlaps the first piece's copy in or the last piece's copy
  // out: split those two into pieces of 1, 2, 4, ... units so that the
  // pipeline fills and drains with small copies.
  {
    // Smallest ramp piece: 16 MB of state or one matrix.
    auto ramp = [groups](const Piece& p, bool up) {
      std::vector<Piece> out;
      int left = p.count;
      const int64_t per = int64_t(groups[p.group].rows) * groups[p.group].cols;
      const int unit = static_cast<int>(
          std::max<int64_t>(1, static_cast<int64_t>((size_t(16) << 20) / (12 * size_t(per)))));
      std::vector<int> sizes;
      for (int s = unit; left > 0; s *= 2) {
        const int take = std::min(s, left);
        sizes.push_back(take);
        left -= take;
        if (2 * s >= left) {        // the rest in one piece (never above the original)
          if (left > 0) sizes.push_back(left);
          break;
        }
      }
      if (!up) std::reverse(sizes.begin(), sizes.end());
      int64_t first = p.first;
      for (int s : sizes) {
        out.push_back({p.group, first, s});
        first += s;
      }
      return out;
    };
    std::vector<Piece> head = ramp(pieces.front(), true);
    std::vector<Piece> rebuilt(head.begin(), head.end());
    if (pieces.size() > 1) {
      rebuilt.insert(rebuilt.end(), pieces.begin() + 1, pieces.end() - 1);
      std::vector<Piece> tail = ramp(pieces.back(), false);
      rebuilt.insert(rebuilt.end(), tail.begin(), tail.end());
    }
    pieces.swap(rebuilt);
  }

  // Size the workspace for the largest piece now: growing it inside the
  // loop would synchronise the device between pieces.
  {
    size_t need = 0;
    for (const Piece& pc : pieces) {
      const muon_group_t pg{groups[pc.group].rows, groups[pc.group].cols, pc.count, 1.0f};
      Plan P;
      st = build_plan(&pg, 1, ns_steps, h->ws_cap, &P);
      if (st != MUON_OK) return st;
      need = std::max(need, P.ws_bytes);
    }
    st = ensure_workspace(h, need);
    if (st != MUON_OK) return st;
  }

  const size_t bytes = size_t(kSlots) * 3 * slot_elems * sizeof(float);
  if (h->staging_bytes < bytes) {
    if (h->staging) {
      cudaDeviceSynchronize();
      cudaFree(h->staging);
      h->staging = nullptr;
      h->staging_bytes = 0;
    }
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&h->staging), bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(MUON_ERR_NOMEM, "staging allocation of %zu bytes failed", bytes);
    }
    h->staging_bytes = bytes;
  }
  if (h->copy_in == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->entry_ev, cudaEventDisableTiming);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&h->slot_in[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->slot_comp[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->slot_out[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(e, "copy stream set-up");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaEventRecord(h->entry_ev, s);  // order after prior work on `stream`
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_in, h->entry_ev, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_out, h->entry_ev, 0);
  if (e != cudaSuccess) return cuda_fail(e, "stream ordering");

  for (size_t k = 0; k < pieces.size(); ++k) {
    const Piece& pc = pieces[k];
    const int slot = static_cast<int>(k % kSlots);
    const muon_group_t& G = groups[pc.group];
    const size_t ne = size_t(G.rows) * G.cols * pc.count;
    const size_t off = size_t(pc.first) * G.rows * G.cols;
    float* dM = h->staging + size_t(slot) * 3 * slot_elems;
    float* dG = dM + slot_elems;
    float* dW = dG + slot_elems;
    // Copy in once the slot's previous piece has been copied out.
    if (k >= static_cast<size_t>(kSlots)) e = cudaStreamWaitEvent(h->copy_in, h->slot_out[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dM, momentum_host[pc.group] + off, ne * 4, cudaMemcpyHostToDevice, h->copy_in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dG, grad_host[pc.group] + off, ne * 4, cudaMemcpyHostToDevice, h->copy_in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dW, weights_host[pc.group] + off, ne * 4, cudaMemcpyHostToDevice, h->copy_in);
    if (e == cudaSuccess) e = cudaEventRecord(h->slot_in[slot], h->copy_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->slot_in[slot], 0);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    const muon_group_t pg{G.rows, G.cols, pc.count, G.update_scale};
    float* pm[1] = {dM};
    const float* pgr[1] = {dG};
    float* pw[1] = {dW};
    st = muon_step(h, &pg, 1, pm, pgr, pw, lr, wd, mu, ns_steps, stream);
    if (st != MUON_OK) return st;
    e = cudaEventRecord(h->slot_comp[slot], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_out, h->slot_comp[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(momentum_host[pc.group] + off, dM, ne * 4, cudaMemcpyDeviceToHost, h->copy_out);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(weights_host[pc.group] + off, dW, ne * 4, cudaMemcpyDeviceToHost, h->copy_out);
    if (e == cudaSuccess) e = cudaEventRecord(h->slot_out[slot], h->copy_out);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
  }
  e = cudaStreamSynchronize(h->copy_out);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  return MUON_OK;
}

muon_status_t muon_shard_momentum_cast(muon_handle_t h, int64_t shard_begin, int64_t shard_end,
                                       int64_t matrix_elems, float* momentum_shard,
                                       const float* grad_shard, float mu, uint16_t* x_shard,
                                       float* sumsq_out, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (matrix_elems < 1 || shard_begin < 0 || shard_end < shard_begin)
    return fail(MUON_ERR_INVALID_ARG, "need matrix_elems >= 1 and 0 <= shard_begin <= shard_end");
  if (!std::isfinite(mu)) return fail(MUON_ERR_INVALID_ARG, "mu must be finite");
  if (shard_end == shard_begin) return MUON_OK;
  if (momentum_shard == nullptr || grad_shard == nullptr || x_shard == nullptr ||
      sumsq_out == nullptr)
    return fail(MUON_ERR_INVALID_ARG, "NULL buffer");
  const int64_t pieces = (shard_end - 1) / matrix_elems - shard_begin / matrix_elems + 1;
  const int blocks =
      muon::shard_cast_blocks(std::min<int64_t>(matrix_elems, shard_end - shard_begin));
  st = ensure_workspace(h, std::max(h->ws_size, align_up(size_t(pieces) * blocks * 4, kAlign)));
  if (st != MUON_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchScope Ls(h, MUON_KERNEL_MOMENTUM_CAST, s);
  cudaError_t e = muon::launch_shard_cast(shard_begin, shard_end, matrix_elems, momentum_shard,
                                          grad_shard, mu, x_shard, static_cast<float*>(h->ws),
                                          blocks, sumsq_out, s);
  if (e != cudaSuccess) return cuda_fail(e, "shard cast launch");
  return MUON_OK;
}

muon_status_t muon_norm_from_sumsq(muon_handle_t h, int32_t m, int32_t n, int32_t count,
                                   int32_t parts, const float* sumsq, uint16_t* x_wide,
                                   float* inv_norm, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (m < 1 || n < 1 || m > n || m > kMaxDim || n > kMaxDim || count < 0 || parts < 1)
    return fail(MUON_ERR_INVALID_ARG, "need 1 <= m <= n <= 2^20, count >= 0, parts >= 1");
  if (count == 0) return MUON_OK;
  if (sumsq == nullptr || x_wide == nullptr || inv_norm == nullptr)
    return fail(MUON_ERR_INVALID_ARG, "NULL buffer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchScope Ls(h, MUON_KERNEL_NORM, s);
  cudaError_t e = muon::launch_norm_finalize(sumsq, parts, count, MUON_NORM_EPS, inv_norm,
                                             h->dev_err, x_wide, n, int64_t(m) * n, m, n, s);
  if (e != cudaSuccess) return cuda_fail(e, "norm launch");
  return MUON_OK;
}

muon_status_t muon_transpose_bf16(muon_handle_t h, int32_t rows, int32_t cols, int32_t count,
                                  const uint16_t* src, uint16_t* dst, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  const muon_group_t g{rows, cols, count, 1.0f};
  st = validate_groups(&g, 1);
  if (st != MUON_OK) return st;
  if (count == 0) return MUON_OK;
  if (src == nullptr || dst == nullptr) return fail(MUON_ERR_INVALID_ARG, "NULL buffer");
  const size_t bytes = size_t(count) * rows * cols * 2;
  const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(dst);
  if (a < b + bytes && b < a + bytes) return fail(MUON_ERR_INVALID_ARG, "src and dst overlap");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchScope Ls(h, MUON_KERNEL_TRANSPOSE, s);
  cudaError_t e = muon::launch_transpose_bf16(rows, cols, count, src, dst, s);
  if (e != cudaSuccess) return cuda_fail(e, "transpose launch");
  return MUON_OK;
}

muon_status_t muon_shard_apply(muon_handle_t h, int64_t n_elems, float* weights_shard,
                               const uint16_t* o_shard, float lr, float wd, float scale,
                               void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (n_elems < 0) return fail(MUON_ERR_INVALID_ARG, "n_elems < 0");
  if (!finite3(lr, wd, scale)) return fail(MUON_ERR_INVALID_ARG, "lr, wd, scale must be finite");
  if (n_elems == 0) return MUON_OK;
  if (weights_shard == nullptr || o_shard == nullptr)
    return fail(MUON_ERR_INVALID_ARG, "NULL buffer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchScope Ls(h, MUON_KERNEL_APPLY, s);
  cudaError_t e = muon::launch_shard_apply(n_elems, weights_shard, o_shard, lr, wd, scale, s);
  if (e != cudaSuccess) return cuda_fail(e, "shard apply launch");
  return MUON_OK;
}

muon_status_t muon_host_alloc(size_t bytes, void** out) {
  if (out == nullptr) return fail(MUON_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (bytes == 0) return fail(MUON_ERR_INVALID_ARG, "bytes must be > 0");
  cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *out = nullptr;
    return fail(MUON_ERR_NOMEM, "page-locked host allocation of %zu bytes failed: %s", bytes,
                cudaGetErrorString(e));
  }
  return MUON_OK;
}

muon_status_t muon_host_free(void* p) {
  if (p == nullptr) return MUON_OK;
  cudaError_t e = cudaFreeHost(p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeHost");
  return MUON_OK;
}

muon_status_t muon_momentum_cast(muon_handle_t h, int32_t rows, int32_t cols, int32_t count,
                                 float* momentum, const float* grad, float mu, uint16_t* x_wide,
                                 float* inv_norm, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  const muon_group_t g{rows, cols, count, 1.0f};
  st = validate_groups(&g, 1);
  if (st != MUON_OK) return st;
  if (!std::isfinite(mu)) return fail(MUON_ERR_INVALID_ARG, "mu must be finite");
  if (count == 0) return MUON_OK;
  if (momentum == nullptr || grad == nullptr || x_wide == nullptr || inv_norm == nullptr)
    return fail(MUON_ERR_INVALID_ARG, "NULL buffer");
  if (!aligned16(momentum) || !aligned16(grad) || !aligned16(x_wide) || !aligned16(inv_norm))
    return fail(MUON_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  const int m = std::min(rows, cols), n = std::max(rows, cols);
  const int tiles = muon::ew_tiles_per_matrix(rows, cols);
  const size_t need = align_up(size_t(count) * tiles * 4, kAlign);
  st = ensure_workspace(h, std::max(need, h->ws_size));
  if (st != MUON_OK) return st;
  float* part = static_cast<float*>(h->ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int64_t done = 0; done < count;) {
    const int take = static_cast<int>(std::min<int64_t>(count - done, 65535));
    const int64_t off = done * int64_t(rows) * cols;
    {
      LaunchScope Ls(h, MUON_KERNEL_MOMENTUM_CAST, s);
      cudaError_t e = muon::launch_momentum_cast(rows, cols, take, momentum + off, grad + off, mu,
                                                 x_wide + done * int64_t(m) * n, n,
                                                 int64_t(m) * n, part + done * tiles, s);
      if (e != cudaSuccess) return cuda_fail(e, "momentum_cast launch");
    }
    done += take;
  }
  LaunchScope Ls(h, MUON_KERNEL_NORM, s);
  cudaError_t e = muon::launch_norm_finalize(part, tiles, count, MUON_NORM_EPS, inv_norm,
                                             h->dev_err, x_wide, n, int64_t(m) * n, m, n, s);
  if (e != cudaSuccess) return cuda_fail(e, "norm launch");
  return MUON_OK;
}

muon_status_t muon_newton_schulz_bf16(muon_handle_t h, int32_t m, int32_t n, int32_t count,
                                      const uint16_t* x, uint16_t* out, const float* inv_norm,
                                      int32_t ns_steps, const float* coeffs, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (m < 1 || n < 1 || m > n || m > kMaxDim || n > kMaxDim || count < 0)
    return fail(MUON_ERR_INVALID_ARG, "need 1 <= m <= n <= %d and count >= 0 (got %d x %d, %d)",
                kMaxDim, m, n, count);
  if ((m % 8) != 0 || (n % 8) != 0)
    return fail(MUON_ERR_INVALID_ARG, "m and n must be multiples of 8 (got %d x %d)", m, n);
  if (ns_steps < 0 || ns_steps > kMaxSteps)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps out of range (%d)", ns_steps);
  Coeffs co{MUON_NS_A, MUON_NS_B, MUON_NS_C};
  if (coeffs != nullptr) {
    co = Coeffs{coeffs[0], coeffs[1], coeffs[2]};
    if (!finite3(co.a, co.b, co.c)) return fail(MUON_ERR_INVALID_ARG, "coefficients not finite");
  }
  const std::vector<Coeffs> sched(ns_steps > 0 ? ns_steps : 1, co);
  if (count == 0) return MUON_OK;
  if (x == nullptr || out == nullptr || inv_norm == nullptr)
    return fail(MUON_ERR_INVALID_ARG, "NULL buffer");
  if (!aligned16(x) || !aligned16(out)) return fail(MUON_ERR_INVALID_ARG, "x/out must be 16-byte aligned");
  const size_t xbytes = size_t(count) * m * n * 2;
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x), ob = reinterpret_cast<uintptr_t>(out);
  if (xb < ob + xbytes && ob < xb + xbytes) return fail(MUON_ERR_INVALID_ARG, "x and out overlap");
  // Scratch: one more X buffer and A, B -- in chunks that fit the cap.
  const size_t pm = align_up(size_t(m) * n * 2, 16) + 2 * align_up(size_t(m) * m * 2, 16);
  int64_t cap = static_cast<int64_t>(h->ws_cap / pm);
  if (cap < 1) cap = 1;
  if (cap > count) cap = count;
  cap = std::min(cap, muon::ns_max_count_per_launch(m, n));
  const size_t need = align_up(size_t(cap) * m * n * 2, kAlign) + 2 * align_up(size_t(cap) * m * m * 2, kAlign);
  st = ensure_workspace(h, need);
  if (st != MUON_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(h->ws);
  uint16_t* other = reinterpret_cast<uint16_t*>(ws);
  uint16_t* A = reinterpret_cast<uint16_t*>(ws + align_up(size_t(cap) * m * n * 2, kAlign));
  uint16_t* B = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(A) +
                                            align_up(size_t(cap) * m * m * 2, kAlign));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t xms = int64_t(m) * n, ams = int64_t(m) * m;
  for (int64_t done = 0; done < count; done += cap) {
    const int take = static_cast<int>(std::min<int64_t>(count - done, cap));
    const muon::BatchView vx{x + done * xms, n, xms}, vo{out + done * xms, n, xms};
    const muon::BatchView vt{other, n, xms}, vA{A, m, ams}, vB{B, m, ams};
    st = run_newton_schulz(h, m, n, take, vx, vo, vt, vA, vB, inv_norm + done, ns_steps,
                           sched.data(), s);
    if (st != MUON_OK) return st;
  }
  return MUON_OK;
}

muon_status_t muon_apply_update(muon_handle_t h, int32_t rows, int32_t cols, int32_t count,
                                float* weights, const uint16_t* o_wide, float lr, float wd,
                                float scale, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  const muon_group_t g{rows, cols, count, scale};
  st = validate_groups(&g, 1);
  if (st != MUON_OK) return st;
  if (!finite3(lr, wd, scale)) return fail(MUON_ERR_INVALID_ARG, "lr, wd, scale must be finite");
  if (count == 0) return MUON_OK;
  if (weights == nullptr || o_wide == nullptr) return fail(MUON_ERR_INVALID_ARG, "NULL buffer");
  if (!aligned16(weights) || !aligned16(o_wide))
    return fail(MUON_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  const int m = std::min(rows, cols), n = std::max(rows, cols);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int64_t done = 0; done < count;) {
    const int take = static_cast<int>(std::min<int64_t>(count - done, 65535));
    LaunchScope Ls(h, MUON_KERNEL_APPLY, s);
    cudaError_t e = muon::launch_apply_update(rows, cols, take, weights + done * int64_t(rows) * cols,
                                              o_wide + done * int64_t(m) * n, n, int64_t(m) * n,
                                              lr, wd, scale, s);
    if (e != cudaSuccess) return cuda_fail(e, "apply launch");
    done += take;
  }
  return MUON_OK;
}

muon_status_t muon_last_device_error(muon_handle_t h, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int flag = 0;
  e = cudaMemcpy(&flag, h->dev_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "error flag read");
  if (flag != 0) {
    cudaMemset(h->dev_err, 0, sizeof(int));
    cudaDeviceSynchronize();
  }
  if (flag & muon::kDevErrTimeout) return fail(MUON_ERR_TIMEOUT, "a device-side wait expired");
  if (flag & muon::kDevErrNonFinite) return fail(MUON_ERR_NONFINITE, "non-finite momentum norm");
  return MUON_OK;
}

muon_status_t muon_adamw_step(muon_handle_t h, int32_t n_tensors, const int64_t* numel,
                              float* const* params, const float* const* grads,
                              float* const* exp_avg, float* const* exp_avg_sq,
                              const muon_adamw_options_t* opts, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (opts == nullptr) return fail(MUON_ERR_INVALID_ARG, "opts is NULL");
  const muon_adamw_options_t& o = *opts;
  if (!finite3(o.lr, o.wd, o.eps) || !finite3(o.beta1, o.beta2, 0.f))
    return fail(MUON_ERR_INVALID_ARG, "AdamW scalars must be finite");
  if (o.beta1 < 0.f || o.beta1 >= 1.f || o.beta2 < 0.f || o.beta2 >= 1.f || o.eps <= 0.f ||
      o.step < 1)
    return fail(MUON_ERR_INVALID_ARG, "need 0 <= beta < 1, eps > 0, step >= 1");
  if (n_tensors < 0) return fail(MUON_ERR_INVALID_ARG, "n_tensors < 0");
  if (n_tensors > 0 && (numel == nullptr || params == nullptr || grads == nullptr ||
                        exp_avg == nullptr || exp_avg_sq == nullptr))
    return fail(MUON_ERR_INVALID_ARG, "NULL array");
  for (int i = 0; i < n_tensors; ++i) {
    if (numel[i] < 0) return fail(MUON_ERR_INVALID_ARG, "tensor %d: numel < 0", i);
    if (numel[i] == 0) continue;
    const void* ptrs[4] = {params[i], grads[i], exp_avg[i], exp_avg_sq[i]};
    for (const void* q : ptrs) {
      if (q == nullptr) return fail(MUON_ERR_INVALID_ARG, "tensor %d: NULL buffer", i);
      if (reinterpret_cast<uintptr_t>(q) & 3u)
        return fail(MUON_ERR_INVALID_ARG, "tensor %d: buffers must be 4-byte aligned", i);
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  muon::AdamwTable table{};
  auto flush = [&]() -> muon_status_t {
    if (table.count == 0) return MUON_OK;
    LaunchScope Ls(h, MUON_KERNEL_ADAMW, s);
    cudaError_t e = muon::launch_adamw(table, o.lr, o.beta1, o.beta2, o.eps, o.wd, o.step, s);
    table = muon::AdamwTable{};
    if (e != cudaSuccess) return cuda_fail(e, "AdamW launch");
    return MUON_OK;
  };
  for (int i = 0; i < n_tensors; ++i) {
    if (numel[i] == 0) continue;
    const int c = table.count;
    table.p[c] = params[i];
    table.g[c] = grads[i];
    table.m[c] = exp_avg[i];
    table.v[c] = exp_avg_sq[i];
    table.n[c] = numel[i];
    table.block_start[c + 1] = table.block_start[c] + muon::adamw_blocks(numel[i]);
    table.count = c + 1;
    if (table.count == muon::kAdamwMaxTensors || table.block_start[table.count] > (int64_t(1) << 30)) {
      st = flush();
      if (st != MUON_OK) return st;
    }
  }
  return flush();
}

muon_status_t muon_selftest_bounded_wait(muon_handle_t h, int32_t limit_ms, void* stream) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (limit_ms < 1 || limit_ms > 2000)
    return fail(MUON_ERR_INVALID_ARG, "limit_ms must be in 1..2000 (got %d)", limit_ms);
  cudaError_t e = muon::launch_bounded_wait_selftest(
      h->dev_err, static_cast<uint64_t>(limit_ms) * 1000000ull, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return MUON_OK;
}

muon_status_t muon_set_kernel_timing(muon_handle_t h, int32_t enable) {
  if (h == nullptr) return fail(MUON_ERR_INVALID_ARG, "handle is NULL");
  h->timing = enable != 0;
  return MUON_OK;
}

muon_status_t muon_kernel_stats(muon_handle_t h, muon_kernel_stats_t* out) {
  muon_status_t st = check_handle(h);
  if (st != MUON_OK) return st;
  if (out == nullptr) return fail(MUON_ERR_INVALID_ARG, "out is NULL");
  if (!h->pending.empty()) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    for (auto& p : h->pending) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) h->stats.total_ms[p.kind] += ms;
      h->free_events.push_back(p.a);
      h->free_events.push_back(p.b);
    }
    h->pending.clear();
  }
  *out = h->stats;
  return MUON_OK;
}

muon_status_t muon_reset_kernel_stats(muon_handle_t h) {
  muon_kernel_stats_t tmp;
  muon_status_t st = muon_kernel_stats(h, &tmp);  // drains pending events
  if (st != MUON_OK) return st;
  h->stats = muon_kernel_stats_t{};
  return MUON_OK;
}

}  // extern "C"
