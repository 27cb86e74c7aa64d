// akv_repos_rotate_noalloc: the repos_rotate kernel for callers that cannot
// allocate device memory.
//
// Who needs it: a serving process that reserves nearly all of HBM for its KV
// pool up front has no room left for further cudaMalloc calls, and a caller
// on a latency-critical path must avoid cudaMalloc / cudaFree because they can
// synchronise the whole device.  The context-based path (akv_create +
// akv_flush) allocates its descriptor buffers on first use; this entry point
// does not allocate at all: the run list and the (cos, sin) table go into a
// fixed-size array in the library's own device memory (a file-scope
// __device__ array that every GPU loading the library keeps until exit).
//
// The array is shared by every call: each call overwrites the part it uses
// (nothing in it has to start at zero), so calls that overlap on the GPU --
// for example on two streams without ordering -- race on it.  Calls on one
// stream are ordered and safe.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address once (cudaGetSymbolAddress) and caches it; make that
// first call before any stream capture.
#include <cmath>
#include <cstdint>
#include <mutex>
#include <algorithm>
#include <vector>

#include "../../include/akv.h"
#include "akv_internal.h"

namespace {

constexpr size_t kScratchBytes = 256 * 1024;  // run descriptors + (cos, sin) table
constexpr int kMaxDevices = 64;

// The scratch array.  In host code its name is only a host-side stand-in:
// kernels receive the device address obtained below.
static __device__ __align__(256) unsigned char g_repos_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
akv_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return AKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_repos_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return AKV_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return AKV_OK;
}

}  // namespace

extern "C" AKV_API akv_status akv_repos_rotate_noalloc(void* k_pool, int32_t n_layers, int32_t n_kv_heads,
                                                       int32_t page_size, int32_t n_pages, int32_t d_rot,
                                                       int32_t rope_layout, double rope_base, const int32_t* runs,
                                                       int32_t n_runs, void* stream) {
  if (n_runs < 0 || (n_runs > 0 && (!runs || !k_pool))) return AKV_ERR_ARG;
  if (n_layers <= 0 || n_kv_heads <= 0 || n_pages <= 0 || !(rope_base > 0.0)) return AKV_ERR_ARG;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return AKV_ERR_ARG;
  if (d_rot != 16 && d_rot != 32 && d_rot != 64 && d_rot != 128 && d_rot != 256) return AKV_ERR_ARG;
  if (rope_layout != AKV_ROPE_INTERLEAVED && rope_layout != AKV_ROPE_HALF) return AKV_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(k_pool) % 16) return AKV_ERR_ARG;
  if (n_runs == 0) return AKV_OK;

  // Run descriptors and the distinct shifts, checked against the pool.
  std::vector<akv::RunDesc> desc(static_cast<size_t>(n_runs));
  std::vector<int32_t> deltas;
  for (int32_t r = 0; r < n_runs; ++r) {
    const int32_t src = runs[5 * r], dst = runs[5 * r + 1], lo = runs[5 * r + 2], hi = runs[5 * r + 3];
    const int32_t d = runs[5 * r + 4];
    if (src < 0 || src >= n_pages || dst < 0 || dst >= n_pages || lo < 0 || lo >= hi || hi > page_size)
      return AKV_ERR_RANGE;
    int32_t di = -1;
    for (size_t k = 0; k < deltas.size(); ++k)
      if (deltas[k] == d) {
        di = int32_t(k);
        break;
      }
    if (di < 0) {
      di = int32_t(deltas.size());
      deltas.push_back(d);
    }
    desc[size_t(r)] = akv::RunDesc{src, dst, lo | (hi << 16), di};
  }
  // Runs of one launch execute concurrently: when a page is both the source
  // of a copy (src != dst) and rotated in place by another run (as a flush of
  // two sequences sharing it lists them), the copies run in a first launch.
  std::stable_partition(desc.begin(), desc.end(), [](const akv::RunDesc& r) { return r.src != r.dst; });
  int32_t n_copy = 0;
  while (n_copy < n_runs && desc[size_t(n_copy)].src != desc[size_t(n_copy)].dst) ++n_copy;
  bool conflict = false;
  if (n_copy > 0 && n_copy < n_runs) {
    std::vector<int32_t> srcs;
    for (int32_t r = 0; r < n_copy; ++r) srcs.push_back(desc[size_t(r)].src);
    std::sort(srcs.begin(), srcs.end());
    for (int32_t r = n_copy; r < n_runs && !conflict; ++r)
      conflict = std::binary_search(srcs.begin(), srcs.end(), desc[size_t(r)].dst);
  }
  const int half = d_rot / 2;
  const size_t runs_bytes = (desc.size() * sizeof(akv::RunDesc) + 255) & ~size_t(255);
  const size_t cs_bytes = deltas.size() * half * sizeof(float2);
  if (runs_bytes + cs_bytes > kScratchBytes) return AKV_ERR_RANGE;  // beyond the fixed scratch size

  // (cos, sin)(delta * theta_j), evaluated in float64, stored as float32.
  std::vector<float2> cs(deltas.size() * half);
  for (size_t k = 0; k < deltas.size(); ++k)
    for (int j = 0; j < half; ++j) {
      const double a = double(deltas[k]) * std::pow(rope_base, -2.0 * j / d_rot);
      cs[k * half + j] = make_float2(float(std::cos(a)), float(std::sin(a)));
    }

  void* base = nullptr;
  if (akv_status s = scratch_address(&base); s != AKV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* dev_runs = static_cast<akv::RunDesc*>(base);
  auto* dev_cs = reinterpret_cast<float2*>(static_cast<unsigned char*>(base) + runs_bytes);
  if (cudaMemcpyAsync(dev_runs, desc.data(), desc.size() * sizeof(akv::RunDesc), cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(dev_cs, cs.data(), cs_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return AKV_ERR_CUDA;
  }
  const int32_t first_n = conflict ? n_copy : n_runs;
  if (akv::launch_repos_rotate(k_pool, dev_runs, dev_cs, first_n, n_layers, n_kv_heads, d_rot, page_size, n_pages,
                               rope_layout == AKV_ROPE_HALF, st) != cudaSuccess)
    return AKV_ERR_CUDA;
  if (conflict && akv::launch_repos_rotate(k_pool, dev_runs + n_copy, dev_cs, n_runs - n_copy, n_layers, n_kv_heads,
                                           d_rot, page_size, n_pages, rope_layout == AKV_ROPE_HALF, st) != cudaSuccess)
    return AKV_ERR_CUDA;
  return AKV_OK;
}
