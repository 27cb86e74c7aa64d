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
#include <unordered_map>
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

  const int half = d_rot / 2;
  // A list whose descriptors alone exceed the array is refused before any work.
  const size_t runs_bytes = (size_t(n_runs) * sizeof(akv::RunDesc) + 255) & ~size_t(255);
  if (runs_bytes > kScratchBytes) return AKV_ERR_RANGE;

  // The run list and the table are copied from temporary host memory, which a
  // graph node would read only at replay, after this call has freed it.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
    cudaGetLastError();
    return AKV_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return AKV_ERR_ARG;

  // Run descriptors and the distinct shifts, checked against the pool.  The
  // table grows with the shifts; a list that cannot fit stops at the shift
  // that overflows the array.
  std::vector<akv::RunDesc> desc(static_cast<size_t>(n_runs));
  std::vector<int32_t> deltas;
  std::unordered_map<int32_t, int32_t> delta_index;
  for (int32_t r = 0; r < n_runs; ++r) {
    const int32_t src = runs[5 * r], dst = runs[5 * r + 1], lo = runs[5 * r + 2], hi = runs[5 * r + 3];
    const int32_t d = runs[5 * r + 4];
    if (src < 0 || src >= n_pages || dst < 0 || dst >= n_pages || lo < 0 || lo >= hi || hi > page_size)
      return AKV_ERR_RANGE;
    auto it = delta_index.find(d);
    if (it == delta_index.end()) {
      if (runs_bytes + (deltas.size() + 1) * half * sizeof(float2) > kScratchBytes) return AKV_ERR_RANGE;
      it = delta_index.emplace(d, int32_t(deltas.size())).first;
      deltas.push_back(d);
    }
    desc[size_t(r)] = akv::RunDesc{src, dst, lo | (hi << 16), it->second};
  }

  // Runs of one launch execute concurrently, so the rows they write must be
  // disjoint: no two runs may write the same (page, row), and a copy (src !=
  // dst) may not read rows another copy writes.  The one overlap allowed is
  // the one a flush of two sequences sharing a page produces: a copy reading
  // rows that an in-place run (src == dst) rotates.  Such copies run in a
  // first launch, the in-place runs in a second.  Rows of a page are at most
  // 128, so each page keeps two 64-bit row masks.
  struct Rows {
    uint64_t w[2] = {0, 0};    // rows written by any run
    uint64_t cw[2] = {0, 0};   // rows written by copies
    uint64_t ip[2] = {0, 0};   // rows rotated in place
  };
  auto mask_of = [](int lo, int hi, uint64_t m[2]) {
    for (int k = 0; k < 2; ++k) {
      const int a = std::max(lo, 64 * k), b = std::min(hi, 64 * k + 64);
      m[k] = a < b ? ((b - a == 64 ? ~uint64_t(0) : ((uint64_t(1) << (b - a)) - 1)) << (a - 64 * k)) : 0;
    }
  };
  std::unordered_map<int32_t, Rows> pages;
  pages.reserve(size_t(n_runs) * 2);
  for (const akv::RunDesc& r : desc) {
    uint64_t m[2];
    mask_of(r.lohi & 0xffff, r.lohi >> 16, m);
    Rows& p = pages[r.dst];
    if ((p.w[0] & m[0]) | (p.w[1] & m[1])) return AKV_ERR_ARG;  // two runs write one row
    p.w[0] |= m[0];
    p.w[1] |= m[1];
    uint64_t* kind = r.src != r.dst ? p.cw : p.ip;
    kind[0] |= m[0];
    kind[1] |= m[1];
  }
  bool conflict = false;
  for (const akv::RunDesc& r : desc) {
    if (r.src == r.dst) continue;
    auto it = pages.find(r.src);
    if (it == pages.end()) continue;
    uint64_t m[2];
    mask_of(r.lohi & 0xffff, r.lohi >> 16, m);
    if ((it->second.cw[0] & m[0]) | (it->second.cw[1] & m[1])) return AKV_ERR_ARG;  // reads another copy's rows
    if ((it->second.ip[0] & m[0]) | (it->second.ip[1] & m[1])) conflict = true;
  }
  std::stable_partition(desc.begin(), desc.end(), [](const akv::RunDesc& r) { return r.src != r.dst; });
  int32_t n_copy = 0;
  while (n_copy < n_runs && desc[size_t(n_copy)].src != desc[size_t(n_copy)].dst) ++n_copy;
  const size_t cs_bytes = deltas.size() * half * sizeof(float2);

  // (cos, sin)(delta * theta_j), evaluated in float64, stored as float32.
  std::vector<float2> cs(deltas.size() * half);
  for (size_t k = 0; k < deltas.size(); ++k)
    for (int j = 0; j < half; ++j) {
      const double a = double(deltas[k]) * std::pow(rope_base, -2.0 * j / d_rot);
      cs[k * half + j] = make_float2(float(std::cos(a)), float(std::sin(a)));
    }

  void* base = nullptr;
  if (akv_status s = scratch_address(&base); s != AKV_OK) return s;
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
                               rope_layout == AKV_ROPE_HALF, nullptr, st) != cudaSuccess)
    return AKV_ERR_CUDA;
  if (conflict && akv::launch_repos_rotate(k_pool, dev_runs + n_copy, dev_cs, n_runs - n_copy, n_layers, n_kv_heads,
                                           d_rot, page_size, n_pages, rope_layout == AKV_ROPE_HALF, nullptr,
                                           st) != cudaSuccess)
    return AKV_ERR_CUDA;
  return AKV_OK;
}
