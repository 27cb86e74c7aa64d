// repos_rotate: materialise pending repositions of cached keys.
//
// [AKV-blog] section 2 "The Repos Primitive and Rotary Position Embeddings":
// RoPE rotations form SO(2), R(a) R(b) = R(a + b), so a key already rotated
// for position p is moved to p + delta by one more rotation of the stored
// vector, k' = R(delta * theta_j) k on every pair j; no hidden state is needed.
// [Leyline] "Method": under MLA only K_pe is rotated (the caller passes the
// K_pe pool), and several directives compose into one shift per token.
//
// Work: the run list (src page, dst page, rows [lo, hi), shift index) times
// every layer and kv head.  dst == src rotates in place; dst != src is the
// copy-on-write of a shared page ([AKV-notes] section 3 "Cache Management").
//
// A float32-output debug mode of the same kernel (launch_repos_rotate_f32)
// writes the unrounded rotation of given rows to a dense array instead of the
// pool, so the rotation arithmetic can be checked against float64 directly.
//
// Design: HBM-bound streaming (0.75 FLOP/B).  A CTA takes one (layer, run)
// unit: H * (hi - lo) rows of d_rot bf16, i.e. up to 32 KiB for a full page of
// 8 heads x 16 slots x 128 dims, contiguous in the pool.  Every thread moves
// 16-byte vectors (8 bf16 = 4 interleaved pairs), issuing four independent
// loads before any store so enough bytes are in flight to saturate HBM3e.
// (cos, sin)(delta * theta_j) comes from a per-shift table that the host
// evaluates in float64 and rounds to float32 (a float32 delta * theta would
// be off by ~1e-2 rad at |delta| = 64K); the rotation itself is float32 with
// one round-to-nearest-even to bf16.
#include <cuda_bf16.h>

#include "akv_internal.h"
#include "rope_rot.cuh"

namespace akv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

#ifdef AKV_CHECKED
// A run descriptor names existing pages and a non-empty row range of one page.
__device__ __forceinline__ bool run_ok(const RunDesc& rd, int page, int64_t n_pages) {
  const int lo = rd.lohi & 0xffff, hi = rd.lohi >> 16;
  return rd.src >= 0 && rd.src < n_pages && rd.dst >= 0 && rd.dst < n_pages && lo < hi && hi <= page &&
         rd.didx >= 0;
}
#endif

// Where a rotated 16-byte vector goes: back into the pool as bf16 (the
// product path), or, in the float32 debug mode, into a dense float32 array
// [L][rows][H][D] so the rotation can be checked before rounding.
struct F32Out {
  float* out;
  const int32_t* row_off;  // first output row of each run
  int64_t total_rows;
};

template <int D, bool F32>
__global__ void __launch_bounds__(kThreads) repos_interleaved_kernel(uint4* __restrict__ pool,
                                                                   const RunDesc* __restrict__ runs,
                                                                   const float2* __restrict__ cs, int n_runs,
                                                                   int n_layers, int heads, int page,
                                                                   int64_t n_pages, F32Out f32, DevErr* err) {
  constexpr int V = D / 8;  // vectors per row
  const int64_t page_vecs = int64_t(heads) * page * V;
  const int64_t layer_vecs = page_vecs * n_pages;
  const int64_t units = int64_t(n_layers) * n_runs;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int r = int(u % n_runs);
    const int64_t layer = u / n_runs;
    const RunDesc rd = runs[r];
    const int lo = rd.lohi & 0xffff, n = (rd.lohi >> 16) - lo;
#ifdef AKV_CHECKED
    if (!run_ok(rd, page, n_pages)) {  // the whole CTA skips this unit
      if (threadIdx.x == 0) report_device_error(err, 1, r, int(layer));
      continue;
    }
#else
    (void)err;
#endif
    const float2* cs_row = cs + int64_t(rd.didx) * (D / 2);
    const uint4* src = pool + layer * layer_vecs + rd.src * page_vecs;
    uint4* dst = pool + layer * layer_vecs + rd.dst * page_vecs;
    const int per_head = n * V;
    const int total = heads * per_head;
    for (int base = 0; base < total; base += kThreads * kUnroll) {
      uint4 x[kUnroll];
      int idx[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        idx[k] = base + k * kThreads + int(threadIdx.x);
        if (idx[k] < total) {
          const int h = idx[k] / per_head;
          x[k] = __ldcs(src + (h * page + lo) * V + (idx[k] - h * per_head));
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (idx[k] >= total) continue;
        const int h = idx[k] / per_head;
        const int rem = idx[k] - h * per_head;  // (slot - lo) * V + v
        const int v = rem % V;
        const float4 a = __ldg(reinterpret_cast<const float4*>(cs_row + 4 * v));
        const float4 b = __ldg(reinterpret_cast<const float4*>(cs_row + 4 * v + 2));
        const float2 y0 = rot2(x[k].x, a.x, a.y), y1 = rot2(x[k].y, a.z, a.w);
        const float2 y2 = rot2(x[k].z, b.x, b.y), y3 = rot2(x[k].w, b.z, b.w);
        if constexpr (F32) {
          const int64_t row = layer * f32.total_rows + f32.row_off[r] + rem / V;
          float4* o = reinterpret_cast<float4*>(f32.out + (row * heads + h) * D + v * 8);
          o[0] = make_float4(y0.x, y0.y, y1.x, y1.y);
          o[1] = make_float4(y2.x, y2.y, y3.x, y3.y);
        } else {
          __stcs(dst + (h * page + lo) * V + rem, make_uint4(pack_rot(y0), pack_rot(y1), pack_rot(y2), pack_rot(y3)));
        }
      }
    }
  }
}

template <int D, bool F32>
__global__ void __launch_bounds__(kThreads) repos_half_kernel(uint4* __restrict__ pool,
                                                            const RunDesc* __restrict__ runs,
                                                            const float2* __restrict__ cs, int n_runs, int n_layers,
                                                            int heads, int page, int64_t n_pages, F32Out f32,
                                                            DevErr* err) {
  constexpr int V = D / 8;
  constexpr int HV = V / 2;  // vector pairs per row: (v, v + V/2)
  const int64_t page_vecs = int64_t(heads) * page * V;
  const int64_t layer_vecs = page_vecs * n_pages;
  const int64_t units = int64_t(n_layers) * n_runs;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int r = int(u % n_runs);
    const int64_t layer = u / n_runs;
    const RunDesc rd = runs[r];
    const int lo = rd.lohi & 0xffff, n = (rd.lohi >> 16) - lo;
#ifdef AKV_CHECKED
    if (!run_ok(rd, page, n_pages)) {  // the whole CTA skips this unit
      if (threadIdx.x == 0) report_device_error(err, 1, r, int(layer));
      continue;
    }
#else
    (void)err;
#endif
    const float2* cs_row = cs + int64_t(rd.didx) * (D / 2);
    const uint4* src = pool + layer * layer_vecs + rd.src * page_vecs;
    uint4* dst = pool + layer * layer_vecs + rd.dst * page_vecs;
    const int per_head = n * HV;
    const int total = heads * per_head;
    for (int i = int(threadIdx.x); i < total; i += kThreads) {
      const int h = i / per_head;
      const int rem = i - h * per_head;
      const int row = rem / HV, v = rem % HV;
      const int off = (h * page + lo + row) * V + v;
      const uint4 a = __ldcs(src + off), b = __ldcs(src + off + HV);
      const float4* c4 = reinterpret_cast<const float4*>(cs_row + 8 * v);
      const float4 c01 = __ldg(c4), c23 = __ldg(c4 + 1), c45 = __ldg(c4 + 2), c67 = __ldg(c4 + 3);
      float2 ya[4], yb[4];
      rot_halves(a.x, b.x, c01.x, c01.y, c01.z, c01.w, ya[0], yb[0]);
      rot_halves(a.y, b.y, c23.x, c23.y, c23.z, c23.w, ya[1], yb[1]);
      rot_halves(a.z, b.z, c45.x, c45.y, c45.z, c45.w, ya[2], yb[2]);
      rot_halves(a.w, b.w, c67.x, c67.y, c67.z, c67.w, ya[3], yb[3]);
      if constexpr (F32) {
        const int64_t orow = layer * f32.total_rows + f32.row_off[r] + row;
        float* o = f32.out + (orow * heads + h) * D;
        float4* oa = reinterpret_cast<float4*>(o + v * 8);
        float4* ob = reinterpret_cast<float4*>(o + D / 2 + v * 8);
        oa[0] = make_float4(ya[0].x, ya[0].y, ya[1].x, ya[1].y);
        oa[1] = make_float4(ya[2].x, ya[2].y, ya[3].x, ya[3].y);
        ob[0] = make_float4(yb[0].x, yb[0].y, yb[1].x, yb[1].y);
        ob[1] = make_float4(yb[2].x, yb[2].y, yb[3].x, yb[3].y);
      } else {
        __stcs(dst + off, make_uint4(pack_rot(ya[0]), pack_rot(ya[1]), pack_rot(ya[2]), pack_rot(ya[3])));
        __stcs(dst + off + HV, make_uint4(pack_rot(yb[0]), pack_rot(yb[1]), pack_rot(yb[2]), pack_rot(yb[3])));
      }
    }
  }
}

template <bool F32>
cudaError_t launch(void* kpool, const RunDesc* runs, const float2* cs, int n_runs, int n_layers, int heads,
                   int d_rot, int page, int64_t n_pages, bool half_layout, F32Out f32, DevErr* err, cudaStream_t st) {
  if (n_runs <= 0) return cudaSuccess;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t units = int64_t(n_layers) * n_runs;
  const unsigned blocks = unsigned(std::min<int64_t>(units, int64_t(sms) * 8));
  uint4* p = static_cast<uint4*>(kpool);
#define AKV_REPOS_CASE(DIM)                                                                                    \
  case DIM:                                                                                                    \
    if (half_layout)                                                                                           \
      repos_half_kernel<DIM, F32><<<blocks, kThreads, 0, st>>>(p, runs, cs, n_runs, n_layers, heads, page,     \
                                                               n_pages, f32, err);                             \
    else                                                                                                       \
      repos_interleaved_kernel<DIM, F32><<<blocks, kThreads, 0, st>>>(p, runs, cs, n_runs, n_layers, heads,    \
                                                                      page, n_pages, f32, err);               \
    break;
  switch (d_rot) {
    AKV_REPOS_CASE(16)
    AKV_REPOS_CASE(32)
    AKV_REPOS_CASE(64)
    AKV_REPOS_CASE(128)
    AKV_REPOS_CASE(256)
    default:
      return cudaErrorInvalidValue;
  }
#undef AKV_REPOS_CASE
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_repos_rotate(void* kpool, const RunDesc* runs, const float2* cs, int n_runs, int n_layers,
                                int heads, int d_rot, int page, int64_t n_pages, bool half_layout, DevErr* err,
                                cudaStream_t st) {
  return launch<false>(kpool, runs, cs, n_runs, n_layers, heads, d_rot, page, n_pages, half_layout,
                       F32Out{nullptr, nullptr, 0}, err, st);
}

cudaError_t launch_repos_rotate_f32(const void* kpool, const RunDesc* runs, const float2* cs, const int32_t* row_off,
                                    int64_t total_rows, float* out, int n_runs, int n_layers, int heads, int d_rot,
                                    int page, int64_t n_pages, bool half_layout, DevErr* err, cudaStream_t st) {
  return launch<true>(const_cast<void*>(kpool), runs, cs, n_runs, n_layers, heads, d_rot, page, n_pages,
                      half_layout, F32Out{out, row_off, total_rows}, err, st);
}

}  // namespace akv
