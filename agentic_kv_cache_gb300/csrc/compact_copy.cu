// compact_copy: the copy pass of sequence compaction.
//
// [AKV-blog] "Dilemma 2: Memory Fragmentation in Paged Pools": once drops
// leave a sequence's pages sparsely used, a compacting allocator copies the
// surviving blocks into contiguous physical spans.  Here the surviving
// (visible) tokens are copied, in logical order, into fresh dense pages; a
// token with a pending shift has its key rotated by R(delta * theta_j) on the
// way (the same float32 arithmetic and float64-built angle table as
// repos_rotate, so compaction and repositioning cost one pass), its value is
// copied unchanged.
//
// Work: the copy-run list (source K / V page and first slot, destination K /
// V page and first slot, row count, shift index or -1) times every layer and
// kv head.  HBM-bound streaming: a CTA takes one (layer, run) unit and moves
// 16-byte vectors with several independent loads in flight before stores;
// keys and values go in two launches so each keeps its register count low.
#include <cuda_bf16.h>

#include "akv_internal.h"
#include "rope_rot.cuh"

namespace akv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// kPart 0: the key rows (rotated or copied); 1: the value rows (copied).  Two
// launches keep each one's registers low, so more warps keep loads in flight.
// Within a (layer, run) unit the (head, row, vector) items are spread flat over
// the CTA's threads, so short runs (a run ends at a page boundary on either
// side) still keep every thread busy; each thread issues its loads for
// kInFlight items before any store.
template <int D, bool kHalf, int kPart>
__global__ void __launch_bounds__(kThreads, kPart == 1 ? 4 : 3) compact_copy_kernel(uint4* __restrict__ kpool, uint4* __restrict__ vpool,
                                                               const CopyRun* __restrict__ runs,
                                                               const float2* __restrict__ cs, int n_runs, int n_layers,
                                                               int heads, int page, int64_t n_pages, int vv_shift,
                                                               DevErr* err) {
  constexpr int VK = D / 8;                  // 16-byte vectors per K row
  constexpr int W = kHalf ? VK / 2 : VK;     // K work items per row: vectors, or (v, v + VK/2) pairs
  constexpr int kInFlight = kPart == 1 ? 8 : 4;
  const int VV = 1 << vv_shift;              // vectors per V row
  const int64_t kpage = int64_t(heads) * page * VK, vpage = int64_t(heads) * page * VV;
  const int64_t units = int64_t(n_layers) * n_runs;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int r = int(u % n_runs);
    const int64_t layer = u / n_runs;
    const CopyRun cr = runs[r];
#ifdef AKV_CHECKED
    // pages exist, both slot ranges lie inside one page, the shift row is valid or -1
    if (!(cr.src_k >= 0 && cr.src_k < n_pages && cr.src_v >= 0 && cr.src_v < n_pages && cr.dst_k >= 0 &&
          cr.dst_k < n_pages && cr.dst_v >= 0 && cr.dst_v < n_pages && cr.n > 0 && cr.src_lo >= 0 &&
          cr.dst_lo >= 0 && cr.src_lo + cr.n <= page && cr.dst_lo + cr.n <= page && cr.didx >= -1)) {
      if (threadIdx.x == 0) report_device_error(err, 3 + kPart, r, int(layer));
      continue;  // the whole CTA skips this unit
    }
#else
    (void)err;
#endif
    // ---- K rows: rotated when the run carries a shift, else copied.
    if constexpr (kPart == 0) {
      const uint4* src = kpool + (layer * n_pages + cr.src_k) * kpage + cr.src_lo * VK;
      uint4* dst = kpool + (layer * n_pages + cr.dst_k) * kpage + cr.dst_lo * VK;
      const float2* cs_row = cr.didx >= 0 ? cs + int64_t(cr.didx) * (D / 2) : nullptr;
      const int per_head = cr.n * W, items = heads * per_head;
#pragma unroll 1
      for (int i0 = 0; i0 < items; i0 += kInFlight * kThreads) {
        uint4 x[kInFlight], y[kInFlight];
        int off[kInFlight], vv[kInFlight];
#pragma unroll
        for (int k = 0; k < kInFlight; ++k) {
          const int it = i0 + k * kThreads + int(threadIdx.x);
          off[k] = -1;
          if (it < items) {
            const int h = it / per_head, rem = it - h * per_head, row = rem / W, v = rem - row * W;
            off[k] = h * page * VK + row * VK + v;
            vv[k] = v;
            x[k] = __ldcs(src + off[k]);
            if (kHalf) y[k] = __ldcs(src + off[k] + VK / 2);
          }
        }
#pragma unroll
        for (int k = 0; k < kInFlight; ++k) {
          if (off[k] < 0) continue;
          uint4* d = dst + off[k];
          const int v = vv[k];
          if (!cs_row) {
            __stcs(d, x[k]);
            if (kHalf) __stcs(d + VK / 2, y[k]);
          } else if constexpr (!kHalf) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(cs_row + 4 * v));
            const float4 b = __ldg(reinterpret_cast<const float4*>(cs_row + 4 * v + 2));
            __stcs(d, make_uint4(pack_rot(rot2(x[k].x, a.x, a.y)), pack_rot(rot2(x[k].y, a.z, a.w)),
                                 pack_rot(rot2(x[k].z, b.x, b.y)), pack_rot(rot2(x[k].w, b.z, b.w))));
          } else {
            const float4* c4 = reinterpret_cast<const float4*>(cs_row + 8 * v);
            const float4 c01 = __ldg(c4), c23 = __ldg(c4 + 1), c45 = __ldg(c4 + 2), c67 = __ldg(c4 + 3);
            float2 ya[4], yb[4];
            rot_halves(x[k].x, y[k].x, c01.x, c01.y, c01.z, c01.w, ya[0], yb[0]);
            rot_halves(x[k].y, y[k].y, c23.x, c23.y, c23.z, c23.w, ya[1], yb[1]);
            rot_halves(x[k].z, y[k].z, c45.x, c45.y, c45.z, c45.w, ya[2], yb[2]);
            rot_halves(x[k].w, y[k].w, c67.x, c67.y, c67.z, c67.w, ya[3], yb[3]);
            __stcs(d, make_uint4(pack_rot(ya[0]), pack_rot(ya[1]), pack_rot(ya[2]), pack_rot(ya[3])));
            __stcs(d + VK / 2, make_uint4(pack_rot(yb[0]), pack_rot(yb[1]), pack_rot(yb[2]), pack_rot(yb[3])));
          }
        }
      }
    }
    // ---- V rows: copied
    if constexpr (kPart == 1) {
      const uint4* src = vpool + (layer * n_pages + cr.src_v) * vpage + int64_t(cr.src_lo) * VV;
      uint4* dst = vpool + (layer * n_pages + cr.dst_v) * vpage + int64_t(cr.dst_lo) * VV;
      const int per_head = cr.n << vv_shift, items = heads * per_head;
#pragma unroll 1
      for (int i0 = 0; i0 < items; i0 += kInFlight * kThreads) {
        uint4 x[kInFlight];
        int off[kInFlight];
#pragma unroll
        for (int k = 0; k < kInFlight; ++k) {
          const int it = i0 + k * kThreads + int(threadIdx.x);
          off[k] = -1;
          if (it < items) {
            const int h = it / per_head, rem = it - h * per_head;
            off[k] = h * page * VV + rem;  // a head's rows are contiguous from the run's first slot
            x[k] = __ldcs(src + off[k]);
          }
        }
#pragma unroll
        for (int k = 0; k < kInFlight; ++k)
          if (off[k] >= 0) __stcs(dst + off[k], x[k]);
      }
    }
  }
}

template <int D, bool kHalf>
cudaError_t launch_variant(void* kpool, void* vpool, const CopyRun* runs, const float2* cs, int n_runs, int n_layers,
                           int heads, int page, int64_t n_pages, int dv, int n_sm, DevErr* err, cudaStream_t st) {
  int vv_shift = 0;
  while ((8 << vv_shift) < dv) ++vv_shift;
  if ((8 << vv_shift) != dv) return cudaErrorInvalidValue;  // d_v must be 8 x a power of two
  const int64_t units = int64_t(n_layers) * n_runs;
  const int grid = int(units < int64_t(n_sm) * 8 ? units : int64_t(n_sm) * 8);
  compact_copy_kernel<D, kHalf, 0><<<grid, kThreads, 0, st>>>(static_cast<uint4*>(kpool), static_cast<uint4*>(vpool),
                                                              runs, cs, n_runs, n_layers, heads, page, n_pages, vv_shift, err);
  compact_copy_kernel<D, kHalf, 1><<<grid, kThreads, 0, st>>>(static_cast<uint4*>(kpool), static_cast<uint4*>(vpool),
                                                              runs, cs, n_runs, n_layers, heads, page, n_pages, vv_shift, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compact_copy(void* kpool, void* vpool, const CopyRun* runs, const float2* cs, int n_runs,
                                int n_layers, int heads, int d_rot, int d_v, int page, int64_t n_pages, bool half,
                                int n_sm, DevErr* err, cudaStream_t st) {
  if (n_runs <= 0) return cudaSuccess;
  if (d_v % 8 != 0) return cudaErrorInvalidValue;
  if (d_rot == 64)
    return half ? launch_variant<64, true>(kpool, vpool, runs, cs, n_runs, n_layers, heads, page, n_pages, d_v, n_sm, err, st)
                : launch_variant<64, false>(kpool, vpool, runs, cs, n_runs, n_layers, heads, page, n_pages, d_v, n_sm, err, st);
  if (d_rot == 128)
    return half ? launch_variant<128, true>(kpool, vpool, runs, cs, n_runs, n_layers, heads, page, n_pages, d_v, n_sm, err, st)
                : launch_variant<128, false>(kpool, vpool, runs, cs, n_runs, n_layers, heads, page, n_pages, d_v, n_sm, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace akv
