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

namespace akv {
namespace {

__device__ __forceinline__ uint32_t rot_pair(uint32_t xy, float c, float s) {
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&xy);
  const float2 f = __bfloat1622float2(b);
  const float y0 = fmaf(c, f.x, -s * f.y);
  const float y1 = fmaf(s, f.x, c * f.y);
  __nv_bfloat162 r = __floats2bfloat162_rn(y0, y1);
  return *reinterpret_cast<uint32_t*>(&r);
}

// Interleaved pairs (2j, 2j+1): one 16-byte vector holds pairs 4v .. 4v+3.
__device__ __forceinline__ uint4 rot_vec_interleaved(uint4 x, const float2* __restrict__ cs_row, int v) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(cs_row + 4 * v));
  const float4 b = __ldg(reinterpret_cast<const float4*>(cs_row + 4 * v + 2));
  x.x = rot_pair(x.x, a.x, a.y);
  x.y = rot_pair(x.y, a.z, a.w);
  x.z = rot_pair(x.z, b.x, b.y);
  x.w = rot_pair(x.w, b.z, b.w);
  return x;
}

__device__ __forceinline__ void rot_halves(uint32_t& a, uint32_t& b, float c0, float s0, float c1, float s1) {
  // a holds first-half elements e, e+1; b the matching second-half elements.
  __nv_bfloat162 ab = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 bb = *reinterpret_cast<__nv_bfloat162*>(&b);
  const float2 fa = __bfloat1622float2(ab), fb = __bfloat1622float2(bb);
  __nv_bfloat162 ra = __floats2bfloat162_rn(fmaf(c0, fa.x, -s0 * fb.x), fmaf(c1, fa.y, -s1 * fb.y));
  __nv_bfloat162 rb = __floats2bfloat162_rn(fmaf(s0, fa.x, c0 * fb.x), fmaf(s1, fa.y, c1 * fb.y));
  a = *reinterpret_cast<uint32_t*>(&ra);
  b = *reinterpret_cast<uint32_t*>(&rb);
}

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int D>
__global__ void __launch_bounds__(kThreads) repos_interleaved_kernel(uint4* __restrict__ pool,
                                                                   const RunDesc* __restrict__ runs,
                                                                   const float2* __restrict__ cs, int n_runs,
                                                                   int n_layers, int heads, int page,
                                                                   int64_t n_pages) {
  constexpr int V = D / 8;  // vectors per row
  const int64_t page_vecs = int64_t(heads) * page * V;
  const int64_t layer_vecs = page_vecs * n_pages;
  const int64_t units = int64_t(n_layers) * n_runs;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int r = int(u % n_runs);
    const int64_t layer = u / n_runs;
    const RunDesc rd = runs[r];
    const int lo = rd.lohi & 0xffff, n = (rd.lohi >> 16) - lo;
    const float2* cs_row = cs + int64_t(rd.didx) * (D / 2);
    const uint4* src = pool + layer * layer_vecs + rd.src * page_vecs;
    uint4* dst = pool + layer * layer_vecs + rd.dst * page_vecs;
    const int per_head = n * V;
    const int total = heads * per_head;
    for (int base = 0; base < total; base += kThreads * kUnroll) {
      uint4 x[kUnroll];
      int off[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int i = base + k * kThreads + int(threadIdx.x);
        off[k] = -1;
        if (i < total) {
          const int h = i / per_head;
          const int rem = i - h * per_head;  // (slot - lo) * V + v
          off[k] = (h * page + lo) * V + rem;
          x[k] = __ldcs(src + off[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (off[k] >= 0) __stcs(dst + off[k], rot_vec_interleaved(x[k], cs_row, off[k] % V));
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) repos_half_kernel(uint4* __restrict__ pool,
                                                            const RunDesc* __restrict__ runs,
                                                            const float2* __restrict__ cs, int n_runs, int n_layers,
                                                            int heads, int page, int64_t n_pages) {
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
      uint4 a = __ldcs(src + off), b = __ldcs(src + off + HV);
      const float4* c4 = reinterpret_cast<const float4*>(cs_row + 8 * v);
      const float4 c01 = __ldg(c4), c23 = __ldg(c4 + 1), c45 = __ldg(c4 + 2), c67 = __ldg(c4 + 3);
      rot_halves(a.x, b.x, c01.x, c01.y, c01.z, c01.w);
      rot_halves(a.y, b.y, c23.x, c23.y, c23.z, c23.w);
      rot_halves(a.z, b.z, c45.x, c45.y, c45.z, c45.w);
      rot_halves(a.w, b.w, c67.x, c67.y, c67.z, c67.w);
      __stcs(dst + off, a);
      __stcs(dst + off + HV, b);
    }
  }
}

}  // namespace

cudaError_t launch_repos_rotate(void* kpool, const RunDesc* runs, const float2* cs, int n_runs, int n_layers,
                                int heads, int d_rot, int page, int64_t n_pages, bool half_layout, cudaStream_t st) {
  if (n_runs <= 0) return cudaSuccess;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t units = int64_t(n_layers) * n_runs;
  const unsigned blocks = unsigned(std::min<int64_t>(units, int64_t(sms) * 8));
  uint4* p = static_cast<uint4*>(kpool);
#define AKV_REPOS_CASE(DIM)                                                                              \
  case DIM:                                                                                              \
    if (half_layout)                                                                                     \
      repos_half_kernel<DIM><<<blocks, kThreads, 0, st>>>(p, runs, cs, n_runs, n_layers, heads, page, n_pages); \
    else                                                                                                 \
      repos_interleaved_kernel<DIM><<<blocks, kThreads, 0, st>>>(p, runs, cs, n_runs, n_layers, heads, page,  \
                                                                 n_pages);                              \
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

}  // namespace akv
