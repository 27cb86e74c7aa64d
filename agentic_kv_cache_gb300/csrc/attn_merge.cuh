// Split-KV merge for segment_batch_attn, run by the last CTA of a split item.
//
// A work item whose KV tiles were cut into parts runs as several CTAs.  Each
// part leaves, per query row, the unnormalised output O_c = sum_j 2^(s_j - m_c) v_j,
// its running maximum m_c (log2 units of scaled scores) and l_c =
// sum_j 2^(s_j - m_c).  Merging is the rescale-and-add of partial softmax sums:
//   m = max_c m_c,  l = sum_c l_c 2^(m_c - m),  O = sum_c O_c 2^(m_c - m) / l,
// with natural-log normaliser (m + log2 l) ln 2.  Parts with l_c = 0 saw no
// visible key and carry no weight.
//
// Ordering follows the fence-and-ticket pattern: every thread writes its
// partial and fences, the group meets at a named barrier, one thread takes a
// ticket from the item's counter (zeroed by the host with each launch's work
// list), and the CTA that draws the last ticket fences again and reads every
// part through L2.  Nothing waits on another CTA.
#pragma once

#include <cuda_bf16.h>

#include <cmath>

#include "akv_internal.h"
#include "sm100_ptx.cuh"

namespace akv {

constexpr int kMaxParts = 8;  // the engine cuts an item into at most 8 parts

// Called by the 128 threads (thread = row r) of one query-tile group, on named
// barrier `bar_id`, after each wrote row r of its partial for tile `t` of
// part `w.part`.  `orow` points at the row's first output column (null for a
// row past the segment's queries), `lse` at its normaliser (null when this
// group does not write it).  W is the number of output columns of the part.
template <int W>
__device__ __forceinline__ void merge_if_last(const AttnParams& p, const AttnWork& w, int t, int r, int bar_id,
                                              __nv_bfloat16* orow, float* lse) {
  CombineItem* ci = p.comb + w.comb;
  const int part0 = ci->part0, n_parts = ci->n_parts;
  __threadfence();
  ptx::bar_red_and(bar_id, 128, true);
  bool last = true;
  if (r == 0) last = atomicAdd(&ci->count[t], 1) == n_parts - 1;
  if (!ptx::bar_red_and(bar_id, 128, last)) return;
  __threadfence();

  const int64_t slot = partial_floats(p.comb_tiles, W);
  const float* base = p.partial + int64_t(part0) * slot + int64_t(t) * (W + 2) * 128 + r;
  float m = -INFINITY;
  float lc[kMaxParts], mc[kMaxParts];
#pragma unroll
  for (int c = 0; c < kMaxParts; ++c) {
    lc[c] = c < n_parts ? __ldcg(base + c * slot + int64_t(W + 1) * 128) : 0.f;
    mc[c] = lc[c] > 0.f ? __ldcg(base + c * slot + int64_t(W) * 128) : -INFINITY;
    m = fmaxf(m, mc[c]);
  }
  float wc[kMaxParts];
  float l = 0.f;
#pragma unroll
  for (int c = 0; c < kMaxParts; ++c) {
    wc[c] = lc[c] > 0.f ? ptx::ex2_approx(mc[c] - m) : 0.f;
    l = fmaf(wc[c], lc[c], l);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (orow == nullptr) return;
#pragma unroll 1
  for (int c32 = 0; c32 < W / 32; ++c32) {
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxParts; ++c) {
      if (wc[c] == 0.f) continue;
      const float* src = base + c * slot + int64_t(c32 * 32) * 128;
#pragma unroll
      for (int k = 0; k < 32; ++k) acc[k] = fmaf(wc[c], __ldcg(src + int64_t(k) * 128), acc[k]);
    }
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
      uint4 v;
      __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[k + 0] * inv, acc[k + 1] * inv);
      __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[k + 2] * inv, acc[k + 3] * inv);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[k + 4] * inv, acc[k + 5] * inv);
      __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[k + 6] * inv, acc[k + 7] * inv);
      v.x = *reinterpret_cast<uint32_t*>(&b0);
      v.y = *reinterpret_cast<uint32_t*>(&b1);
      v.z = *reinterpret_cast<uint32_t*>(&b2);
      v.w = *reinterpret_cast<uint32_t*>(&b3);
      *reinterpret_cast<uint4*>(orow + c32 * 32 + k) = v;
    }
  }
  if (lse) *lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace akv
