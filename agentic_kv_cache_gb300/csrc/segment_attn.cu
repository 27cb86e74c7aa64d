// segment_batch_attn: one fused launch of causal attention over many segments,
// each reading its own piecewise-discontinuous list of KV pages.
//
// [AKV-blog] section 4 "Segment-Batch Attention Kernel Architecture": after
// drops and repositions the logical-to-physical page map is piecewise
// discontinuous; a FlashAttention-style tile loop walks the segment's pages,
// with online softmax, in one grid over all segments.  [AKV-notes] section 3
// "Segment-Batch Attention": queries are partitioned by visible history, each
// segment selects its KV pages and runs standard causal attention with no
// dense mask.  [AKV-blog] section 2 "The Drop Primitive" fixes what is
// computed: softmax(Q K^T * scale + M) V with M = -inf on invisible entries.
//
// GB300 design (one CTA = one 128-row query tile of one kv head):
//   * rows are (query token, query head of the kv group) pairs, so the G query
//     heads that share a kv head share every K/V tile load (GQA packing);
//   * warp 0 issues TMA loads: the Q tile once, then per 128-key tile one box
//     of page_size rows per run ("page") straight from the paged pool into a
//     128-byte-swizzled shared-memory tile, double buffered; slots of a tile
//     past the segment's last run load the segment's first page again (finite
//     data, masked out like every slot outside a run);
//   * warp 1 owns TMEM (512 columns: S0, S1, O) and issues tcgen05.mma from one
//     thread: S_j = Q K_j^T into TMEM, then O += P_j V_j with P from shared memory;
//   * warps 2-5 (128 threads, one per row = one TMEM lane) run the online
//     softmax: each thread holds a whole score row, so row max and row sum need
//     no shuffles; rescaling of O is lazy (only when the running max grows by
//     more than 2^8), done in TMEM; the epilogue normalises O and writes bf16.
//   * every wait is bounded; on time-out the CTA records AKV_ERR_DEVICE_TIMEOUT
//     in the device error word, drains its copies and MMAs, frees TMEM, exits.
#include <cuda_bf16.h>

#include <climits>
#include <cstdint>

#include "akv_internal.h"
#include "sm100_ptx.cuh"

namespace akv {
namespace {

constexpr int kThreads = 192;
constexpr int kTileKeys = 128;
constexpr int kRows = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait
constexpr int32_t kErrTimeout = 7;                 // AKV_ERR_DEVICE_TIMEOUT

template <int D>
struct Layout {
  static constexpr int kBlocks = D / 64;                 // 64-element (128-byte) K blocks
  static constexpr uint32_t kBlockBytes = 128 * 128;     // 128 rows x 128 bytes
  static constexpr uint32_t kTileBytes = kBlocks * kBlockBytes;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK0 = kQ + kTileBytes;
  static constexpr uint32_t kV0 = kK0 + 2 * kTileBytes;
  static constexpr uint32_t kP = kV0 + 2 * kTileBytes;
  static constexpr uint32_t kBars = kP + 2 * kBlockBytes;  // P: 128 rows x 128 keys
  static constexpr uint32_t kColE = kBars + 256;           // int32 [2][128]: entry index per key column
  static constexpr uint32_t kBytes = kColE + 2 * 128 * 4;
};

// barrier slots (8 bytes each) after the tiles
enum Bar { kBarQ = 0, kBarK0, kBarK1, kBarV0, kBarV1, kBarE0, kBarE1, kBarS0, kBarS1, kBarP, kBarO, kBarFin, kNumBars };

__device__ __forceinline__ void raise_error(DevErr* err, int32_t code, int a, int b, int c) {
  if (atomicCAS(&err->code, 0, code) == 0) {
    err->info[0] = a;
    err->info[1] = b;
    err->info[2] = c;
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) segment_attn_kernel(const __grid_constant__ AttnParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBars + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBars + 8 * kNumBars + 8);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const AttnWork w = p.work[blockIdx.x];
  const AttnSeg seg = p.segs[w.seg];
  const int G = p.group;
  const int tpt = kRows / G;  // query tokens per tile
  const int n_tiles = w.n_tiles;
  const int rpt = kTileKeys / p.page;  // runs (pages) per key tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;
      if (i == kBarP) count = 128;
      ptx::mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&p.q_map);
    ptx::prefetch_tensormap(&p.k_map);
    ptx::prefetch_tensormap(&p.v_map);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int q_tok0 = seg.q_row0 + w.qt * tpt;
      int armed[2] = {0, 0};
      bool ok = true;
      ptx::mbar_arrive_expect_tx(bar(kBarQ), L::kTileBytes);
      for (int kb = 0; kb < L::kBlocks; ++kb)
        ptx::tma_load_3d(sbase + L::kQ + kb * L::kBlockBytes, &p.q_map, bar(kBarQ), kb * 64, w.kvh * G, q_tok0);
      const int layer_base = p.layer * p.n_pages;
      // Slots past the last run: reload the first run's pages (finite, masked out).
      const int fill_k = layer_base + __ldg(&p.runs[seg.run_off].kp);
      const int fill_v = layer_base + __ldg(&p.runs[seg.run_off].vp);
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        if (j >= 2 && !ptx::mbar_wait(bar(kBarE0 + s), ((j >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t kdst = sbase + L::kK0 + s * L::kTileBytes;
        const uint32_t vdst = sbase + L::kV0 + s * L::kTileBytes;
        ptx::mbar_arrive_expect_tx(bar(kBarK0 + s), L::kTileBytes);
        for (int g = 0; g < rpt; ++g) {
          const int ri = j * rpt + g;
          const int pg = ri < seg.n_runs ? layer_base + __ldg(&p.runs[seg.run_off + ri].kp) : fill_k;
          for (int kb = 0; kb < L::kBlocks; ++kb)
            ptx::tma_load_4d(kdst + kb * L::kBlockBytes + g * p.page * 128, &p.k_map, bar(kBarK0 + s), kb * 64, 0,
                             w.kvh, pg);
        }
        ptx::mbar_arrive_expect_tx(bar(kBarV0 + s), L::kTileBytes);
        for (int g = 0; g < rpt; ++g) {
          const int ri = j * rpt + g;
          const int pg = ri < seg.n_runs ? layer_base + __ldg(&p.runs[seg.run_off + ri].vp) : fill_v;
          for (int kb = 0; kb < L::kBlocks; ++kb)
            ptx::tma_load_4d(vdst + kb * L::kBlockBytes + g * p.page * 128, &p.v_map, bar(kBarV0 + s), kb * 64, 0,
                             w.kvh, pg);
        }
        ++armed[s];
      }
      if (!ok) {
        raise_error(p.err, kErrTimeout, blockIdx.x, 0, 0);
        *abort_flag = 1;
      }
      // Drain: every copy this thread issued has landed before the CTA can exit.
      ptx::mbar_wait(bar(kBarQ), 0, abort_flag, 100000000ull);
      for (int s = 0; s < 2; ++s)
        if (armed[s]) {
          ptx::mbar_wait(bar(kBarK0 + s), (armed[s] - 1) & 1, abort_flag, 100000000ull);
          ptx::mbar_wait(bar(kBarV0 + s), (armed[s] - 1) & 1, abort_flag, 100000000ull);
        }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16(kRows, kTileKeys, false);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16(kRows, D, true);
      auto issue_qk = [&](int j) {
        const int s = j & 1;
        const uint32_t kt = sbase + L::kK0 + s * L::kTileBytes;
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * L::kBlockBytes + (ks & 3) * 32;
          ptx::mma_bf16(tS[s], ptx::smem_desc(sbase + L::kQ + off, 16, 1024), ptx::smem_desc(kt + off, 16, 1024),
                        idesc_qk, ks > 0);
        }
        ptx::mma_commit(bar(kBarS0 + s));
      };
      bool ok = ptx::mbar_wait(bar(kBarQ), 0, abort_flag, kWaitLimitNs);
      if (ok && n_tiles > 0) {
        ok = ptx::mbar_wait(bar(kBarK0), 0, abort_flag, kWaitLimitNs);
        if (ok) {
          ptx::tc_fence_after();
          issue_qk(0);
        }
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (j + 1 < n_tiles) {
          const int s1 = (j + 1) & 1;
          if (!(ok = ptx::mbar_wait(bar(kBarK0 + s1), ((j + 1) >> 1) & 1, abort_flag, kWaitLimitNs))) break;
          ptx::tc_fence_after();
          issue_qk(j + 1);
        }
        if (!(ok = ptx::mbar_wait(bar(kBarP), j & 1, abort_flag, kWaitLimitNs))) break;
        if (!(ok = ptx::mbar_wait(bar(kBarV0 + (j & 1)), (j >> 1) & 1, abort_flag, kWaitLimitNs))) break;
        ptx::tc_fence_after();
        const uint32_t vt = sbase + L::kV0 + (j & 1) * L::kTileBytes;
        for (int ks = 0; ks < kTileKeys / 16; ++ks) {
          const uint32_t poff = (ks >> 2) * L::kBlockBytes + (ks & 3) * 32;
          ptx::mma_bf16(tO, ptx::smem_desc(sbase + L::kP + poff, 16, 1024),
                        ptx::smem_desc(vt + ks * 16 * 128, L::kBlockBytes, 1024), idesc_pv, (j > 0 || ks > 0));
        }
        ptx::mma_commit(bar(kBarE0 + (j & 1)));
        ptx::mma_commit(bar(kBarO));
      }
      if (!ok) {
        raise_error(p.err, kErrTimeout, blockIdx.x, 1, 0);
        *abort_flag = 1;
      }
      // Every MMA issued above has completed before TMEM is released.
      ptx::mma_commit(bar(kBarFin));
      ptx::mbar_wait(bar(kBarFin), 0, abort_flag, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_addr = uint32_t(quad * 32) << 16;
    const int t_loc = r / G, g = r % G;
    const int qi = w.qt * tpt + t_loc;  // query index inside the segment
    const bool row_valid = qi < seg.q_len;
    const int lim = seg.kv_len - seg.q_len + (row_valid ? qi : seg.q_len - 1);
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    uint8_t* prow = smem + L::kP + r * 128;
    int* colE = reinterpret_cast<int*>(smem + L::kColE);
    int page_shift = 4;
    while ((1 << page_shift) < p.page) ++page_shift;
    for (int j = 0; j < n_tiles; ++j) {
      // Entry index of key column r of this tile (INT_MAX: no entry there).
      // Columns are (run g = c / page, slot = c % page) of the tile's runs.
      int e = INT_MAX;
      {
        const int gg = r >> page_shift, sl = r & (p.page - 1);
        const int ri = j * rpt + gg;
        if (ri < seg.n_runs) {
          const AttnRun ar = p.runs[seg.run_off + ri];
          const int lo = ar.lohi & 0xffff, hi = ar.lohi >> 16;
          if (sl >= lo && sl < hi) e = ar.es + (sl - lo);
        }
        colE[(j & 1) * 128 + r] = e;
      }
      ok = ptx::mbar_wait(bar(kBarS0 + (j & 1)), (j >> 1) & 1, abort_flag, kWaitLimitNs);
      if (!ptx::bar_red_and(1, 128, ok)) {
        ok = false;
        break;
      }
      const bool all_valid = ptx::bar_red_and(1, 128, e != INT_MAX);
      ptx::tc_fence_after();
      float sc[kTileKeys];
#pragma unroll
      for (int c = 0; c < kTileKeys / 32; ++c) {
        uint32_t u[32];
        ptx::tmem_load32(tS[j & 1] + lane_addr + c * 32, u);
#pragma unroll
        for (int k = 0; k < 32; ++k) sc[c * 32 + k] = __uint_as_float(u[k]);
      }
      // Visibility: missing slots of partial runs, missing runs, causal limit.
      // With every column valid the entries are consecutive, so the last
      // column holds the tile's largest entry index.
      const int* ce = colE + (j & 1) * 128;
      if (!all_valid || ce[kTileKeys - 1] > lim) {
#pragma unroll
        for (int c = 0; c < kTileKeys; ++c)
          if (ce[c] > lim) sc[c] = -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTileKeys; ++c) mt = fmaxf(mt, sc[c]);
      mt *= sl2;
      const float m_new = fmaxf(m_run, mt);
      const bool resc = m_new > m_run + 8.0f;
      const float m_use = resc ? m_new : m_run;
      const float alpha = resc ? ptx::ex2_approx(m_run - m_new) : 1.0f;
      const float msub = m_use == -INFINITY ? 0.f : m_use;
      float rowsum = 0.f;
      uint32_t pk[kTileKeys / 2];
#pragma unroll
      for (int c = 0; c < kTileKeys; c += 2) {
        const float p0 = ptx::ex2_approx(fmaf(sc[c], sl2, -msub));
        const float p1 = ptx::ex2_approx(fmaf(sc[c + 1], sl2, -msub));
        rowsum += p0 + p1;
        pk[c / 2] = pack_bf16(p0, p1);
      }
      if (j > 0) {
        ok = ptx::mbar_wait(bar(kBarO), (j - 1) & 1, abort_flag, kWaitLimitNs);
        if (!ptx::bar_red_and(1, 128, ok)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      // P row -> shared memory, K-major 128-byte swizzle (16-byte chunk c of
      // row r lands in chunk c ^ (r & 7)), two 64-key blocks.
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int k0 = kb * 32 + c * 4;
          uint4 v = make_uint4(pk[k0], pk[k0 + 1], pk[k0 + 2], pk[k0 + 3]);
          *reinterpret_cast<uint4*>(prow + kb * L::kBlockBytes + ((c ^ (r & 7)) << 4)) = v;
        }
      }
      ptx::fence_proxy_async_smem();
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          ptx::tmem_load32(tO + lane_addr + c * 32, u);
#pragma unroll
          for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
          ptx::tmem_store32(tO + lane_addr + c * 32, u);
        }
      }
      l_run = l_run * alpha + rowsum;
      m_run = m_use;
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(kBarP));
    }
    if (ok && n_tiles > 0) {
      ok = ptx::mbar_wait(bar(kBarO), (n_tiles - 1) & 1, abort_flag, kWaitLimitNs);
      ok = ptx::bar_red_and(1, 128, ok);
    }
    if (!ok) {
      raise_error(p.err, kErrTimeout, blockIdx.x, 2, 0);
      *abort_flag = 1;
    } else {
      ptx::tc_fence_after();
      const float inv = (n_tiles > 0 && l_run > 0.f) ? 1.0f / l_run : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) +
                            (int64_t(seg.q_row0 + qi) * p.hq + int64_t(w.kvh) * G + g) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        ptx::tmem_load32(tO + lane_addr + c * 32, u);
        if (n_tiles == 0) {
#pragma unroll
          for (int k = 0; k < 32; ++k) u[k] = 0u;
        }
        if (row_valid) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(u[k + 0]) * inv, __uint_as_float(u[k + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(u[k + 2]) * inv, __uint_as_float(u[k + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(u[k + 4]) * inv, __uint_as_float(u[k + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(u[k + 6]) * inv, __uint_as_float(u[k + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + k) = v;
          }
        }
      }
      if (row_valid && p.lse) {
        const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        p.lse[int64_t(seg.q_row0 + qi) * p.hq + int64_t(w.kvh) * G + g] = lse;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// Every CTA allocates all 512 TMEM columns, so exactly one CTA may live on an
// SM: both head dims request the d=128 footprint, which is over half of the
// shared memory of an SM.
int segment_attn_smem_bytes(int dim) {
  if (dim != 64 && dim != 128) return -1;
  return int(Layout<128>::kBytes) + 1024;
}

cudaError_t launch_segment_attn(const AttnParams& p, int dim, cudaStream_t st) {
  if (p.n_work <= 0) return cudaSuccess;
  const int smem = segment_attn_smem_bytes(dim);
  if (smem < 0) return cudaErrorInvalidValue;
  cudaError_t e;
  if (dim == 64) {
    e = cudaFuncSetAttribute(segment_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    segment_attn_kernel<64><<<p.n_work, kThreads, smem, st>>>(p);
  } else {
    e = cudaFuncSetAttribute(segment_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    segment_attn_kernel<128><<<p.n_work, kThreads, smem, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace akv
