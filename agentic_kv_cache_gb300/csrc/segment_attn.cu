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
// GB300 design (one CTA = two consecutive 128-row query tiles A, B of one kv
// head; rows are (query token, query head of the kv group) pairs so the G
// query heads sharing a kv head share every K/V load):
//   * warp 0 issues TMA loads: both Q tiles once, then K_j and V_j of every
//     128-key tile into a ring of five shared-memory slots (K0 V0 K1 V1 ...),
//     one box of page_size rows per run (page), 128-byte swizzled; slots past
//     the segment's last run reload its first page (finite, masked out);
//   * warp 1 owns TMEM (S_A, S_B, O_A, O_B: 4 x 128 columns) and issues
//     tcgen05.mma from one thread, per KV tile j and per query tile T:
//     O_T += P_T(j-1) V_{j-1}, then S_T(j) = Q_T K_j^T, then one commit -- so
//     "S_T(j) is ready" also means "O_T is stable and P_T may be rewritten";
//   * warpgroups 1 (tile A) and 2 (tile B) run the online softmax, one thread
//     per row = one TMEM lane: a whole score row comes in with one 128-column
//     TMEM load, row max and row sum need no shuffles, O is rescaled lazily in
//     TMEM (only when the running max grows by more than 2^8), and P (bf16) is
//     written back into the S columns already consumed, where the next PV MMA
//     reads it as its TMEM A operand (the MMA thread issues that PV before the
//     QK that overwrites S, and one thread's MMAs execute in issue order).
//     While one warpgroup computes exponentials the tensor core runs the other
//     tile's MMAs;
//   * every wait is bounded; on time-out the CTA records AKV_ERR_DEVICE_TIMEOUT
//     in the device error word, drains its copies and MMAs, frees TMEM, exits.
#include <cuda_bf16.h>

#include <climits>
#include <cstdint>

#include "akv_internal.h"
#include "sm100_ptx.cuh"

namespace akv {
namespace {

constexpr int kThreads = 384;  // 3 warpgroups: control (producer, MMA), softmax A, softmax B
constexpr int kLaunchRegs = 168;  // per thread at launch: 65536 / 384, rounded down to 8
constexpr int kCtlRegs = 120;     // control warpgroup after re-allocation (producer + MMA loops)
constexpr int kSoftmaxRegs = 192; // each softmax warpgroup after re-allocation
static_assert(4 * 32 * kCtlRegs + 8 * 32 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kTileKeys = 128;
constexpr int kRows = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr int32_t kErrTimeout = 7;  // AKV_ERR_DEVICE_TIMEOUT
constexpr int32_t kErrDevice = 8;   // AKV_ERR_DEVICE
constexpr int kSlots = 5;

template <int D>
struct Layout {
  static constexpr int kBlocks = D / 64;              // 64-element (128-byte) column blocks
  static constexpr uint32_t kBlockBytes = 128 * 128;  // 128 rows x 128 bytes
  static constexpr uint32_t kTile = kBlocks * kBlockBytes;
  static constexpr uint32_t kQ = 0;                          // Q_A, Q_B
  static constexpr uint32_t kSlot = kQ + 2 * kTile;          // K/V slots
  static constexpr uint32_t kBars = kSlot + kSlots * kTile;
  static constexpr uint32_t kBytes = kBars + 256;
};

enum Bar {
  kBarQ = 0,
  kBarFull0,  // + slot
  kBarEmpty0 = kBarFull0 + kSlots,
  kBarS0 = kBarEmpty0 + kSlots,  // + tile
  kBarP0 = kBarS0 + 2,
  kBarO0 = kBarP0 + 2,
  kBarFin = kBarO0 + 2,
  kNumBars
};
static_assert(kNumBars * 8 + 8 <= 256, "barrier area");

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

// ---------------------------------------------------------------- producer
template <int D>
__device__ __forceinline__ void produce(const AttnParams& p, const AttnWork& w, const AttnSeg& seg, uint32_t sbase,
                        volatile int* abort_flag) {
  using L = Layout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int G = p.group, tpt = kRows / G, rpt = kTileKeys / p.page;
  const int n_max = max(w.n_a, w.n_b);
  const int q_tok0 = seg.q_row0 + w.qt0 * tpt;
  ptx::mbar_arrive_expect_tx(bar(kBarQ), (w.n_b > 0 ? 2 : 1) * L::kTile);
  for (int t = 0; t < (w.n_b > 0 ? 2 : 1); ++t)
    for (int kb = 0; kb < L::kBlocks; ++kb)
      ptx::tma_load_3d(sbase + L::kQ + t * L::kTile + kb * L::kBlockBytes, &p.q_map, bar(kBarQ), kb * 64,
                       w.kvh * G, q_tok0 + t * tpt);
  const int layer_base = p.layer * p.n_pages;
  const AttnRun first = p.runs[seg.run_off];
  bool ok = true;
  int issued = 0;  // loads issued
  for (int ld = 0; ld < 2 * n_max; ++ld) {
    const int j = ld >> 1, is_v = ld & 1, slot = ld % kSlots, use = ld / kSlots;
    if (use >= 1 && !ptx::mbar_wait(bar(kBarEmpty0 + slot), (use - 1) & 1, abort_flag, kWaitLimitNs)) {
      ok = false;
      break;
    }
    const uint32_t dst = sbase + L::kSlot + slot * L::kTile;
    const CUtensorMap* map = is_v ? &p.v_map : &p.k_map;
    ptx::mbar_arrive_expect_tx(bar(kBarFull0 + slot), L::kTile);
    for (int g = 0; g < rpt; ++g) {
      const int ri = j * rpt + g;
      const AttnRun run = ri < seg.n_runs ? p.runs[seg.run_off + ri] : first;
      const int pg = layer_base + (is_v ? run.vp : run.kp);
      for (int kb = 0; kb < L::kBlocks; ++kb)
        ptx::tma_load_4d(dst + kb * L::kBlockBytes + g * p.page * 128, map, bar(kBarFull0 + slot), kb * 64, 0, w.kvh,
                         pg);
    }
    issued = ld + 1;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 0, 0);
    *abort_flag = 1;
  }
  // Drain: every copy issued here has landed before the CTA may exit.
  ptx::mbar_wait(bar(kBarQ), 0, abort_flag, kDrainLimitNs);
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    const int uses = issued > s ? (issued - s + kSlots - 1) / kSlots : 0;  // loads that went to slot s
    if (uses) ptx::mbar_wait(bar(kBarFull0 + s), (uses - 1) & 1, abort_flag, kDrainLimitNs);
  }
}

// --------------------------------------------------------------------- MMA
// Per KV tile j and query tile T: O_T += P_T(j-1) V_{j-1} (once P_T(j-1) is
// written), then S_T(j) = Q_T K_j^T, then one commit to S_T's barrier.  Slots
// are released (commit to their empty barrier) after their last reader.
template <int D>
__device__ __forceinline__ void issue_mma(const AttnParams& p, const AttnWork& w, uint32_t sbase, uint32_t tmem,
                          volatile int* abort_flag) {
  using L = Layout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  constexpr uint32_t idesc_qk = ptx::idesc_bf16(kRows, kTileKeys, false);
  constexpr uint32_t idesc_pv = ptx::idesc_bf16(kRows, D, true);
  const int n_t[2] = {w.n_a, w.n_b};
  const int n_max = max(w.n_a, w.n_b);
  auto slot_of = [](int ld) { return ld % kSlots; };
  auto full_parity = [](int ld) { return (ld / kSlots) & 1; };
  bool ok = ptx::mbar_wait(bar(kBarQ), 0, abort_flag, kWaitLimitNs);
  for (int j = 0; j <= n_max && ok; ++j) {
    bool k_ready = false, v_ready = false;
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {
      if (!ok) break;
      const uint32_t tS = tmem + 128u * t, tO = tmem + 256u + 128u * t;
      if (j >= 1 && j - 1 < n_t[t]) {
        if (!v_ready) {
          const int ld = 2 * (j - 1) + 1;
          if (!(ok = ptx::mbar_wait(bar(kBarFull0 + slot_of(ld)), full_parity(ld), abort_flag, kWaitLimitNs))) break;
          v_ready = true;
        }
        if (!(ok = ptx::mbar_wait(bar(kBarP0 + t), (j - 1) & 1, abort_flag, kWaitLimitNs))) break;
        ptx::tc_fence_after();
        const uint32_t vt = sbase + L::kSlot + slot_of(2 * (j - 1) + 1) * L::kTile;
#pragma unroll 1
        for (int ks = 0; ks < kTileKeys / 16; ++ks)  // P: 16 keys = 8 packed TMEM columns per step
          ptx::mma_bf16_tmem_a(tO, tS + 8u * ks, ptx::smem_desc(vt + ks * 16 * 128, L::kBlockBytes, 1024), idesc_pv,
                               (j > 1 || ks > 0));
        if (j - 1 == n_t[t] - 1) ptx::mma_commit(bar(kBarO0 + t));
      }
      if (j < n_t[t]) {
        if (!k_ready) {
          const int ld = 2 * j;
          if (!(ok = ptx::mbar_wait(bar(kBarFull0 + slot_of(ld)), full_parity(ld), abort_flag, kWaitLimitNs))) break;
          k_ready = true;
          ptx::tc_fence_after();
        }
        const uint32_t kt = sbase + L::kSlot + slot_of(2 * j) * L::kTile;
        const uint32_t qt = sbase + L::kQ + t * L::kTile;
#pragma unroll 1
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * L::kBlockBytes + (ks & 3) * 32;
          ptx::mma_bf16(tS, ptx::smem_desc(qt + off, 16, 1024), ptx::smem_desc(kt + off, 16, 1024), idesc_qk, ks > 0);
        }
        ptx::mma_commit(bar(kBarS0 + t));
      }
    }
    if (!ok) break;
    if (j >= 1) ptx::mma_commit(bar(kBarEmpty0 + slot_of(2 * (j - 1) + 1)));  // V_{j-1} done
    if (j < n_max) ptx::mma_commit(bar(kBarEmpty0 + slot_of(2 * j)));        // K_j done
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 1, 0);
    *abort_flag = 1;
  }
  // Every MMA issued above has completed before TMEM is released.
  ptx::mma_commit(bar(kBarFin));
  ptx::mbar_wait(bar(kBarFin), 0, abort_flag, kDrainLimitNs);
}

// ----------------------------------------------------------------- softmax
// Visibility of the 128 key columns of one KV tile for one query row, as a
// 128-bit mask: column c = run c / PAGE, slot c % PAGE of the tile's runs is
// visible when the slot lies in the run and its entry index is within the
// row's causal limit.  all_full tells whether every column is visible.
template <int PAGE>
struct TileMask {
  static constexpr int kRuns = kTileKeys / PAGE;
  uint32_t m[4];
  bool all_full;

  __device__ __forceinline__ void build(const AttnRun* runs, int first, int n_runs, int lim) {
    // One run at a time: its visible slots are [lo, min(hi, lo + (lim - es) + 1)).
    bool full = true;
    m[0] = m[1] = m[2] = m[3] = 0u;
#pragma unroll
    for (int g = 0; g < kRuns; ++g) {
      const int ri = first + g;
      if (ri >= n_runs) {
        full = false;
        continue;
      }
      const int2 rr = *reinterpret_cast<const int2*>(&runs[ri].lohi);
      const int lo = rr.x & 0xffff, hi = rr.x >> 16;
      const int64_t cap = int64_t(lo) + int64_t(lim) - int64_t(rr.y) + 1;
      const int vhi = int(cap < hi ? (cap < lo ? lo : cap) : hi);
      full = full && lo == 0 && vhi == PAGE;
      const int a = g * PAGE + lo, b = g * PAGE + vhi;  // bit range [a, b)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (32 * w + 32 <= g * PAGE || 32 * w >= (g + 1) * PAGE) continue;  // word outside this run
        const int wa = min(max(a - 32 * w, 0), 32), wb = min(max(b - 32 * w, 0), 32);
        if (wb > wa) {
          const uint32_t upper = wb == 32 ? 0xffffffffu : ((1u << wb) - 1u);
          m[w] |= upper & ~((1u << wa) - 1u);
        }
      }
    }
    all_full = full;
  }
};

// One warpgroup per query tile t; thread = row r = TMEM lane r.  No barrier
// across warps inside the loop: each warp synchronises only through mbarriers
// and its own warp-collective TMEM accesses.
template <int D, int PAGE>
__device__ __forceinline__ void softmax_tile(const AttnParams& p, const AttnWork& w, const AttnSeg& seg, int t, uint32_t sbase,
                             uint32_t tmem, volatile int* abort_flag) {
  using L = Layout<D>;
  constexpr int kRuns = kTileKeys / PAGE;
  const int n_t = t == 0 ? w.n_a : w.n_b;
  if (n_t == 0) return;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int quad = (threadIdx.x / 32) & 3;  // TMEM lane quadrant this warp may access (warp % 4)
  const int lane = threadIdx.x % 32;
  const int r = quad * 32 + lane;
  const uint32_t lane_addr = uint32_t(quad * 32) << 16;
  const uint32_t tS = tmem + 128u * t, tO = tmem + 256u + 128u * t;
  const int G = p.group, tpt = kRows / G;
  const int t_loc = r / G, g = r % G;
  const int qi = (w.qt0 + t) * tpt + t_loc;  // query index inside the segment
  const bool row_valid = qi < seg.q_len;
  const int lim = seg.kv_len - seg.q_len + (row_valid ? qi : seg.q_len - 1);
  const float sl2 = p.scale_log2;
  const AttnRun* runs = p.runs + seg.run_off;
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  TileMask<PAGE> mask;
  mask.build(runs, 0, seg.n_runs, lim);
  for (int j = 0; j < n_t; ++j) {
    ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarS0 + t), j & 1, abort_flag, kWaitLimitNs));
    if (!ok) break;
    ptx::tc_fence_after();
    if (lane == 0 && (j + 1) * kRuns < seg.n_runs) ptx::prefetch_l1(runs + (j + 1) * kRuns);
    uint32_t u[kTileKeys];
    ptx::tmem_load64_async(tS + lane_addr, u);
    ptx::tmem_load64_async(tS + lane_addr + 64, u + 64);
    ptx::tmem_wait_load128(u);
    if (!mask.all_full) {
#pragma unroll
      for (int c = 0; c < kTileKeys; ++c)
        if (!((mask.m[c >> 5] >> (c & 31)) & 1u)) u[c] = 0xff800000u;  // -inf
    }
    float mx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) mx[k] = __uint_as_float(u[k]);
#pragma unroll
    for (int c = 4; c < kTileKeys; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(u[c]));
    const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
    const float m_new = fmaxf(m_run, mt);
    const bool resc = m_new > m_run + 8.0f;
    const float m_use = resc ? m_new : m_run;
    const float alpha = resc ? ptx::ex2_approx(m_run - m_new) : 1.0f;
    const float msub = m_use == -INFINITY ? 0.f : m_use;
    // P = exp2(s * scale * log2 e - m) as bf16 pairs (keys 2c, 2c+1 -> column c),
    // stored over the S columns already read; the PV MMA reads it from TMEM.
    float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < kTileKeys / 2; ++c) {
      const float p0 = ptx::ex2_approx(fmaf(__uint_as_float(u[2 * c]), sl2, -msub));
      const float p1 = ptx::ex2_approx(fmaf(__uint_as_float(u[2 * c + 1]), sl2, -msub));
      sum[(2 * c) & 3] += p0;
      sum[(2 * c + 1) & 3] += p1;
      u[c] = pack_bf16(p0, p1);  // u[c] was consumed by an earlier pair
    }
    ptx::tmem_store32_async(tS + lane_addr, u);
    ptx::tmem_store32_async(tS + lane_addr + 32, u + 32);
    const float rowsum = (sum[0] + sum[1]) + (sum[2] + sum[3]);
    ptx::tmem_wait_store64(u);
    // Lazy rescale of O (after P is stored, before PV_T(j) may start): O_T is
    // stable here because S_T(j) completes after PV_T(j-1).
    if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_load32(tO + lane_addr + c * 32, o);
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
        ptx::tmem_store32(tO + lane_addr + c * 32, o);
      }
    }
    // The next tile's visibility (its runs were prefetched into L1 above).
    if (j + 1 < n_t) mask.build(runs, (j + 1) * kRuns, seg.n_runs, lim);
    l_run = l_run * alpha + rowsum;
    m_run = m_use;
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(kBarP0 + t));
  }
  if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarO0 + t), 0, abort_flag, kWaitLimitNs));
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 2 + t, 0);
    *abort_flag = 1;
    return;
  }
  ptx::tc_fence_after();
  const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
  __nv_bfloat16* orow =
      static_cast<__nv_bfloat16*>(p.o) + (int64_t(seg.q_row0 + qi) * p.hq + int64_t(w.kvh) * G + g) * D;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    ptx::tmem_load32(tO + lane_addr + c * 32, o);
    if (row_valid) {
#pragma unroll
      for (int k = 0; k < 32; k += 8) {
        uint4 v;
        v.x = pack_bf16(__uint_as_float(o[k + 0]) * inv, __uint_as_float(o[k + 1]) * inv);
        v.y = pack_bf16(__uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
        v.z = pack_bf16(__uint_as_float(o[k + 4]) * inv, __uint_as_float(o[k + 5]) * inv);
        v.w = pack_bf16(__uint_as_float(o[k + 6]) * inv, __uint_as_float(o[k + 7]) * inv);
        *reinterpret_cast<uint4*>(orow + c * 32 + k) = v;
      }
    }
  }
  if (row_valid && p.lse) {
    const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    p.lse[int64_t(seg.q_row0 + qi) * p.hq + int64_t(w.kvh) * G + g] = lse;
  }
}

template <int D, int PAGE>
__global__ void __launch_bounds__(kThreads, 1) segment_attn_kernel(const __grid_constant__ AttnParams p, int smem_bytes) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  uint8_t* smem = reinterpret_cast<uint8_t*>((raw + 1023) & ~uintptr_t(1023));
  if (smem + L::kBytes > smem_raw + smem_bytes) {  // layout does not fit: report, touch nothing
    if (threadIdx.x == 0) raise_error(p.err, kErrDevice, blockIdx.x, int(raw & 1023), 0);
    return;
  }
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + L::kBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBars + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBars + 8 * kNumBars + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) ptx::mbar_init(bars + 8u * i, (i == kBarP0 || i == kBarP0 + 1) ? 128 : 1);
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

  // Each role loads its work item itself, so nothing but a few addresses is
  // live across the register re-allocation.
  if (warp < 4) {
    ptx::regs_decrease<kCtlRegs>();
    if (warp == 0 && lane == 0) {
      const AttnWork w = p.work[blockIdx.x];
      produce<D>(p, w, p.segs[w.seg], sbase, abort_flag);
    }
    if (warp == 1 && lane == 0) issue_mma<D>(p, p.work[blockIdx.x], sbase, tmem, abort_flag);
    __syncwarp();
    ptx::regs_increase<kLaunchRegs>();
  } else {
    ptx::regs_increase<kSoftmaxRegs>();
    const AttnWork w = p.work[blockIdx.x];
    softmax_tile<D, PAGE>(p, w, p.segs[w.seg], warp < 8 ? 0 : 1, sbase, tmem, abort_flag);
    __syncwarp();
    ptx::regs_decrease<kLaunchRegs>();
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
// SM; both head dims request enough shared memory to guarantee that.
int segment_attn_smem_bytes(int dim) {
  if (dim != 64 && dim != 128) return -1;
  return int(Layout<128>::kBytes) + 1024;
}

template <int D, int PAGE>
cudaError_t launch_one(const AttnParams& p, int smem, cudaStream_t st) {
  // The register re-allocation inside the kernel needs the launch to hold
  // kLaunchRegs per thread; refuse to launch otherwise (it would never finish).
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, segment_attn_kernel<D, PAGE>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(segment_attn_kernel<D, PAGE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  segment_attn_kernel<D, PAGE><<<p.n_work, kThreads, smem, st>>>(p, smem);
  return cudaGetLastError();
}

cudaError_t launch_segment_attn(const AttnParams& p, int dim, cudaStream_t st) {
  if (p.n_work <= 0) return cudaSuccess;
  const int smem = segment_attn_smem_bytes(dim);
  if (smem < 0) return cudaErrorInvalidValue;
  if (dim == 64 && p.page == 16) return launch_one<64, 16>(p, smem, st);
  if (dim == 64 && p.page == 64) return launch_one<64, 64>(p, smem, st);
  if (dim == 128 && p.page == 16) return launch_one<128, 16>(p, smem, st);
  if (dim == 128 && p.page == 64) return launch_one<128, 64>(p, smem, st);
  return cudaErrorInvalidValue;
}

}  // namespace akv
