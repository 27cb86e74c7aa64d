// attn_mass: per-token attention mass of a segment-batch attention launch.
//
// [AKV-blog] "Dilemma 1: Client-Side vs Server-Side Drop Policy": a serving
// engine can pick droppable blocks itself by watching the cumulative
// attention weight historical blocks receive.  This pass measures it: for
// every visible entry of a segment, the softmax probability it receives,
// summed over the segment's query rows and query heads,
//     mass[e] = sum_rows sum_heads exp(scale * q . k_e - lse_row),
// with lse the natural-log normaliser the attention pass returned (so the
// probabilities are the final ones).  The policy on top (an epsilon over
// three decode turns) is the caller's.
//
// GB300 design (one CTA per (segment, kv head, pair of 128-row query tiles,
// range of K tiles); the mass needs no online rescaling, since the lse is
// final, so the host may cut a pair's K tiles into ranges that run as
// separate CTAs and add into the same outputs):
//   * warp 0 loads both Q tiles once and streams K tiles (128 keys) through a
//     2-slot ring by TMA, whole-tile copies when the runs sit on consecutive
//     pages; each K tile feeds both query tiles;
//   * warp 1 issues, per K tile j and query tile t, S_t(j) = Q_t K_j^T into
//     the TMEM score buffer of t, then the column sums of t's probability tile
//     of j - 1 as a second MMA, D_t = ones(128 x 128) P_t(j-1), whose every
//     row is the vector of column sums (P_t is bf16 in shared memory as the B
//     operand);
//   * warps 2-5 (query tile 0) and 6-9 (query tile 1), one row per thread,
//     turn scores into probabilities with the final lse; a warpgroup frees its
//     score buffer as soon as it has read it (so the next QK runs under its
//     exponentials), reads back the column sums of its previous tile (lane l
//     of quadrant q takes column 32q + l) just before overwriting its P tile,
//     and adds them into the output of the entry's token with one atomic each.
//     The two warpgroups keep the tensor pipe fed while either one waits.
// Every wait is bounded; on time-out the CTA records AKV_ERR_DEVICE_TIMEOUT.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "akv_internal.h"
#include "sm100_ptx.cuh"

namespace akv {
namespace {

constexpr int kThreads = 320;  // producer, MMA, 2 x 4 softmax warps
constexpr int kKeys = 128;
constexpr int kRows = 128;
constexpr int kRing = 2;
constexpr int kMaxRuns = 8;
constexpr uint32_t kTmemCols = 512;  // S_0, S_1, D_0, D_1 (128 columns each)
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr int32_t kErrTimeout = 7;
constexpr int32_t kErrDevice = 8;

template <int D>
struct MLayout {
  static constexpr int kBlocks = D / 64;
  static constexpr uint32_t kBlockBytes = 128 * 128;
  static constexpr uint32_t kTile = kBlocks * kBlockBytes;
  static constexpr uint32_t kQ = 0;                        // two Q tiles
  static constexpr uint32_t kSlot = kQ + 2 * kTile;        // K ring
  static constexpr uint32_t kP = kSlot + kRing * kTile;    // one probability tile per query tile
  static constexpr uint32_t kPTile = 2 * kBlockBytes;      // 2 x 64-key blocks
  static constexpr uint32_t kOnes = kP + 2 * kPTile;       // one 128 x 64 block of bf16 ones
  static constexpr uint32_t kColE = kOnes + kBlockBytes;   // int32 [2 query tiles][2 buffers][128]
  static constexpr uint32_t kBars = kColE + 2 * 2 * 128 * 4;
  static constexpr uint32_t kBytes = kBars + 256;
};

enum MBar {
  kMQ = 0,
  kMFull0,
  kMEmpty0 = kMFull0 + kRing,
  kMS0 = kMEmpty0 + kRing,  // + query tile
  kMSFree0 = kMS0 + 2,      // + query tile, 128 arrivals
  kMPFull0 = kMSFree0 + 2,  // + query tile, 128 arrivals
  kMD0 = kMPFull0 + 2,      // + query tile
  kMFin = kMD0 + 2,
  kMNumBars
};
static_assert(kMNumBars * 8 + 8 <= 256, "barrier area");

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

// K tiles [t0, t0 + n) of this CTA; na / nb of them are read by query tile 0 / 1.
struct MassRange {
  int t0, na, nb, n;
};
__device__ __forceinline__ MassRange mass_range(const AttnWork& w) {
  const int na = max(0, min(w.n_a, w.t1) - w.t0), nb = max(0, min(w.n_b, w.t1) - w.t0);
  return MassRange{w.t0, na, nb, max(na, nb)};
}

// ---------------------------------------------------------------- producer
template <int D>
__device__ void m_produce(const MassParams& p, const AttnWork& w, const AttnSeg& seg, uint32_t sbase,
                          volatile int* abort_flag) {
  using L = MLayout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int G = p.group, tpt = kRows / G, rpt = kKeys / p.page;
  const MassRange rg = mass_range(w);
  const int n = rg.n;
  const int n_q = rg.nb > 0 ? 2 : 1;
  ptx::mbar_arrive_expect_tx(bar(kMQ), n_q * L::kTile);
  for (int t = 0; t < n_q; ++t)
    for (int kb = 0; kb < L::kBlocks; ++kb)
      ptx::tma_load_3d(sbase + L::kQ + t * L::kTile + kb * L::kBlockBytes, &p.q_map, bar(kMQ), kb * 64, w.kvh * G,
                       seg.q_row0 + (w.qt0 + t) * tpt);
  const int layer_base = p.layer * p.n_pages;
  const int first = p.runs[seg.run_off].kp;
  int kpg[kMaxRuns], nkp[kMaxRuns];
  auto fetch = [&](int j, int (&kk)[kMaxRuns]) {  // K pages of local tile j's runs, one tile ahead
#pragma unroll
    for (int g = 0; g < kMaxRuns; ++g) {
      const int ri = (rg.t0 + j) * rpt + g;
      kk[g] = layer_base + ((g < rpt && ri < seg.n_runs) ? p.runs[seg.run_off + ri].kp : first);
    }
  };
  fetch(0, kpg);
  int armed[kRing] = {};
  bool ok = true;
  for (int j = 0; j < n; ++j) {
    const int slot = j % kRing, use = j / kRing;
    if (j + 1 < n) fetch(j + 1, nkp);
    if (use >= 1 && !(ok = ptx::mbar_wait(bar(kMEmpty0 + slot), (use - 1) & 1, abort_flag, kWaitLimitNs))) break;
    const uint32_t dst = sbase + L::kSlot + slot * L::kTile;
    ptx::mbar_arrive_expect_tx(bar(kMFull0 + slot), L::kTile);
    bool cons = true;
#pragma unroll
    for (int g = 1; g < kMaxRuns; ++g) cons = cons && (g >= rpt || kpg[g] == kpg[0] + g);
    if (cons) {
#pragma unroll
      for (int kb = 0; kb < L::kBlocks; ++kb)
        ptx::tma_load_4d(dst + kb * L::kBlockBytes, &p.k_tile_map, bar(kMFull0 + slot), kb * 64, 0, w.kvh, kpg[0]);
    } else {
#pragma unroll
      for (int g = 0; g < kMaxRuns; ++g) {
        if (g >= rpt) break;
#pragma unroll
        for (int kb = 0; kb < L::kBlocks; ++kb)
          ptx::tma_load_4d(dst + kb * L::kBlockBytes + g * p.page * 128, &p.k_map, bar(kMFull0 + slot), kb * 64, 0,
                           w.kvh, kpg[g]);
      }
    }
    armed[slot] = use + 1;
#pragma unroll
    for (int g = 0; g < kMaxRuns; ++g) kpg[g] = nkp[g];
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 0, 0);
    *abort_flag = 1;
  }
  ptx::mbar_wait_drain(bar(kMQ), 0, kDrainLimitNs);
#pragma unroll
  for (int s = 0; s < kRing; ++s)
    if (armed[s]) ptx::mbar_wait_drain(bar(kMFull0 + s), (armed[s] - 1) & 1, kDrainLimitNs);
}

// --------------------------------------------------------------------- MMA
// Per K tile j, for each query tile t that reads it: S_t(j) = Q_t K_j^T once
// t's softmax has read S_t(j-1); then, for each t whose probabilities of tile
// j - 1 are in shared memory, D_t = ones P_t(j-1).  D_t and P_t have one
// buffer each: P_t(j-1) is written only after t's softmax has read D_t(j-2),
// so the sum MMA of j - 1 never overwrites unread sums.
template <int D>
__device__ void m_mma(const MassParams& p, const AttnWork& w, uint32_t sbase, uint32_t tmem, volatile int* abort_flag) {
  using L = MLayout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  constexpr uint32_t idesc_qk = ptx::idesc_bf16(kRows, kKeys, false);
  constexpr uint32_t idesc_sum = ptx::idesc_bf16(kRows, kKeys, true);  // B = P, keys (N) contiguous
  const MassRange rg = mass_range(w);
  const int nt[2] = {rg.na, rg.nb};
  const int n = rg.n;
  const uint64_t ones = ptx::smem_desc(sbase + L::kOnes, 16, 1024);
  bool ok = ptx::mbar_wait(bar(kMQ), 0, abort_flag, kWaitLimitNs);
  for (int j = 0; j <= n && ok; ++j) {
    if (j < n) {
      const int slot = j % kRing;
      if (!(ok = ptx::mbar_wait(bar(kMFull0 + slot), (j / kRing) & 1, abort_flag, kWaitLimitNs))) break;
      const uint64_t kd = ptx::smem_desc(sbase + L::kSlot + slot * L::kTile, 16, 1024);
#pragma unroll 1
      for (int t = 0; t < 2 && ok; ++t) {
        if (j >= nt[t]) continue;
        if (j >= 1 && !(ok = ptx::mbar_wait(bar(kMSFree0 + t), (j - 1) & 1, abort_flag, kWaitLimitNs))) break;
        ptx::tc_fence_after();
        const uint64_t qd = ptx::smem_desc(sbase + L::kQ + t * L::kTile, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * L::kBlockBytes + (ks & 3) * 32;
          ptx::mma_bf16(tmem + 128u * t, ptx::desc_advance(qd, off), ptx::desc_advance(kd, off), idesc_qk, ks > 0);
        }
        ptx::mma_commit(bar(kMS0 + t));
      }
      if (!ok) break;
      ptx::mma_commit(bar(kMEmpty0 + slot));
    }
    if (j >= 1) {
#pragma unroll 1
      for (int t = 0; t < 2 && ok; ++t) {
        if (j - 1 >= nt[t]) continue;
        if (!(ok = ptx::mbar_wait(bar(kMPFull0 + t), (j - 1) & 1, abort_flag, kWaitLimitNs))) break;
        ptx::tc_fence_after();
        const uint64_t pd = ptx::smem_desc(sbase + L::kP + t * L::kPTile, L::kBlockBytes, 1024);
#pragma unroll
        for (int ks = 0; ks < kRows / 16; ++ks)  // 16 probability rows per step; every A element is 1
          ptx::mma_bf16(tmem + 256u + 128u * t, ptx::desc_advance(ones, (ks & 3) * 32),
                        ptx::desc_advance(pd, ks * 16 * 128), idesc_sum, ks > 0);
        ptx::mma_commit(bar(kMD0 + t));
      }
    }
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 1, 0);
    *abort_flag = 1;
  }
  ptx::mma_commit(bar(kMFin));
  ptx::mbar_wait_drain(bar(kMFin), 0, kDrainLimitNs);
}

// ----------------------------------------------------------------- softmax
// Warpgroup t, thread = row r = TMEM lane r: probabilities of its row with the
// final lse, bf16 into t's shared P tile (128-byte swizzle, keys contiguous);
// thread r also owns key column r when the column sums come back.
template <int D>
__device__ void m_softmax(const MassParams& p, const AttnWork& w, const AttnSeg& seg, int t, uint8_t* smem,
                          uint32_t sbase, uint32_t tmem, volatile int* abort_flag) {
  using L = MLayout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const MassRange rg = mass_range(w);
  const int n = t == 0 ? rg.na : rg.nb;
  const int bar_id = 1 + t;  // named barrier of this warpgroup
  const int quad = (threadIdx.x / 32) & 3, lane = threadIdx.x % 32;
  const int r = quad * 32 + lane;
  const uint32_t lane_addr = uint32_t(quad * 32) << 16;
  const uint32_t tS = tmem + 128u * t, tD = tmem + 256u + 128u * t;
  const int G = p.group, tpt = kRows / G, rpt = kKeys / p.page;
  const int qi = (w.qt0 + t) * tpt + r / G, g = r % G;
  const bool row_valid = qi < seg.q_len;
  const int lim = seg.kv_len - seg.q_len + (row_valid ? qi : seg.q_len - 1);
  // log2-domain normaliser of this row; rows past the segment's queries contribute nothing
  const float lse2 = row_valid ? p.lse[int64_t(seg.q_row0 + qi) * p.hq + int64_t(w.kvh) * G + g] * 1.4426950408889634f
                               : INFINITY;
  const float2 sl2v = make_float2(p.scale_log2, p.scale_log2), neg = make_float2(-lse2, -lse2);
  int* const colE_base = reinterpret_cast<int*>(smem + L::kColE) + 256 * t;  // two buffers, by tile parity
  int* colE = colE_base;
  uint8_t* P = smem + L::kP + t * L::kPTile;
  int page_shift = 4;
  while ((1 << page_shift) < p.page) ++page_shift;
  const int sl_own = r & (p.page - 1);
  const int2* run_le = reinterpret_cast<const int2*>(p.runs + seg.run_off);
  int2 run_cur = make_int2(0, 0);
  if (rg.t0 * rpt + (r >> page_shift) < seg.n_runs) run_cur = run_le[2 * (rg.t0 * rpt + (r >> page_shift)) + 1];
  bool ok = true;
  // token of key column r of the previous tile (-1: no entry); its index is loaded a tile
  // before the column sums need it, off the path that releases the next P tile
  int tok_prev = -1;
  // column sums of tile jj come back in D_t: lane l of quadrant q reads column 32q + l
  auto take_sums = [&](int jj) {
    ok = ptx::mbar_wait(bar(kMD0 + t), jj & 1, abort_flag, kWaitLimitNs);
    if (!ptx::bar_red_and(bar_id, 128, ok)) return false;
    ptx::tc_fence_after();
    uint32_t v[32];
    ptx::tmem_load32(tD + lane_addr + quad * 32, v);
    float mine = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) mine = lane == k ? __uint_as_float(v[k]) : mine;
    if (tok_prev >= 0) atomicAdd(p.mass + seg.mass_off + tok_prev, mine);
    return true;
  };
  // probabilities of 64 scores, packed as bf16 pairs
  auto probs = [&](uint32_t (&u)[64], bool need_mask, int h, uint32_t (&pk)[32]) {
    const int4* ce4 = reinterpret_cast<const int4*>(colE);
    if (need_mask) {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int4 e4 = ce4[h * 16 + c];
        if (e4.x > lim) u[4 * c + 0] = 0xff800000u;
        if (e4.y > lim) u[4 * c + 1] = 0xff800000u;
        if (e4.z > lim) u[4 * c + 2] = 0xff800000u;
        if (e4.w > lim) u[4 * c + 3] = 0xff800000u;
      }
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float2 x = __ffma2_rn(make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])), sl2v, neg);
      pk[c] = pack_bf16(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
    }
  };
  auto store = [&](int h, const uint32_t (&pk)[32]) {
    uint8_t* rowp = P + h * L::kBlockBytes + r * 128;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
      *reinterpret_cast<uint4*>(rowp + ((c8 ^ (r & 7)) << 4)) =
          make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
  };
  for (int j = 0; j < n && ok; ++j) {
    // Entry and token of key column r of tile j need no score, so they are
    // formed before S is waited for (the token lookup's latency hides behind
    // the wait); the entries go to the buffer of this tile's parity: the other
    // buffer may still be read by a thread finishing tile j - 1.
    colE = colE_base + (j & 1) * 128;
    int e = INT_MAX;  // entry index of key column r of tile j
    int tok = -1;     // its logical token
    {
      const int lo = run_cur.x & 0xffff, hi = run_cur.x >> 16;
      if (sl_own >= lo && sl_own < hi) e = run_cur.y + (sl_own - lo);
      if (e != INT_MAX) tok = __ldg(p.ent_tok + seg.ent_off + e);
      colE[r] = e;
      const int ri = (rg.t0 + j + 1) * rpt + (r >> page_shift);
      run_cur = ri < seg.n_runs ? run_le[2 * ri + 1] : make_int2(0, 0);
    }
    ok = ptx::mbar_wait(bar(kMS0 + t), j & 1, abort_flag, kWaitLimitNs);
    // One barrier per tile: every thread's S arrived and every column has an
    // entry; only when that fails does a second one tell a time-out from masking.
    const bool all_valid = ptx::bar_red_and(bar_id, 128, ok && e != INT_MAX);
    if (!all_valid && !ptx::bar_red_and(bar_id, 128, ok)) {
      ok = false;
      break;
    }
    ptx::tc_fence_after();
    const bool need_mask = !all_valid || colE[kKeys - 1] > lim;
    uint32_t pk0[32], pk1[32];
    {
      uint32_t u[64];
      ptx::tmem_load64(tS + lane_addr, u);
      probs(u, need_mask, 0, pk0);
    }
    {
      uint32_t u[64];
      ptx::tmem_load64(tS + lane_addr + 64, u);
      // S_t is read: the next QK of this query tile may overwrite it
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(kMSFree0 + t));
      probs(u, need_mask, 1, pk1);
    }
    // the sums of tile j - 1 are read before its P tile is overwritten
    if (j >= 1 && !(ok = take_sums(j - 1))) break;
    store(0, pk0);
    store(1, pk1);
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(bar(kMPFull0 + t));
    tok_prev = tok;
  }
  if (ok && n >= 1) ok = take_sums(n - 1);
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 2 + t, 0);
    *abort_flag = 1;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_mass_kernel(const __grid_constant__ MassParams p, int smem_bytes) {
  using L = MLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  uint8_t* smem = reinterpret_cast<uint8_t*>((raw + 1023) & ~uintptr_t(1023));
  if (smem + L::kBytes > smem_raw + smem_bytes) {
    if (threadIdx.x == 0) raise_error(p.err, kErrDevice, blockIdx.x, int(raw & 1023), 1);
    return;
  }
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + L::kBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBars + 8 * kMNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBars + 8 * kMNumBars + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
#ifdef AKV_CHECKED
  {  // the whole CTA returns together, before any barrier or TMEM use
    const bool ok = int(blockIdx.x) < p.n_work && p.work[blockIdx.x].kvh >= 0 &&
                    p.work[blockIdx.x].kvh < p.hq / p.group &&
                    attn_item_ok(p.work[blockIdx.x], p.segs, p.runs, p.n_segs, p.n_runs, p.n_q_rows, p.n_pages,
                                 p.page, int(threadIdx.x), int(blockDim.x));
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) report_device_error(p.err, 12, int(blockIdx.x), 0);
      return;
    }
  }
#endif
  const AttnWork w = p.work[blockIdx.x];
  const AttnSeg seg = p.segs[w.seg];
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMNumBars; ++i) {
      const bool many = (i >= kMSFree0 && i < kMSFree0 + 2) || (i >= kMPFull0 && i < kMPFull0 + 2);
      ptx::mbar_init(bars + 8u * i, many ? 128 : 1);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  // the all-ones A operand of the column-sum MMA (bf16 1.0 = 0x3f80)
  for (uint32_t i = threadIdx.x; i < L::kBlockBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L::kOnes)[i] = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
  ptx::fence_proxy_async_smem();
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&p.q_map);
    ptx::prefetch_tensormap(&p.k_map);
    ptx::prefetch_tensormap(&p.k_tile_map);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0) {
    if (lane == 0) m_produce<D>(p, w, seg, sbase, abort_flag);
  } else if (warp == 1) {
    if (lane == 0) m_mma<D>(p, w, sbase, tmem, abort_flag);
  } else {
    m_softmax<D>(p, w, seg, warp < 6 ? 0 : 1, smem, sbase, tmem, abort_flag);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_variant(const MassParams& p, cudaStream_t st) {
  const int smem = int(MLayout<D>::kBytes) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_mass_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_mass_kernel<D><<<p.n_work, kThreads, smem, st>>>(p, smem);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_mass(const MassParams& p, int dim, cudaStream_t st) {
  if (p.n_work <= 0) return cudaSuccess;
  if (dim == 64) return launch_variant<64>(p, st);
  if (dim == 128) return launch_variant<128>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace akv
