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
//   * warps 2-5 (tile A) and 6-9 (tile B) run the online softmax, one thread
//     per row = one TMEM lane: a whole score row comes in with one 128-column
//     TMEM load, row max and row sum need no shuffles, O is rescaled lazily in
//     TMEM (only when the running max grows by more than 2^8), and P (bf16) is
//     written back into the S columns already consumed, where the next PV MMA
//     reads it as its TMEM A operand (the MMA thread issues that PV before the
//     QK that overwrites S, and one thread's MMAs execute in issue order).
//     While one warpgroup computes exponentials the tensor core runs the other
//     tile's MMAs;
//   * every wait is bounded (p.wait_ns, 4 s unless a test lowers it); on
//     time-out the CTA records AKV_ERR_DEVICE_TIMEOUT in the device error
//     word, drains its copies and MMAs, frees TMEM, exits.
#include <cuda_bf16.h>

#include <climits>
#include <cstdint>

#include "akv_internal.h"
#include "attn_merge.cuh"
#include "rope_rot.cuh"
#include "sm100_ptx.cuh"

namespace akv {
namespace {

constexpr int kThreads = 320;       // producer, MMA, 2 x 4 softmax warps
constexpr int kThreadsFused = 384;  // + 2 warps rotating K tiles in shared memory
constexpr int kRotThreads = 64;
constexpr int kTileKeys = 128;
constexpr int kRows = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr int32_t kErrTimeout = 7;  // AKV_ERR_DEVICE_TIMEOUT
constexpr int32_t kErrDevice = 8;   // AKV_ERR_DEVICE
constexpr int kSlots = 4;
constexpr int kMaxRuns = 8;  // runs per 128-key tile: 128 / page, page >= 16

template <int D>
struct Layout {
  static constexpr int kBlocks = D / 64;              // 64-element (128-byte) column blocks
  static constexpr uint32_t kBlockBytes = 128 * 128;  // 128 rows x 128 bytes
  static constexpr uint32_t kTile = kBlocks * kBlockBytes;
  static constexpr uint32_t kQ = 0;                          // Q_A, Q_B
  static constexpr uint32_t kSlot = kQ + 2 * kTile;          // K/V slots
  static constexpr uint32_t kColE = kSlot + kSlots * kTile;  // int32 [2 tiles][2 buffers][128]: entry per key column
  static constexpr uint32_t kBars = kColE + 2 * 2 * 128 * 4;
  static constexpr uint32_t kBytes = kBars + 256;
};

enum Bar {
  kBarQ = 0,
  kBarFull0,  // + slot
  kBarEmpty0 = kBarFull0 + kSlots,
  kBarS0 = kBarEmpty0 + kSlots,  // + tile
  kBarP0 = kBarS0 + 2,
  kBarO0 = kBarP0 + 2,
  kBarQFree = kBarO0 + 2,  // committed after a unit's last QK MMA: Q buffers may be reloaded
  kBarFin,
  kBarRdy0,  // + slot, fused rotation only: the slot's tile is ready for the MMA (K rotated)
  kNumBars = kBarRdy0 + kSlots
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
// Units run back to back: the K/V stream position ld continues across units
// (K_j of a unit is ld0 + 2j, V_j is ld0 + 2j + 1), and a unit's Q tiles
// are loaded once the previous unit's last QK MMA has released the Q buffers.
template <int D>
__device__ void produce(const AttnParams& p, int u0, int u1, uint32_t sbase, volatile int* abort_flag) {
  using L = Layout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int G = p.group, tpt = kRows / G, rpt = kTileKeys / p.page;
  const int layer_base = p.layer * p.n_pages;
  int armed[kSlots] = {0, 0, 0, 0};
  int ld0 = 0, q_loads = 0;
  bool ok = true, capped = false;
  // Test hook: with p.load_cap >= 0 the producer issues at most that many
  // K/V tile copies and then stops (no error of its own); the waits of the
  // MMA thread and the softmax on the missing tiles then run out after
  // p.wait_ns and report AKV_ERR_DEVICE_TIMEOUT.
  int n_copies = 0;
  for (int u = u0; u < u1 && ok && !capped; ++u) {
    const AttnWork w = p.work[u];
    const AttnSeg seg = p.segs[w.seg];
    // KV tiles [t0, t1) of this unit; local tile j is global tile t0 + j
    const int span = w.t1 - w.t0;
    const int n_max = max(min(max(w.n_a - w.t0, 0), span), min(max(w.n_b - w.t0, 0), span));
    const int q_tok0 = seg.q_row0 + w.qt0 * tpt;
    if (u > u0 && !(ok = ptx::mbar_wait(bar(kBarQFree), (u - u0 - 1) & 1, abort_flag, p.wait_ns))) break;
    ptx::mbar_arrive_expect_tx(bar(kBarQ), (w.n_b > 0 ? 2 : 1) * L::kTile);
    for (int t = 0; t < (w.n_b > 0 ? 2 : 1); ++t)
      for (int kb = 0; kb < L::kBlocks; ++kb)
        ptx::tma_load_3d(sbase + L::kQ + t * L::kTile + kb * L::kBlockBytes, &p.q_map, bar(kBarQ), kb * 64,
                         w.kvh * G, q_tok0 + t * tpt);
    ++q_loads;
    // Pages of a tile's runs (K and V pages of run g).  They are fetched one
    // tile ahead, so the run-table loads are in flight while the producer
    // waits for ring slots instead of sitting between TMA issues.  Past the
    // last run the segment's first page stands in (finite values, masked out).
    const int2 first = *reinterpret_cast<const int2*>(p.runs + seg.run_off);
    int kpg[kMaxRuns], vpg[kMaxRuns], nkp[kMaxRuns], nvp[kMaxRuns];
    auto fetch = [&](int j, int (&kk)[kMaxRuns], int (&vv)[kMaxRuns]) {
#pragma unroll
      for (int g = 0; g < kMaxRuns; ++g) {
        const int ri = (w.t0 + j) * rpt + g;
        int2 kv = first;
        if (g < rpt && ri < seg.n_runs) kv = *reinterpret_cast<const int2*>(p.runs + seg.run_off + ri);
        kk[g] = layer_base + kv.x;
        vv[g] = layer_base + kv.y;
      }
    };
    // A tile whose runs sit on consecutive pages loads with one copy per
    // 64-column block (the tile map's box spans 128 / page pages).
    auto consecutive = [&](const int (&pg)[kMaxRuns]) {
      bool c = true;
#pragma unroll
      for (int g = 1; g < kMaxRuns; ++g) c = c && (g >= rpt || pg[g] == pg[0] + g);
      return c;
    };
    fetch(0, kpg, vpg);
    for (int l = 0; l < 2 * n_max; ++l) {
      if (p.load_cap >= 0 && n_copies >= p.load_cap) {
        capped = true;
        break;
      }
      ++n_copies;
      const int ld = ld0 + l, j = l >> 1, is_v = l & 1, slot = ld % kSlots, use = ld / kSlots;
      if (!is_v && j + 1 < n_max) fetch(j + 1, nkp, nvp);
      if (use >= 1 && !ptx::mbar_wait(bar(kBarEmpty0 + slot), (use - 1) & 1, abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t dst = sbase + L::kSlot + slot * L::kTile;
      const CUtensorMap* map = is_v ? &p.v_map : &p.k_map;
      ptx::mbar_arrive_expect_tx(bar(kBarFull0 + slot), L::kTile);
      if (consecutive(is_v ? vpg : kpg)) {
        const CUtensorMap* tmap = is_v ? &p.v_tile_map : &p.k_tile_map;
        const int pg = is_v ? vpg[0] : kpg[0];
#pragma unroll
        for (int kb = 0; kb < L::kBlocks; ++kb)
          ptx::tma_load_4d(dst + kb * L::kBlockBytes, tmap, bar(kBarFull0 + slot), kb * 64, 0, w.kvh, pg);
      } else {
#pragma unroll
        for (int g = 0; g < kMaxRuns; ++g) {
          if (g >= rpt) break;
          const int pg = is_v ? vpg[g] : kpg[g];
#pragma unroll
          for (int kb = 0; kb < L::kBlocks; ++kb)
            ptx::tma_load_4d(dst + kb * L::kBlockBytes + g * p.page * 128, map, bar(kBarFull0 + slot), kb * 64, 0,
                             w.kvh, pg);
        }
      }
      armed[slot] = use + 1;
      if (is_v) {
#pragma unroll
        for (int g = 0; g < kMaxRuns; ++g) {
          kpg[g] = nkp[g];
          vpg[g] = nvp[g];
        }
      }
    }
    ld0 += 2 * n_max;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 0, 0);
    *abort_flag = 1;
  }
  // Drain: every copy issued here has landed before the CTA may exit.
  if (q_loads) ptx::mbar_wait_drain(bar(kBarQ), (q_loads - 1) & 1, kDrainLimitNs);
#pragma unroll
  for (int s = 0; s < kSlots; ++s)
    if (armed[s]) ptx::mbar_wait_drain(bar(kBarFull0 + s), (armed[s] - 1) & 1, kDrainLimitNs);
}

// --------------------------------------------------------------------- MMA
// Per KV tile j and query tile T: O_T += P_T(j-1) V_{j-1} (once P_T(j-1) is
// written), then S_T(j) = Q_T K_j^T, then one commit to S_T's barrier.  Slots
// are released (commit to their empty barrier) after their last reader.
// Across units the S/P phase of tile T continues from the previous units
// (cs[T] events so far).  The first PV of a unit overwrites O_T; it waits for
// P_T(0) of that unit, which the softmax threads arrive only after reading
// out the previous unit's O_T, so O_T is free by then.
template <int D, bool kFused>
__device__ void issue_mma(const AttnParams& p, int u0, int u1, uint32_t sbase, uint32_t tmem,
                          volatile int* abort_flag) {
  using L = Layout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  constexpr uint32_t idesc_qk = ptx::idesc_bf16(kRows, kTileKeys, false);
  constexpr uint32_t idesc_pv = ptx::idesc_bf16(kRows, D, true);
  auto slot_of = [](int ld) { return ld % kSlots; };
  auto full_parity = [](int ld) { return (ld / kSlots) & 1; };
  // a slot's tile may be read once TMA has landed it (and, with fused rotation, once K is rotated)
  auto ready_bar = [&](int ld) { return bar((kFused ? kBarRdy0 : kBarFull0) + ld % kSlots); };
  int ld0 = 0, cs0 = 0, cs1 = 0;
  bool ok = true, issued = false;  // a commit is only issued after this thread's first MMA
  const uint64_t qd0 = ptx::smem_desc(sbase + L::kQ, 16, 1024), qd1 = ptx::smem_desc(sbase + L::kQ + L::kTile, 16, 1024);
  for (int u = u0; u < u1 && ok; ++u) {
    const AttnWork w = p.work[u];
    const int span = w.t1 - w.t0;  // local tile counts of this KV range
    const int nt0 = min(max(w.n_a - w.t0, 0), span), nt1 = min(max(w.n_b - w.t0, 0), span);
    const int n_max = max(nt0, nt1);
    if (!(ok = ptx::mbar_wait(bar(kBarQ), (u - u0) & 1, abort_flag, p.wait_ns))) break;
    for (int j = 0; j <= n_max && ok; ++j) {
      bool v_ready = false;
      // K_j is waited for before P_A(j-1): the thread would wait for P_A
      // anyway, and a wait between PV_A and QK_A idles the tensor pipe.
      if (j < n_max) {
        const int ld = ld0 + 2 * j;
        ok = ptx::mbar_wait(ready_bar(ld), full_parity(ld), abort_flag, p.wait_ns);
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int nt = t ? nt1 : nt0, cs = t ? cs1 : cs0;
        const uint32_t tS = tmem + 128u * t, tO = tmem + 256u + 128u * t;
        if (ok && j >= 1 && j - 1 < nt) {
          if (!v_ready) {
            const int ld = ld0 + 2 * (j - 1) + 1;
            ok = ptx::mbar_wait(ready_bar(ld), full_parity(ld), abort_flag, p.wait_ns);
            v_ready = true;
          }
          if (ok) ok = ptx::mbar_wait(bar(kBarP0 + t), (cs + j - 1) & 1, abort_flag, p.wait_ns);
          if (ok) {
            ptx::tc_fence_after();
            const uint64_t vd = ptx::smem_desc(sbase + L::kSlot + slot_of(ld0 + 2 * (j - 1) + 1) * L::kTile,
                                               L::kBlockBytes, 1024);
            // P: 16 keys = 8 packed TMEM columns per step; V: 16 key rows = 2 KiB per step
            ptx::mma_bf16_tmem_a(tO, tS, vd, idesc_pv, j > 1);
            issued = true;
#pragma unroll
            for (int ks = 1; ks < kTileKeys / 16; ++ks)
              ptx::mma_bf16_tmem_a(tO, tS + 8u * ks, ptx::desc_advance(vd, ks * 16 * 128), idesc_pv, 1);
            if (j - 1 == nt - 1) ptx::mma_commit(bar(kBarO0 + t));
          }
        }
        if (ok && j < nt) {
          ptx::tc_fence_after();
          if (ok) {
            const uint64_t kd = ptx::smem_desc(sbase + L::kSlot + slot_of(ld0 + 2 * j) * L::kTile, 16, 1024);
            const uint64_t qd = t ? qd1 : qd0;
            // 16 head dims per step: 32 bytes inside a 128-byte swizzle row, a new block every 4 steps
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * L::kBlockBytes + (ks & 3) * 32;
              ptx::mma_bf16(tS, ptx::desc_advance(qd, off), ptx::desc_advance(kd, off), idesc_qk, ks > 0);
            }
            issued = true;
            ptx::mma_commit(bar(kBarS0 + t));
          }
        }
      }
      if (!ok) break;
      if (j >= 1) ptx::mma_commit(bar(kBarEmpty0 + slot_of(ld0 + 2 * (j - 1) + 1)));  // V_{j-1} done
      if (j < n_max) ptx::mma_commit(bar(kBarEmpty0 + slot_of(ld0 + 2 * j)));        // K_j done
      if (j == n_max - 1) ptx::mma_commit(bar(kBarQFree));                           // last QK of the unit
    }
    cs0 += nt0;
    cs1 += nt1;
    ld0 += 2 * n_max;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 1, 0);
    *abort_flag = 1;
  }
  // Every MMA issued above has completed before TMEM is released.
  if (issued) {
    ptx::mma_commit(bar(kBarFin));
    ptx::mbar_wait_drain(bar(kBarFin), 0, kDrainLimitNs);
  }
}

// ------------------------------------------------------------ K rotation
// Fused rotation ([AKV-blog] section 4: rotate keys on their way to the
// tensor core instead of writing transient position versions to HBM).  Two
// warps take every ring slot in stream order after TMA has filled it; for a
// K tile they rotate each key row whose run carries a pending shift by
// R(delta * theta_j) in shared memory, with the same arithmetic and angle
// table as repos_rotate (so the bits equal the materialised key), then make
// the writes visible to the tensor core and arrive on the slot's ready
// barrier, which the MMA thread waits on instead of the TMA barrier.
template <int D>
__device__ void rotate_k(const AttnParams& p, int u0, int u1, uint32_t sbase, uint8_t* smem,
                         volatile int* abort_flag) {
  using L = Layout<D>;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int i = int(threadIdx.x) - kThreads;  // 0 .. kRotThreads - 1
  const int rpt = kTileKeys / p.page;
  int page_shift = 4;
  while ((1 << page_shift) < p.page) ++page_shift;
  int ld0 = 0;
  bool ok = true;
  for (int u = u0; u < u1 && ok; ++u) {
    const AttnWork w = p.work[u];
    const AttnSeg seg = p.segs[w.seg];
    const int span = w.t1 - w.t0;
    const int n_max = max(min(max(w.n_a - w.t0, 0), span), min(max(w.n_b - w.t0, 0), span));
    for (int l = 0; l < 2 * n_max; ++l) {
      const int ld = ld0 + l, slot = ld % kSlots;
      if (!(ok = ptx::mbar_wait(bar(kBarFull0 + slot), (ld / kSlots) & 1, abort_flag, p.wait_ns))) break;
      if ((l & 1) == 0) {
        uint8_t* tile = smem + L::kSlot + slot * L::kTile;
#pragma unroll 1
        for (int rr = i; rr < kTileKeys; rr += kRotThreads) {
          const int ri = (w.t0 + (l >> 1)) * rpt + (rr >> page_shift);
          const int didx = ri < seg.n_runs ? p.run_didx[seg.run_off + ri] : -1;
          if (didx < 0) continue;
          const float2* cs = p.cs + int64_t(didx) * (D / 2);
          auto at = [&](int v) {  // 16-byte vector v of row rr (128-byte swizzle, 64-column blocks)
            return reinterpret_cast<uint4*>(tile + (v >> 3) * L::kBlockBytes + rr * 128 + (((v & 7) ^ (rr & 7)) << 4));
          };
          if (!p.rope_half) {
#pragma unroll 4
            for (int v = 0; v < D / 8; ++v) {  // pairs 4v .. 4v + 3
              uint4* q = at(v);
              const uint4 x = *q;
              const float4 a = __ldg(reinterpret_cast<const float4*>(cs + 4 * v));
              const float4 b = __ldg(reinterpret_cast<const float4*>(cs + 4 * v + 2));
              *q = make_uint4(pack_rot(rot2(x.x, a.x, a.y)), pack_rot(rot2(x.y, a.z, a.w)),
                              pack_rot(rot2(x.z, b.x, b.y)), pack_rot(rot2(x.w, b.z, b.w)));
            }
          } else {
#pragma unroll 2
            for (int v = 0; v < D / 16; ++v) {  // dims 8v .. 8v + 7 pair with dims D/2 + 8v ..
              uint4* qa = at(v);
              uint4* qb = at(v + D / 16);
              const uint4 a = *qa, b = *qb;
              const float4* c4 = reinterpret_cast<const float4*>(cs + 8 * v);
              const float4 c01 = __ldg(c4), c23 = __ldg(c4 + 1), c45 = __ldg(c4 + 2), c67 = __ldg(c4 + 3);
              float2 ya[4], yb[4];
              rot_halves(a.x, b.x, c01.x, c01.y, c01.z, c01.w, ya[0], yb[0]);
              rot_halves(a.y, b.y, c23.x, c23.y, c23.z, c23.w, ya[1], yb[1]);
              rot_halves(a.z, b.z, c45.x, c45.y, c45.z, c45.w, ya[2], yb[2]);
              rot_halves(a.w, b.w, c67.x, c67.y, c67.z, c67.w, ya[3], yb[3]);
              *qa = make_uint4(pack_rot(ya[0]), pack_rot(ya[1]), pack_rot(ya[2]), pack_rot(ya[3]));
              *qb = make_uint4(pack_rot(yb[0]), pack_rot(yb[1]), pack_rot(yb[2]), pack_rot(yb[3]));
            }
          }
        }
        ptx::fence_proxy_async_smem();  // generic-proxy writes -> tensor-core (async proxy) reads
      }
      ptx::mbar_arrive(bar(kBarRdy0 + slot));
    }
    ld0 += 2 * n_max;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 4, 0);
    *abort_flag = 1;
  }
}

// Split part of query tile t, row r: if this CTA drew the item's last ticket,
// merge every part's partial into row r's output.
template <int D>
__device__ __forceinline__ void merge_tile(const AttnParams& p, const AttnWork& w, const AttnSeg& seg, int t, int r) {
  const int G = p.group, tpt = kRows / G;
  const int qi = (w.qt0 + t) * tpt + r / G, g = r % G;
  const bool valid = qi < seg.q_len;
  const int64_t row = int64_t(seg.q_row0 + qi) * p.hq + int64_t(w.kvh) * G + g;
  merge_if_last<D>(p, w, t, r, 1 + t, valid ? static_cast<__nv_bfloat16*>(p.o) + row * D : nullptr,
                   valid && p.lse ? p.lse + row : nullptr);
}

// ----------------------------------------------------------------- softmax
// One warpgroup per query tile t; thread = row r = TMEM lane r.  One unit:
// bit 0 of ph is the parity of the S/P phases of tile t consumed by earlier
// units, bit 1 that of its O phases; both advance here.  Returns false when a
// wait gave up.
template <int D>
__device__ bool softmax_tile(const AttnParams& p, const AttnWork& w, const AttnSeg& seg, int t, uint8_t* smem,
                             uint32_t sbase, uint32_t tmem, volatile int* abort_flag, int& ph) {
  using L = Layout<D>;
  const int n_glob = t == 0 ? w.n_a : w.n_b;
  const int n_t = min(max(n_glob - w.t0, 0), w.t1 - w.t0);  // local tiles of this KV range
  if (n_t == 0) {
    // A split part in which this query tile sees no key: record an empty partial (l = 0).
    if (n_glob > 0 && w.part >= 0) {
      const int r0 = ((threadIdx.x / 32) & 3) * 32 + threadIdx.x % 32;
      p.partial[w.part * partial_floats(2, D) + (int64_t(t) * (D + 2) + D + 1) * 128 + r0] = 0.f;
      p.partial[w.part * partial_floats(2, D) + (int64_t(t) * (D + 2) + D) * 128 + r0] = -INFINITY;
      merge_tile<D>(p, w, seg, t, r0);
    }
    return true;
  }
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int wg_warp = (threadIdx.x / 32 - 2) % 4;
  const int quad = (threadIdx.x / 32) & 3;  // TMEM lane quadrant this warp may access
  const int lane = threadIdx.x % 32;
  const int r = quad * 32 + lane;
  (void)wg_warp;
  const uint32_t lane_addr = uint32_t(quad * 32) << 16;
  const uint32_t tS = tmem + 128u * t, tO = tmem + 256u + 128u * t;
  const int G = p.group, tpt = kRows / G, rpt = kTileKeys / p.page;
  const int t_loc = r / G, g = r % G;
  const int qi = (w.qt0 + t) * tpt + t_loc;  // query index inside the segment
  const bool row_valid = qi < seg.q_len;
  const int lim = seg.kv_len - seg.q_len + (row_valid ? qi : seg.q_len - 1);
  const float sl2 = p.scale_log2;
  const int bar_id = 1 + t;  // named barrier of this warpgroup
  int* colE_base = reinterpret_cast<int*>(smem + L::kColE) + t * 256;  // two buffers, by tile parity
  int page_shift = 4;
  while ((1 << page_shift) < p.page) ++page_shift;
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  const int sl_own = r & (p.page - 1);
  // (lohi, es) of the run holding key column r of the current tile; lo = hi = 0
  // past the segment's last run, so no slot matches
  int2 run_cur = make_int2(0, 0);
  const int2* run_le = reinterpret_cast<const int2*>(p.runs + seg.run_off);
  {
    const int ri0 = w.t0 * rpt + (r >> page_shift);
    if (ri0 < seg.n_runs) run_cur = run_le[2 * ri0 + 1];
  }
  for (int j = 0; j < n_t; ++j) {
    // Entry index of key column r of tile j (INT_MAX: no entry there);
    // columns are (run c / page, slot c % page) of the tile's runs.  It needs
    // no score, so it is formed before S_t(j) is waited for, and the run of
    // the next tile is fetched now so its latency hides behind this tile.  The
    // entries go to the buffer of this tile's parity: the other buffer may
    // still be read by a thread finishing tile j - 1.
    int* colE = colE_base + (j & 1) * 128;
    int e = INT_MAX;
    {
      const int lo = run_cur.x & 0xffff, hi = run_cur.x >> 16;
      if (sl_own >= lo && sl_own < hi) e = run_cur.y + (sl_own - lo);
      colE[r] = e;
      const int ri = (w.t0 + j + 1) * rpt + (r >> page_shift);
      run_cur = ri < seg.n_runs ? run_le[2 * ri + 1] : make_int2(0, 0);
    }
    ok = ptx::mbar_wait(bar(kBarS0 + t), (ph ^ j) & 1, abort_flag, p.wait_ns);
    // One barrier per tile: every thread's S arrived and every column has an
    // entry; only when that fails does a second one tell a time-out from masking.
    const bool all_valid = ptx::bar_red_and(bar_id, 128, ok && e != INT_MAX);
    if (!all_valid && !ptx::bar_red_and(bar_id, 128, ok)) {
      ok = false;
      break;
    }
    ptx::tc_fence_after();
    // With every column valid the entries are consecutive, so the last column
    // holds the tile's largest entry index.
    const bool need_mask = !all_valid || colE[kTileKeys - 1] > lim;
    const int4* ce4 = reinterpret_cast<const int4*>(colE);
    // One pass over the row: the 128 scores are read from TMEM with one load
    // (one wait), the row max is taken (three-input max, two scores per
    // instruction), and P = exp2(s * scale * log2 e - m) is formed with the
    // running max m, packed to bf16 pairs in place (pair c, keys 2c and 2c+1,
    // goes to register c, whose score is already used) and stored with one
    // 64-column store over the S columns, where the PV MMA reads it as its A
    // operand.  m is raised only when the row max exceeds it by more than 2^8
    // (lazy rescale).  The scale-and-shift and the row sum run on float pairs.
    const float2 sl2v = make_float2(sl2, sl2);
    float2 sum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float m_use = m_run, alpha = 1.0f;
    bool resc = false;
    {
      uint32_t u[128];
      ptx::tmem_load128(tS + lane_addr, u);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int4 e4 = ce4[c];
          if (e4.x > lim) u[4 * c + 0] = 0xff800000u;  // -inf
          if (e4.y > lim) u[4 * c + 1] = 0xff800000u;
          if (e4.z > lim) u[4 * c + 2] = 0xff800000u;
          if (e4.w > lim) u[4 * c + 3] = 0xff800000u;
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 32; ++c)
        mx[c & 3] = ptx::max3(mx[c & 3], __uint_as_float(u[4 * c]), __uint_as_float(u[4 * c + 1]));
#pragma unroll
      for (int c = 0; c < 32; ++c)
        mx[c & 3] = ptx::max3(mx[c & 3], __uint_as_float(u[4 * c + 2]), __uint_as_float(u[4 * c + 3]));
      const float mh = fmaxf(ptx::max3(mx[0], mx[1], mx[2]), mx[3]) * sl2;
      if (mh > m_use + 8.0f) {
        alpha = m_use == -INFINITY ? 0.f : ptx::ex2_approx(m_use - mh);
        m_use = mh;
        resc = true;
      }
      const float msub = m_use == -INFINITY ? 0.f : m_use;
      const float2 negm = make_float2(-msub, -msub);
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])), sl2v, negm);
        const float2 pr = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
        sum[c & 1] = __fadd2_rn(sum[c & 1], pr);
        u[c] = pack_bf16(pr.x, pr.y);
      }
      ptx::tmem_store64(tS + lane_addr, u);
    }
    // O_T is stable here (S_T(j) completes after PV_T(j-1)); PV_T(j) waits for P below.
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
    const float rowsum = (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
    l_run = l_run * alpha + rowsum;
    m_run = m_use;
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(kBarP0 + t));
  }
  if (ok) {
    ok = ptx::mbar_wait(bar(kBarO0 + t), (ph >> 1) & 1, abort_flag, p.wait_ns);
    ok = ptx::bar_red_and(bar_id, 128, ok);
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 2 + t, 0);
    *abort_flag = 1;
    return false;
  }
  ph ^= (n_t & 1) | 2;
  ptx::tc_fence_after();
  if (w.part >= 0) {
    // Split part: unnormalised O, running max and sum for the combine kernel,
    // column-major per tile so a warp writes consecutive rows.
    float* base = p.partial + w.part * partial_floats(2, D) + int64_t(t) * (D + 2) * 128 + r;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      ptx::tmem_load32(tO + lane_addr + c * 32, o);
#pragma unroll
      for (int k = 0; k < 32; ++k) base[int64_t(c * 32 + k) * 128] = __uint_as_float(o[k]);
    }
    base[int64_t(D) * 128] = m_run;
    base[int64_t(D + 1) * 128] = l_run;
    ptx::tc_fence_before();
    merge_tile<D>(p, w, seg, t, r);
    return true;
  }
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
  return true;
}

template <int D>
__device__ void softmax_units(const AttnParams& p, int u0, int u1, int t, uint8_t* smem, uint32_t sbase,
                              uint32_t tmem, volatile int* abort_flag) {
  int ph = 0;
  for (int u = u0; u < u1; ++u) {
    const AttnWork w = p.work[u];
    const AttnSeg seg = p.segs[w.seg];
    if (!softmax_tile<D>(p, w, seg, t, smem, sbase, tmem, abort_flag, ph)) return;
  }
}

template <int D, bool kFused>
__global__ void __launch_bounds__(kFused ? kThreadsFused : kThreads, 1)
    segment_attn_kernel(const __grid_constant__ AttnParams p, int smem_bytes) {
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
  const int u0 = p.cta_units ? p.cta_units[blockIdx.x] : int(blockIdx.x);
  const int u1 = p.cta_units ? p.cta_units[blockIdx.x + 1] : int(blockIdx.x) + 1;
#ifdef AKV_CHECKED
  {  // every thread takes part, so the whole CTA returns together, before any barrier or TMEM use
    bool ok = u0 >= 0 && u0 <= u1 && u1 <= p.n_work;
    for (int u = u0; u < u1 && ok; ++u) {
      const AttnWork w = p.work[u];
      ok = w.kvh >= 0 && w.kvh < p.hq / p.group &&
           attn_item_ok(w, p.segs, p.runs, p.n_segs, p.n_runs, p.n_q_rows, p.n_pages, p.page, int(threadIdx.x),
                        int(blockDim.x));
    }
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) report_device_error(p.err, 10, int(blockIdx.x), u0);
      return;
    }
  }
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      ptx::mbar_init(bars + 8u * i, (i == kBarP0 || i == kBarP0 + 1) ? 128 : i >= kBarRdy0 ? kRotThreads : 1);
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
    ptx::prefetch_tensormap(&p.k_tile_map);
    ptx::prefetch_tensormap(&p.v_tile_map);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) produce<D>(p, u0, u1, sbase, abort_flag);
  } else if (warp == 1) {
    if (lane == 0) issue_mma<D, kFused>(p, u0, u1, sbase, tmem, abort_flag);
  } else if (warp < 10) {
    softmax_units<D>(p, u0, u1, warp < 6 ? 0 : 1, smem, sbase, tmem, abort_flag);
  } else if (kFused) {
    rotate_k<D>(p, u0, u1, sbase, smem, abort_flag);
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

namespace {
template <int D, bool kFused>
cudaError_t launch_variant(const AttnParams& p, int grid, int smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(segment_attn_kernel<D, kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  segment_attn_kernel<D, kFused><<<grid, kFused ? kThreadsFused : kThreads, smem, st>>>(p, smem);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_segment_attn(const AttnParams& p, int dim, cudaStream_t st) {
  if (p.n_work <= 0) return cudaSuccess;
  const int grid = p.cta_units ? p.n_cta : p.n_work;
  const int smem = segment_attn_smem_bytes(dim);
  if (smem < 0) return cudaErrorInvalidValue;
  if (dim == 64) return p.fused ? launch_variant<64, true>(p, grid, smem, st) : launch_variant<64, false>(p, grid, smem, st);
  return p.fused ? launch_variant<128, true>(p, grid, smem, st) : launch_variant<128, false>(p, grid, smem, st);
}

}  // namespace akv
