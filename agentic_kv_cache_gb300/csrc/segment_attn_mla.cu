// segment_batch_attn, MLA variant ([Leyline] "Method": under MLA the cached
// key is a position-free latent -- which also serves as the value -- plus a
// RoPE'd K_pe; 16 query heads share one latent).  What it computes is the
// same as the GQA kernel ([AKV-notes] section 3 "Segment-Batch Attention";
// [AKV-blog] section 2 "The Drop Primitive"): per segment, causal softmax
// attention of its queries over its visible entries, with
//   score = q_latent . c + q_pe . k_pe   (d_qk = 512 + 64)
//   out   = sum_j p_j c_j                (d_v = 512).
//
// GB300 design: a CTA pair (cluster of 2, tcgen05 cta_group::2).  Each CTA
// holds one 128-row query tile (8 tokens x 16 heads) and the pair shares one
// half of the 512 output columns: O for all 512 columns would fill TMEM by
// itself, so each half recomputes S (+53% MMA over the algorithmic count; the
// two halves run as separate pairs).  Every MMA covers the pair's 256 rows
// (M = 256, N = 128) and each CTA supplies half of its B operand: for QK^T the
// 64 keys of its half of the 128-key tile, for PV 64 of the 128 output columns
// of each quarter.  Per SM that halves the key bytes streamed per MMA clock;
// two rings of 16 KiB rounds (QK^T: 3 slots, PV: 2 slots; 80 KiB) sit beside
// the resident 144 KiB Q tile.  TMEM (allocated for the pair): S0, S1
// (double-buffered, P written back over the consumed S columns as bf16 pairs)
// and the 256-column O half.  Warps 0 and 6: TMA producers of the QK^T ring,
// warp 7: of the PV ring (their copies count on the even CTA's barriers);
// warp 1: TMEM allocation and, in the even CTA, the thread issuing the QK^T
// MMAs; warp 8 (even CTA): the thread issuing the PV MMAs; warps 2-5: softmax
// of the CTA's own rows; warps 9-10, with fused rotation only: the K_pe
// rotation of the CTA's key half.  Every wait is bounded.
//
// A pair runs a list of units (persistent schedule: the engine cuts the work
// end to end by the smallest per-pair budget that fits the resident pairs,
// so a unit may be part of an item whose partials the last part merges).  The
// ring positions and the S / P / O phases continue across units; after a
// unit's last QK^T MMA the even CTA commits to both CTAs' Q-free barrier, on
// which each CTA reloads its Q tile for the next unit.  The softmax threads
// signal P of a tile before PV of the previous tile has completed, unless
// their warp rescales O, so the PV thread queues consecutive PVs back to back;
// P and O therefore have one barrier per tile parity (the CTAs of the pair may
// be a tile apart on P).
#include <cuda_bf16.h>

#include <climits>
#include <cstdint>

#include "akv_internal.h"
#include "attn_merge.cuh"
#include "rope_rot.cuh"
#include "sm100_ptx.cuh"

namespace akv {
namespace {

constexpr int kThreads = 352;
constexpr int kRotWarps = 2;  // fused rotation: warps 9 and 10, one K_pe row per lane
constexpr int kKeys = 128;     // keys per KV tile (the pair MMA's N for QK^T)
constexpr int kRows = 128;     // rows per CTA; the pair covers 256
constexpr int kLat = 512;      // latent width
constexpr int kPe = 64;        // K_pe width
constexpr int kQChunks = (kLat + kPe) / 64;  // 9 chunks of the QK contraction
constexpr int kQKRounds = 5;                 // latent chunks in pairs, then K_pe
constexpr int kPVRounds = 2;                 // one per O quarter
// Two rings of 16 KiB slots, one per MMA thread: each ring has one consumer,
// which takes its rounds in order, and no more producers than slots, so a
// wait on a slot's barrier phase can never see the phase of an older use.
constexpr int kQKSlots = 3;     // QK^T rounds, filled by warps 0 and 6 (by position in the tile)
constexpr int kQKProducers = 2;
constexpr int kPVSlots = 2;     // PV rounds, filled by warp 7
static_assert(kQKProducers <= kQKSlots, "a ring needs at least as many slots as producers");
constexpr int kMaxRuns = 8;  // runs per 128-key tile: 128 / page, page >= 16
constexpr uint32_t kQChunk = 128 * 128;      // 128 rows x 64 bf16
constexpr uint32_t kUnit = 64 * 128;         // 64 keys x 64 bf16: one copy
constexpr uint32_t kSlot = 2 * kUnit;        // one round: two copies
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr int32_t kErrTimeout = 7;
constexpr uint16_t kBoth = 0x3;  // CTA mask of the pair

// shared memory layout (bytes)
constexpr uint32_t kQ = 0;                           // 9 chunks of Q
constexpr uint32_t kSlots = kQ + kQChunks * kQChunk;  // QK^T ring, then PV ring (16 KiB slots)
constexpr uint32_t kVSlots = kSlots + kQKSlots * kSlot;
constexpr uint32_t kColE = kVSlots + kPVSlots * kSlot;  // int32[2][128], by tile parity
constexpr uint32_t kBars = kColE + 2 * 128 * 4;
constexpr uint32_t kBytes = kBars + 512;
static_assert(kBytes + 1024 <= 232448, "shared memory");

// Full and Q count both CTAs' bytes and live in the even CTA; Empty, S and O
// are signalled to both CTAs by multicast commits; P (even CTA) collects the
// 256 softmax threads of the pair.  Only the wait on P acquires at cluster
// scope (thread arrivals from the peer); the others are completed by copies
// and commits, whose CTA-scope waits are much cheaper on the producer's and
// the MMA thread's per-unit path.
enum Bar {
  kBarQ = 0,
  kBarFull0,                           // + QK^T slot
  kBarEmpty0 = kBarFull0 + kQKSlots,   // + QK^T slot
  kBarVFull0 = kBarEmpty0 + kQKSlots,  // + PV slot
  kBarVEmpty0 = kBarVFull0 + kPVSlots,
  kBarS0 = kBarVEmpty0 + kPVSlots,  // + S buffer
  kBarP0 = kBarS0 + 2,  // + tile parity (two, so a CTA a tile ahead never completes the other's phase)
  kBarO0 = kBarP0 + 2,  // + tile parity: PV of that tile done (O stable)
  kBarQFree = kBarO0 + 2,
  kBarFin,   // the QK^T thread's MMAs done
  kBarPVd0,  // + S buffer: the PV that read P from that buffer is done
  kBarFin2 = kBarPVd0 + 2,  // the PV thread's MMAs done
  kBarProd,  // both QK^T producers have published their last round per slot (count 2)
  kBarPeFull0,  // + QK^T slot, fused rotation: this CTA's K_pe copy landed (each CTA its own)
  kBarRdy0 = kBarPeFull0 + kQKSlots,  // + QK^T slot, fused rotation: both CTAs' K_pe rotated (even CTA, 128 lanes)
  kNumBars = kBarRdy0 + kQKSlots
};
// after the barriers: abort flag, TMEM address, the QK^T producers' last round per slot
static_assert(kNumBars * 8 + 8 + kQKProducers * kQKSlots * 4 <= 512, "barrier area");

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

// The key stream is cut into rounds, each one ring slot filled by one or two
// copies counted on one barrier (a copy and its barrier cost a producer thread
// far more than the bytes, so rounds are large and two threads issue the
// QK^T rounds).  QK^T ring: per tile, round m < 4 holds latent chunks 2m and
// 2m+1 of the CTA's own 64 keys, m = 4 its K_pe chunk; QK^T round qr (counted
// over all units) uses slot qr % kQKSlots.  PV ring: per tile, round q holds
// latent columns 256 half + 128 q + 64 rank of all 128 keys (two copies, one
// per key half); PV round vr uses slot vr % kPVSlots.

// Pages of one KV tile per 64-key half h: the K_pe and latent pages of the
// half's first run and whether the half's pages are consecutive (then one
// copy loads the unit).
struct TilePages {
  int k0, k1, v0, v1;
  uint32_t cons;  // bit h: K_pe pages of half h consecutive; bit 2 + h: latent pages
};

__device__ __forceinline__ void load_runs(const AttnParams& p, const AttnSeg& seg, int tile, int rpt, int2 first,
                                          int2 (&kv)[kMaxRuns]) {
#pragma unroll
  for (int g = 0; g < kMaxRuns; ++g) {
    const int ri = tile * rpt + g;
    kv[g] = first;  // past the last run the segment's first page stands in (finite values, masked out)
    if (g < rpt && ri < seg.n_runs) kv[g] = *reinterpret_cast<const int2*>(p.runs + seg.run_off + ri);
  }
}

__device__ __forceinline__ TilePages tile_pages(const int2 (&kv)[kMaxRuns], int page, int rpu, int layer_base) {
  TilePages t;
  t.cons = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int g0 = page > 64 ? 0 : h * rpu;  // a 128-slot page holds both halves
    int kf = kv[0].x, vf = kv[0].y;
#pragma unroll
    for (int g = 1; g < kMaxRuns; ++g)
      if (g == g0) {
        kf = kv[g].x;
        vf = kv[g].y;
      }
    bool kc = true, vc = true;
#pragma unroll
    for (int g = 1; g < kMaxRuns; ++g) {
      const int rel = g - g0;
      if (rel > 0 && rel < rpu) {
        kc = kc && kv[g].x == kf + rel;
        vc = vc && kv[g].y == vf + rel;
      }
    }
    if (h == 0) {
      t.k0 = layer_base + kf;
      t.v0 = layer_base + vf;
    } else {
      t.k1 = layer_base + kf;
      t.v1 = layer_base + vf;
    }
    t.cons |= (kc ? 1u << h : 0u) | (vc ? 4u << h : 0u);
  }
  return t;
}

// One producer thread.  pv: the PV ring (warp 7); else the QK^T ring, whose
// rounds are owned by position in the tile: rounds 0, 2 and K_pe by who = 0
// (warp 0, which also loads the Q tiles), rounds 1 and 3 by who = 1, so each
// owns a round in every 3 consecutive ones (the ring's slot count).  With
// fused rotation each CTA's K_pe copy lands on a barrier of its own CTA (the
// rotation warp waits there) and the ring's Full barrier takes a plain arrive
// in its place, so its phases stay in step.
template <bool kFused>
__device__ __forceinline__ void produce(const AttnParams& p, int u0, int u1, uint32_t sbase, uint32_t rank, bool pv,
                                        int who, volatile int* abort_flag, volatile int* prod_last) {
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int G = p.group, tpt = kRows / G, rpt = kKeys / p.page;
  const int rpu = p.page >= 64 ? 1 : 64 / p.page;  // runs per 64-key half
  const int n_slots = pv ? kPVSlots : kQKSlots;
  const int full0 = pv ? kBarVFull0 : kBarFull0, empty0 = pv ? kBarVEmpty0 : kBarEmpty0;
  const uint32_t ring = sbase + (pv ? kVSlots : kSlots);
  const uint32_t lead_full0 = ptx::mapa(bar(full0), 0);
  const uint32_t lead_q = ptx::mapa(bar(kBarQ), 0);
  const bool loads_q = !pv && who == 0;
  const int layer_base = p.layer * p.n_pages;
  if (loads_q) {
    ptx::prefetch_tensormap(&p.q_map);
    ptx::prefetch_tensormap(&p.k_map);
    ptx::prefetch_tensormap(&p.v_map);
    ptx::prefetch_tensormap(&p.k_tile_map);
    ptx::prefetch_tensormap(&p.v_tile_map);
  }
  // the unit being streamed (read by the lambdas below)
  AttnWork w = p.work[2 * u0 + int(rank)];
  AttnSeg seg = p.segs[w.seg];
  int2 first = make_int2(0, 0);
  int half = 0;  // which 256 output columns
  bool ok = true;
  // One 64-key x 64-column block: keys of half kh of local tile j (pages tp),
  // columns col of K_pe (pe) or of the latent.
  // local: the copy completes on barrier fb of this CTA (else on the even CTA's).
  auto copy = [&](uint32_t dst, uint32_t fb, bool pe, int kh, int col, int j, const TilePages& tp, bool local = false) {
    auto load = [&](uint32_t d, const CUtensorMap* map, int c0, int c1, int c3) {
      if (local)
        ptx::tma_load_4d(d, map, fb, c0, c1, 0, c3);
      else
        ptx::tma_load_4d_pair(d, map, fb, c0, c1, 0, c3);
    };
    const int pg = pe ? (kh ? tp.k1 : tp.k0) : (kh ? tp.v1 : tp.v0);
    const bool cons = (tp.cons >> ((pe ? 0 : 2) + kh)) & 1u;
    if (p.page > 64) {  // one page per tile, the block is its half kh
      load(dst, pe ? &p.k_tile_map : &p.v_tile_map, col, 64 * kh, pg);
    } else if (cons) {
      load(dst, pe ? &p.k_tile_map : &p.v_tile_map, col, 0, pg);
    } else {  // pages of the half one by one (copied pages of a fork)
      const CUtensorMap* map = pe ? &p.k_map : &p.v_map;
      for (int g = 0; g < rpu; ++g) {
        const int ri = (w.t0 + j) * rpt + kh * rpu + g;
        int2 kv = first;
        if (ri < seg.n_runs) kv = *reinterpret_cast<const int2*>(p.runs + seg.run_off + ri);
        load(dst + g * p.page * 128, map, col, 0, layer_base + (pe ? kv.x : kv.y));
      }
    }
  };
  int rd = 0;  // rounds of this ring so far, over all units
  // Test hook: with p.load_cap >= 0 this thread issues at most that many
  // rounds and then stops (no error of its own); the waits for the missing
  // rounds run out after p.wait_ns and report AKV_ERR_DEVICE_TIMEOUT.
  int n_issued = 0;
  bool capped = false;
  int last[kQKSlots] = {-1, -1, -1};     // the last round this thread issued into each slot
  int last_pe[kQKSlots] = {-1, -1, -1};  // fused rotation: the last K_pe round (local barrier) per slot
  // Round m of local tile j: QK^T round m (< kQKRounds) or PV round m.
  auto round = [&](int m, int j, const TilePages& tp) {
    const bool mine = pv || ((m == 1 || m == 3) == (who == 1));
    if (ok && mine && !capped && p.load_cap >= 0 && n_issued >= p.load_cap) capped = true;
    if (ok && mine && !capped) {
      ++n_issued;
      const int slot = rd % n_slots, use = rd / n_slots;
      if (use >= 1 && !ptx::mbar_wait(bar(empty0 + slot), (use - 1) & 1, abort_flag, p.wait_ns)) {
        ok = false;
      } else {
#pragma unroll
        for (int s = 0; s < kQKSlots; ++s)
          if (s == slot) last[s] = rd;
        const uint32_t dst = ring + slot * kSlot;
        const uint32_t fb = lead_full0 + 8u * uint32_t(slot);
        const int kr = int(rank);
        if (pv) {
          const int col = 256 * half + 128 * m + 64 * kr;
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar(full0 + slot), 2 * kSlot);
          copy(dst, fb, false, 0, col, j, tp);
          copy(dst + kUnit, fb, false, 1, col, j, tp);
        } else if (m < kQKRounds - 1) {
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar(full0 + slot), 2 * kSlot);
          copy(dst, fb, false, kr, 128 * m, j, tp);
          copy(dst + kUnit, fb, false, kr, 128 * m + 64, j, tp);
        } else if (kFused) {
          if (rank == 0) ptx::mbar_arrive(bar(full0 + slot));  // the phase only: the copy completes locally
          ptx::mbar_arrive_expect_tx(bar(kBarPeFull0 + slot), kUnit);
          copy(dst, bar(kBarPeFull0 + slot), true, kr, 0, j, tp, true);
#pragma unroll
          for (int s = 0; s < kQKSlots; ++s)
            if (s == slot) last_pe[s] = rd;
        } else {
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar(full0 + slot), 2 * kUnit);
          copy(dst, fb, true, kr, 0, j, tp);
        }
      }
    }
    ++rd;
  };
  const int n_rounds = pv ? kPVRounds : kQKRounds;
  int q_loads = 0;
  for (int u = u0; u < u1 && ok && !capped; ++u) {
    w = p.work[2 * u + int(rank)];
    seg = p.segs[w.seg];
    half = w.n_b;
    first = *reinterpret_cast<const int2*>(p.runs + seg.run_off);
    const int n_loc = min(max(w.n_a - w.t0, 0), w.t1 - w.t0);  // local tile j is global tile t0 + j
    if (loads_q) {
      // Q tiles of this unit, once the previous unit's last QK MMA has released
      // both CTAs' Q buffers (a multicast commit to each CTA's Q-free barrier).
      if (u > u0 && !(ok = ptx::mbar_wait(bar(kBarQFree), (u - u0 - 1) & 1, abort_flag, p.wait_ns))) break;
      const int q_tok0 = seg.q_row0 + w.qt0 * tpt;
      if (rank == 0) ptx::mbar_arrive_expect_tx(bar(kBarQ), 2 * kQChunks * kQChunk);
      for (int c = 0; c < kQChunks; ++c)
        ptx::tma_load_3d_pair(sbase + kQ + c * kQChunk, &p.q_map, lead_q, c * 64, 0, q_tok0);
      ++q_loads;
    }
    // runs of tile j + 1 are loaded while tile j's rounds are issued
    int2 raw[kMaxRuns];
    load_runs(p, seg, w.t0, rpt, first, raw);
    for (int j = 0; j < n_loc && ok; ++j) {
      const TilePages tp = tile_pages(raw, p.page, rpu, layer_base);
      if (j + 1 < n_loc) load_runs(p, seg, w.t0 + j + 1, rpt, first, raw);
      for (int m = 0; m < n_rounds; ++m) round(m, j, tp);
    }
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 10, pv ? 2 : who);
    *abort_flag = 1;
  }
  // Drain (one producer per ring): every round of the ring issued so far has
  // landed (the Full barriers, in the even CTA, count both CTAs' bytes) and
  // been consumed (the consumer's multicast commit has reached this CTA's
  // Empty barrier), and the Q barrier's last phase completed.  A slot is
  // drained at the last round any producer issued into it: no later phase
  // exists, so the parity wait cannot match an older or a newer phase.
  if (!pv) {
#pragma unroll
    for (int s = 0; s < kQKSlots; ++s) prod_last[who * kQKSlots + s] = last[s];
    ptx::mbar_arrive(bar(kBarProd));
    if (who != 0) return;
    if (!ptx::mbar_wait_drain(bar(kBarProd), 0, kDrainLimitNs)) raise_error(p.err, kErrTimeout, blockIdx.x, 15, 0);
#pragma unroll
    for (int s = 0; s < kQKSlots; ++s)
      for (int q = 1; q < kQKProducers; ++q) last[s] = max(last[s], prod_last[q * kQKSlots + s]);
  }
  bool drained = true;
  if (loads_q && rank == 0 && q_loads) drained = ptx::mbar_wait_drain(bar(kBarQ), (q_loads - 1) & 1, kDrainLimitNs);
#pragma unroll
  for (int s = 0; s < kQKSlots; ++s) {
    if (last[s] < 0) continue;
    const uint32_t parity = uint32_t(last[s] / n_slots) & 1u;
    if (rank == 0) drained = ptx::mbar_wait_drain(bar(full0 + s), parity, kDrainLimitNs) && drained;
    drained = ptx::mbar_wait_drain(bar(empty0 + s), parity, kDrainLimitNs) && drained;
  }
  // K_pe copies of fused rotation: round 5T + 4 of tile T is the (T / 3)-th use of its slot.
#pragma unroll
  for (int s = 0; s < kQKSlots; ++s)
    if (last_pe[s] >= 0)
      drained = ptx::mbar_wait_drain(bar(kBarPeFull0 + s), uint32_t((last_pe[s] / kQKRounds) / kQKSlots) & 1u,
                                     kDrainLimitNs) && drained;
  if (!drained) raise_error(p.err, kErrTimeout, blockIdx.x, 14, pv ? 2 : who);  // copies may still be in flight
}

// --------------------------------------------------------------------- MMA
// Even CTA only, two issuing threads.  A thread's tensor-core queue is short
// and every shared-memory access it makes between MMAs (a barrier wait above
// all) leaves the tensor pipe idle for about 200 clocks; with the QK^T and the
// PV MMAs issued by different threads, one thread's MMAs fill the other's
// waits.  QK^T: D (S, 128 columns per CTA) = Q (256 rows) x K (128 keys, 64
// from each CTA).  PV: O quarter q (128 columns) += P (256 rows x 128 keys,
// from each CTA's TMEM) x V (128 keys x 128 columns, 64 from each CTA).

// Local tiles of a unit (local tile j is global tile t0 + j).
__device__ __forceinline__ int unit_tiles(const AttnWork& w) { return min(max(w.n_a - w.t0, 0), w.t1 - w.t0); }

// QK^T thread.  S of global tile gt (tiles of earlier units included: the S,
// P and O phases continue across units) goes to S buffer gt & 1, which holds
// P(gt - 2) until that tile's PV is done.  After a unit's last QK^T MMA both
// CTAs may reload their Q tiles.  With fused rotation the K_pe round is read
// once both CTAs' rotation warps have rotated it (the ready barrier).
template <bool kFused>
__device__ __forceinline__ void issue_qk(const AttnParams& p, int u0, int u1, uint32_t sbase, uint32_t tmem,
                                         volatile int* abort_flag) {
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  constexpr uint32_t idesc_qk = ptx::idesc_bf16(2 * kRows, kKeys, false);
  bool issued = false;  // a commit is only issued after this thread's first MMA
  bool ok = true;
  // Descriptors are built once and advanced by constants (only the start
  // address changes).
  const uint64_t qd0 = ptx::smem_desc(sbase + kQ, 16, 1024);
  auto chunk = [&](uint32_t tS, int c, uint32_t kt) {  // S (+)= Q chunk c x K chunk at kt
    const uint64_t kd = ptx::smem_desc(kt, 16, 1024), qd = ptx::desc_advance(qd0, c * kQChunk);
    ptx::mma_bf16_pair(tS, qd, kd, idesc_qk, c > 0);
#pragma unroll
    for (int ks = 1; ks < 4; ++ks)
      ptx::mma_bf16_pair(tS, ptx::desc_advance(qd, ks * 32), ptx::desc_advance(kd, ks * 32), idesc_qk, 1);
  };
  int g = 0, rd0 = 0;  // tiles and key-stream rounds of earlier units
  for (int u = u0; u < u1 && ok; ++u) {
    const int n = unit_tiles(p.work[2 * u]);
    const bool more = u + 1 < u1;
    if (!(ok = ptx::mbar_wait(bar(kBarQ), (u - u0) & 1, abort_flag, p.wait_ns))) break;
    for (int j = 0; j < n && ok; ++j) {
      const int gt = g + j;
      if (gt >= 2 && !(ok = ptx::mbar_wait(bar(kBarPVd0 + (gt & 1)), ((gt >> 1) - 1) & 1, abort_flag, p.wait_ns)))
        break;
      const uint32_t tS = tmem + 128u * (gt & 1);
      int rd = rd0 + kQKRounds * j;  // QK^T ring round
#pragma unroll 1
      for (int m = 0; m < kQKRounds; ++m, ++rd) {
        const int slot = rd % kQKSlots;
        if (kFused && m == kQKRounds - 1)  // the (gt / 3)-th K_pe round in this slot
          ok = ptx::mbar_wait_cl(bar(kBarRdy0 + slot), (gt / kQKSlots) & 1, abort_flag, p.wait_ns);
        else
          ok = ptx::mbar_wait(bar(kBarFull0 + slot), (rd / kQKSlots) & 1, abort_flag, p.wait_ns);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t kt = sbase + kSlots + slot * kSlot;
        if (m < kQKRounds - 1) {
          chunk(tS, 2 * m, kt);
          chunk(tS, 2 * m + 1, kt + kUnit);
        } else {
          chunk(tS, kQChunks - 1, kt);
        }
        issued = true;
        ptx::mma_commit_pair_mc(bar(kBarEmpty0 + slot), kBoth);
      }
      if (!ok) break;
      ptx::mma_commit_pair_mc(bar(kBarS0 + (gt & 1)), kBoth);
      if (more && j == n - 1) ptx::mma_commit_pair_mc(bar(kBarQFree), kBoth);
    }
    g += n;
    rd0 += kQKRounds * n;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 11, 0);
    *abort_flag = 1;
  }
  if (issued) {
    ptx::mma_commit_pair(bar(kBarFin));
    if (!ptx::mbar_wait_drain(bar(kBarFin), 0, kDrainLimitNs)) raise_error(p.err, kErrTimeout, blockIdx.x, 16, 0);
  }
}

// PV thread.  PV of global tile gt reads P from S buffer gt & 1 once the
// softmax threads of both CTAs have written it; the commit after it releases
// that buffer to the QK^T thread (and O to the softmax threads).  A unit's
// first PV overwrites O: the softmax threads arrived on its P only after
// reading out the previous unit's O.
__device__ __forceinline__ void issue_pv(const AttnParams& p, int u0, int u1, uint32_t sbase, uint32_t tmem,
                                         volatile int* abort_flag) {
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  constexpr uint32_t idesc_pv = ptx::idesc_bf16(2 * kRows, 128, true);
  const uint32_t tO = tmem + 256;
  bool issued = false;
  bool ok = true;
  int g = 0, rd0 = 0;
  for (int u = u0; u < u1 && ok; ++u) {
    const int n = unit_tiles(p.work[2 * u]);
    for (int j = 0; j < n && ok; ++j) {
      const int gt = g + j;
      if (!(ok = ptx::mbar_wait_cl(bar(kBarP0 + (gt & 1)), (gt >> 1) & 1, abort_flag, p.wait_ns))) break;
      ptx::tc_fence_after();
      const uint32_t tP = tmem + 128u * (gt & 1);  // P of tile gt, packed over S
      int rd = rd0 + kPVRounds * j;  // PV ring round
#pragma unroll 1
      for (int q = 0; q < kPVRounds; ++q, ++rd) {
        const int slot = rd % kPVSlots;
        if (!(ok = ptx::mbar_wait(bar(kBarVFull0 + slot), (rd / kPVSlots) & 1, abort_flag, p.wait_ns))) break;
        ptx::tc_fence_after();
        const uint64_t vd = ptx::smem_desc(sbase + kVSlots + slot * kSlot, kSlot, 1024);
        ptx::mma_bf16_tmem_a_pair(tO + 128u * q, tP, vd, idesc_pv, j > 0);
#pragma unroll
        for (int ks = 1; ks < kKeys / 16; ++ks)
          ptx::mma_bf16_tmem_a_pair(tO + 128u * q, tP + 8u * ks, ptx::desc_advance(vd, ks * 2048), idesc_pv, 1);
        issued = true;
        ptx::mma_commit_pair_mc(bar(kBarVEmpty0 + slot), kBoth);
      }
      if (!ok) break;
      ptx::mma_commit_pair_mc(bar(kBarO0 + (gt & 1)), kBoth);
      ptx::mma_commit_pair(bar(kBarPVd0 + (gt & 1)));
    }
    g += n;
    rd0 += kPVRounds * n;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 13, 0);
    *abort_flag = 1;
  }
  if (issued) {
    ptx::mma_commit_pair(bar(kBarFin2));
    if (!ptx::mbar_wait_drain(bar(kBarFin2), 0, kDrainLimitNs)) raise_error(p.err, kErrTimeout, blockIdx.x, 17, 0);
  }
}

// ------------------------------------------------------------ K_pe rotation
// Fused rotation ([Leyline] "Method": under MLA only K_pe carries position;
// [AKV-blog] section 4: rotate keys on their way to the tensor core instead of
// writing them back).  Two warps per CTA (part 0, 1: 32 rows each, one per
// lane) take the K_pe round of every tile in order once their CTA's copy has
// landed, rotate each of its 64 key rows whose run carries a pending shift by
// R(delta * theta_j) in shared memory -- the arithmetic and angle table of
// repos_rotate, so the bits equal the materialised key -- make the writes
// visible to the tensor core and arrive (every lane; the odd CTA remotely) on
// the even CTA's ready barrier.
__device__ __forceinline__ void rotate_pe(const AttnParams& p, int u0, int u1, uint8_t* smem, uint32_t sbase,
                                          uint32_t rank, int part, volatile int* abort_flag) {
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int lane = threadIdx.x % 32, rpt = kKeys / p.page;
  int page_shift = 4;
  while ((1 << page_shift) < p.page) ++page_shift;
  bool ok = true;
  int g = 0;  // tiles of earlier units
  for (int u = u0; u < u1 && ok; ++u) {
    const AttnWork w = p.work[2 * u + int(rank)];
    const AttnSeg seg = p.segs[w.seg];
    const int n = unit_tiles(w);
    for (int j = 0; j < n; ++j) {
      const int gt = g + j, slot = (kQKRounds * gt + kQKRounds - 1) % kQKSlots;
      if (!(ok = ptx::mbar_wait(bar(kBarPeFull0 + slot), (gt / kQKSlots) & 1, abort_flag, p.wait_ns))) break;
      uint8_t* tile = smem + kSlots + slot * kSlot;
      {
        const int row = 32 * part + lane;  // this CTA's key 64 rank + row of the tile
        const int ri = (w.t0 + j) * rpt + ((64 * int(rank) + row) >> page_shift);
        const int didx = ri < seg.n_runs ? p.run_didx[seg.run_off + ri] : -1;
        if (didx >= 0) {
        const float2* cs = p.cs + int64_t(didx) * (kPe / 2);
        auto at = [&](int v) {  // 16-byte vector v of the row (128-byte swizzle)
          return reinterpret_cast<uint4*>(tile + row * 128 + (((v & 7) ^ (row & 7)) << 4));
        };
        if (!p.rope_half) {
#pragma unroll
          for (int v = 0; v < kPe / 8; ++v) {  // pairs 4v .. 4v + 3
            uint4* q = at(v);
            const uint4 x = *q;
            const float4 a = __ldg(reinterpret_cast<const float4*>(cs + 4 * v));
            const float4 b = __ldg(reinterpret_cast<const float4*>(cs + 4 * v + 2));
            *q = make_uint4(pack_rot(rot2(x.x, a.x, a.y)), pack_rot(rot2(x.y, a.z, a.w)), pack_rot(rot2(x.z, b.x, b.y)),
                            pack_rot(rot2(x.w, b.z, b.w)));
          }
        } else {
#pragma unroll
          for (int v = 0; v < kPe / 16; ++v) {  // dims 8v .. 8v + 7 pair with dims kPe/2 + 8v ..
            uint4* qa = at(v);
            uint4* qb = at(v + kPe / 16);
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
      }
      ptx::fence_proxy_async_smem();  // generic-proxy writes -> tensor-core (async proxy) reads
      if (rank == 0)
        ptx::mbar_arrive(bar(kBarRdy0 + slot));
      else
        ptx::mbar_arrive_cluster(ptx::mapa(bar(kBarRdy0 + slot), 0));
    }
    g += n;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 18, 2 * int(rank) + part);
    *abort_flag = 1;
  }
}

// ----------------------------------------------------------------- softmax
__device__ __forceinline__ void softmax(const AttnParams& p, int u0, int u1, uint8_t* smem, uint32_t sbase,
                                        uint32_t tmem, uint32_t rank, volatile int* abort_flag) {
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int quad = (threadIdx.x / 32) & 3;  // warps 2..5 -> TMEM lane quadrants 2, 3, 0, 1
  const int lane = threadIdx.x % 32;
  const int r = quad * 32 + lane;
  const uint32_t lane_addr = uint32_t(quad * 32) << 16;
  const uint32_t tO = tmem + 256;
  const int G = p.group, tpt = kRows / G, rpt = kKeys / p.page;
  const int t_loc = r / G, g = r % G;
  const float sl2 = p.scale_log2;
  int page_shift = 4;
  while ((1 << page_shift) < p.page) ++page_shift;
  const int sl_own = r & (p.page - 1);
  const uint32_t lead_p0 = ptx::mapa(bar(kBarP0), 0);  // P barriers of the even CTA
  const uint32_t lead_p1 = ptx::mapa(bar(kBarP0 + 1), 0);
  bool ok = true;
  int gbase = 0;  // tiles of earlier units: the S, P and O phases continue across units
  for (int u = u0; u < u1; ++u) {
  const AttnWork w = p.work[2 * u + int(rank)];
  const AttnSeg seg = p.segs[w.seg];
  const int n = min(max(w.n_a - w.t0, 0), w.t1 - w.t0);  // local tile j is global tile t0 + j
  const int qi = w.qt0 * tpt + t_loc;
  const bool row_valid = qi < seg.q_len;
  const int lim = seg.kv_len - seg.q_len + (row_valid ? qi : seg.q_len - 1);
  float m_run = -INFINITY, l_run = 0.f;
  // (lohi, es) of the run holding key column r of the current tile, fetched one tile ahead;
  // lo = hi = 0 past the segment's last run, so no slot matches
  const int2* run_le = reinterpret_cast<const int2*>(p.runs + seg.run_off);
  int2 run_cur = make_int2(0, 0);
  {
    const int ri0 = w.t0 * rpt + (r >> page_shift);
    if (ri0 < seg.n_runs) run_cur = run_le[2 * ri0 + 1];
  }
  for (int j = 0; j < n; ++j) {
    const int gt = gbase + j;
    const uint32_t tS = tmem + 128u * (gt & 1);
    // Column entries need no score, so they are formed before S is waited for;
    // they go to the buffer of this tile's parity: the other buffer may still
    // be read by a thread finishing the previous tile.
    int* colE = reinterpret_cast<int*>(smem + kColE) + (gt & 1) * 128;
    int e = INT_MAX;  // entry index of key column r (INT_MAX: none)
    {
      const int lo = run_cur.x & 0xffff, hi = run_cur.x >> 16;
      if (sl_own >= lo && sl_own < hi) e = run_cur.y + (sl_own - lo);
      colE[r] = e;
      const int ri = (w.t0 + j + 1) * rpt + (r >> page_shift);
      run_cur = ri < seg.n_runs ? run_le[2 * ri + 1] : make_int2(0, 0);
    }
    // One barrier per tile: every thread's S arrived (and no warp's O wait of
    // the previous tile ran out) and every column has an entry; only when that
    // fails does a second one tell a failure from masking, and then every
    // thread leaves together.
    const bool s_ok = ok && ptx::mbar_wait(bar(kBarS0 + (gt & 1)), (gt >> 1) & 1, abort_flag, p.wait_ns);
    const bool all_valid = ptx::bar_red_and(1, 128, s_ok && e != INT_MAX);
    if (!all_valid && !ptx::bar_red_and(1, 128, s_ok)) {
      ok = false;
      break;
    }
    ptx::tc_fence_after();
    const bool need_mask = !all_valid || colE[kKeys - 1] > lim;
    const int4* ce4 = reinterpret_cast<const int4*>(colE);
    // One TMEM pass per 64-column half: max in registers, P with the running
    // max (raised lazily, beyond 2^8), stored packed over consumed S columns;
    // the first half's P is rescaled afterwards if the second half raised it.
    float sum[4] = {0.f, 0.f, 0.f, 0.f};
    float m_use = m_run, alpha = 1.0f, a_first = 1.0f;
    bool resc = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t u[64];
      ptx::tmem_load64(tS + lane_addr + h * 64, u);
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
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 32; ++c)  // three-input max: two scores per instruction
        mx[c & 3] = ptx::max3(mx[c & 3], __uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1]));
      const float mh = fmaxf(ptx::max3(mx[0], mx[1], mx[2]), mx[3]) * sl2;
      if (mh > m_use + 8.0f) {
        const float a = m_use == -INFINITY ? 0.f : ptx::ex2_approx(m_use - mh);
        if (h == 1) {
#pragma unroll
          for (int k = 0; k < 4; ++k) sum[k] *= a;
          a_first = a;
        }
        alpha *= a;
        m_use = mh;
        resc = true;
      }
      const float msub = m_use == -INFINITY ? 0.f : m_use;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {  // scale-and-shift as one packed FMA per score pair
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])),
                                    make_float2(sl2, sl2), make_float2(-msub, -msub));
        const float p0 = ptx::ex2_approx(x.x), p1 = ptx::ex2_approx(x.y);
        sum[(2 * c) & 3] += p0;
        sum[(2 * c + 1) & 3] += p1;
        pk[c] = pack_bf16(p0, p1);
      }
      ptx::tmem_store32(tS + lane_addr + h * 32, pk);  // over S columns already read
    }
    // TMEM loads / stores are warp-collective: the whole warp takes these branches.
    if (__any_sync(0xffffffffu, a_first != 1.0f)) {
      uint32_t q[32];
      ptx::tmem_load32(tS + lane_addr, q);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q[c]));
        q[c] = pack_bf16(f.x * a_first, f.y * a_first);
      }
      ptx::tmem_store32(tS + lane_addr, q);
    }
    // A warp that raised its running max rescales its rows of O, which must be
    // stable first (PV of tile j-1 done), before it arrives on P; the other
    // warps arrive first and wait after, so P of tile j reaches the PV thread
    // while PV of tile j-1 may still run (PV of tile j queues behind it on the
    // same thread).  That later wait costs nothing: S of tile j+1 needs PV of
    // tile j-1 done anyway.  O and P have one barrier per tile parity and
    // every warp waits for every tile's O in order, so no parity wait can
    // alias: the barrier of tile j-1 cannot complete tile j+1 before this
    // warp arrives on P of tile j+1.  A wait that runs out leaves ok false
    // for the next tile's barrier (or the unit's end), where every thread
    // learns of it.
    bool o_waited = j == 0;
    if (j > 0 && __any_sync(0xffffffffu, resc)) {
      const bool o_ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarO0 + ((gt - 1) & 1)), ((gt - 1) >> 1) & 1,
                                                               abort_flag, p.wait_ns));
      o_waited = true;
      ptx::tc_fence_after();
      if (o_ok) {  // TMEM loads / stores are warp-collective: the whole warp takes this branch
#pragma unroll 1
        for (int c = 0; c < 256 / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_load32(tO + lane_addr + c * 32, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          ptx::tmem_store32(tO + lane_addr + c * 32, o);
        }
      } else {
        ok = false;
      }
    }
    l_run = l_run * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
    m_run = m_use;
    ptx::tc_fence_before();
    if (rank == 0)
      ptx::mbar_arrive(bar(kBarP0 + (gt & 1)));
    else
      ptx::mbar_arrive_cluster((gt & 1) ? lead_p1 : lead_p0);
    if (!o_waited && !ptx::mbar_wait(bar(kBarO0 + ((gt - 1) & 1)), ((gt - 1) >> 1) & 1, abort_flag, p.wait_ns))
      ok = false;
  }
  if (n > 0) {  // every thread takes this barrier: ok may differ between warps here
    const int gl = gbase + n - 1;
    const bool o_ok = ok && ptx::mbar_wait(bar(kBarO0 + (gl & 1)), (gl >> 1) & 1, abort_flag, p.wait_ns);
    ok = ptx::bar_red_and(1, 128, o_ok);
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 12, 0);
    *abort_flag = 1;
    return;
  }
  ptx::tc_fence_after();
  // A shadow (stand-in for a missing query tile) computes and writes nothing.
  // The next unit's first PV overwrites O only after this unit's O is read
  // out here: this thread arrives on its first P after the epilogue.
  const int half = w.n_b;
  if (!(w.kvh & kShadow) && w.part >= 0) {
    // Split part: unnormalised O half, running max and sum, [column][row] layout.
    float* base = p.partial + w.part * partial_floats(1, 256) + r;
#pragma unroll 1
    for (int c = 0; c < 256 / 32; ++c) {
      uint32_t o[32];
      ptx::tmem_load32(tO + lane_addr + c * 32, o);
#pragma unroll
      for (int k = 0; k < 32; ++k) base[int64_t(c * 32 + k) * 128] = __uint_as_float(o[k]);
    }
    base[int64_t(256) * 128] = n > 0 ? m_run : -INFINITY;
    base[int64_t(257) * 128] = n > 0 ? l_run : 0.f;
    const int64_t row = int64_t(seg.q_row0 + qi) * p.hq + g;
    merge_if_last<256>(p, w, 0, r, 1,
                       row_valid ? static_cast<__nv_bfloat16*>(p.o) + row * kLat + 256 * half : nullptr,
                       row_valid && p.lse && half == 0 ? p.lse + row : nullptr);
  } else if (!(w.kvh & kShadow)) {
    const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(p.o) + (int64_t(seg.q_row0 + qi) * p.hq + g) * kLat + 256 * half;
#pragma unroll 1
    for (int c = 0; c < 256 / 32; ++c) {
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
    if (row_valid && p.lse && half == 0) {
      const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      p.lse[int64_t(seg.q_row0 + qi) * p.hq + g] = lse;
    }
  }
  ptx::tc_fence_before();  // the O reads above precede this thread's next arrive on P
  gbase += n;
  }
}

template <bool kFused>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    segment_attn_mla_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + kBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBars + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBars + 8 * kNumBars + 4);
  volatile int* prod_last = reinterpret_cast<volatile int*>(smem + kBars + 8 * kNumBars + 8);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ptx::cluster_ctarank();
  // The pair runs units [u0, u1); unit u is work entries 2u (even CTA) and 2u + 1.
  const int pair = int(blockIdx.x) >> 1;
  const int u0 = p.cta_units ? p.cta_units[pair] : pair;
  const int u1 = p.cta_units ? p.cta_units[pair + 1] : pair + 1;
#ifdef AKV_CHECKED
  {  // both CTAs of the pair check the same items, so the pair returns together, before any cluster barrier
    bool ok = u0 >= 0 && u0 < u1 && 2 * u1 <= p.n_work;
    for (int k = 2 * u0; ok && k < 2 * u1; ++k)
      ok = attn_item_ok(p.work[k], p.segs, p.runs, p.n_segs, p.n_runs, p.n_q_rows, p.n_pages, p.page,
                        int(threadIdx.x), int(blockDim.x));
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) report_device_error(p.err, 11, int(blockIdx.x), 0);
      return;
    }
  }
#endif
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      ptx::mbar_init(bars + 8u * i, i == kBarP0 || i == kBarP0 + 1           ? 2 * 128
                                    : i == kBarProd                          ? kQKProducers
                                    : (i >= kBarRdy0 && i < kBarRdy0 + kQKSlots) ? 2 * 32 * kRotWarps
                                                                               : 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  ptx::cluster_sync();  // both CTAs' barriers initialised before any remote arrive or copy
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // the pair's TMEM is allocated in both CTAs before the first MMA
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0 || warp == 6 || warp == 7) {
    if (lane == 0) produce<kFused>(p, u0, u1, sbase, rank, warp == 7, warp == 6 ? 1 : 0, abort_flag, prod_last);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) issue_qk<kFused>(p, u0, u1, sbase, tmem, abort_flag);
  } else if (warp == 8) {
    if (lane == 0 && rank == 0) issue_pv(p, u0, u1, sbase, tmem, abort_flag);
  } else if (warp == 9 || warp == 10) {
    if (kFused) rotate_pe(p, u0, u1, smem, sbase, rank, warp - 9, abort_flag);
  } else {
    softmax(p, u0, u1, smem, sbase, tmem, rank, abort_flag);
  }
  ptx::tc_fence_before();
  __syncwarp();
  ptx::cluster_sync();  // every MMA of the pair done and every remote signal delivered
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
  ptx::cluster_sync();
}

}  // namespace

// CTAs of this kernel that can be resident at once (pairs x 2): the planner's
// wave size.  0 if the occupancy query fails.
int segment_attn_mla_slots() {
  const int smem = int(kBytes) + 1024;
  if (cudaFuncSetAttribute(segment_attn_mla_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, segment_attn_mla_kernel<false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return 2 * clusters;
}

namespace {
template <bool kFused>
cudaError_t launch_mla_variant(const AttnParams& p, int grid, int smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(segment_attn_mla_kernel<kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  segment_attn_mla_kernel<kFused><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_segment_attn_mla(const AttnParams& p, cudaStream_t st) {
  if (p.n_work <= 0) return cudaSuccess;
  if (p.n_work % 2) return cudaErrorInvalidValue;  // CTA pairs
  const int grid = p.cta_units ? 2 * p.n_cta : p.n_work;  // persistent: one CTA pair per unit list
  const int smem = int(kBytes) + 1024;
  return p.fused ? launch_mla_variant<true>(p, grid, smem, st) : launch_mla_variant<false>(p, grid, smem, st);
}

}  // namespace akv
