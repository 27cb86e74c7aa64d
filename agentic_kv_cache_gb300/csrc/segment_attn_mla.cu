// segment_batch_attn, MLA variant ([Leyline] "Method": under MLA the cached
// key is a position-free latent -- which also serves as the value -- plus a
// RoPE'd K_pe; 16 query heads share one latent).  What it computes is the
// same as the GQA kernel ([AKV-notes] section 3 "Segment-Batch Attention";
// [AKV-blog] section 2 "The Drop Primitive"): per segment, causal softmax
// attention of its queries over its visible entries, with
//   score = q_latent . c + q_pe . k_pe   (d_qk = 512 + 64)
//   out   = sum_j p_j c_j                (d_v = 512).
//
// GB300 design.  One CTA = one 128-row query tile (8 tokens x 16 heads) and
// one half of the 512 output columns: O for all 512 columns would fill TMEM
// by itself, so each half recomputes S (+53% MMA over the algorithmic count;
// the two halves run as separate CTAs).  TMEM: S0, S1 (double-buffered, P
// written back over the consumed S columns as bf16 pairs) and the 256-column O
// half.  The Q tile (144 KiB) stays in shared memory; keys stream through a
// 4-slot ring of 16 KiB chunks: per 128-key tile, the 8 latent chunks and the
// K_pe chunk for QK^T, then the 4 latent chunks of this half for PV.
// Warp 0: TMA producer; warp 1: TMEM owner and single-thread MMA issuer;
// warps 2-5: softmax (one row per thread).  Every wait is bounded.
#include <cuda_bf16.h>

#include <climits>
#include <cstdint>

#include "akv_internal.h"
#include "attn_merge.cuh"
#include "sm100_ptx.cuh"

namespace akv {
namespace {

constexpr int kThreads = 192;
constexpr int kKeys = 128;     // keys per KV tile
constexpr int kRows = 128;     // rows per query tile
constexpr int kLat = 512;      // latent width
constexpr int kPe = 64;        // K_pe width
constexpr int kQChunks = (kLat + kPe) / 64;  // 9 chunks of the QK contraction
constexpr int kVChunks = 256 / 64;           // 4 chunks of one output half
constexpr int kRing = 4;
constexpr int kMaxRuns = 8;  // runs per 128-key tile: 128 / page, page >= 16
constexpr uint32_t kChunk = 128 * 128;       // 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr int32_t kErrTimeout = 7;

// shared memory layout (bytes)
constexpr uint32_t kQ = 0;                          // 9 chunks of Q
constexpr uint32_t kSlots = kQ + kQChunks * kChunk;  // ring
constexpr uint32_t kColE = kSlots + kRing * kChunk;  // int32[128]
constexpr uint32_t kBars = kColE + 128 * 4;
constexpr uint32_t kBytes = kBars + 256;

enum Bar { kBarQ = 0, kBarFull0, kBarEmpty0 = kBarFull0 + kRing, kBarS0 = kBarEmpty0 + kRing, kBarP = kBarS0 + 2,
           kBarO, kBarFin, kNumBars };
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

// Chunks are loaded in the order the MMA thread consumes them:
//   QK chunks of tile 0, then for each tile j: QK chunks of tile j+1 (if
//   any), PV chunks of tile j.
// Stream position ld goes to ring slot ld % kRing.  chunk_at() maps a stream
// position to (tile, chunk), chunk < 9: QK (latent 0..7, K_pe 8), 9..12: PV.
constexpr int kPerTile = kQChunks + kVChunks;

__device__ __forceinline__ void chunk_at(int ld, int n_tiles, int& tile, int& chunk) {
  if (ld < kQChunks) {
    tile = 0;
    chunk = ld;
    return;
  }
  int rest = ld - kQChunks;
  // blocks of (QK of j+1, PV of j) for j = 0 .. n-2 (13 chunks each), then PV of n-1
  const int j = rest / kPerTile;
  if (j < n_tiles - 1) {
    const int c = rest % kPerTile;
    if (c < kQChunks) {
      tile = j + 1;
      chunk = c;
    } else {
      tile = j;
      chunk = c;
    }
  } else {
    tile = n_tiles - 1;
    chunk = kQChunks + (rest - (n_tiles - 1) * kPerTile);
  }
}

__device__ __forceinline__ void produce(const AttnParams& p, const AttnWork& w, const AttnSeg& seg, uint32_t sbase,
                                        volatile int* abort_flag) {
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int G = p.group, tpt = kRows / G, rpt = kKeys / p.page;
  const int half = w.n_b;  // which 256 output columns
  const int q_tok0 = seg.q_row0 + w.qt0 * tpt;
  ptx::mbar_arrive_expect_tx(bar(kBarQ), kQChunks * kChunk);
  for (int c = 0; c < kQChunks; ++c)
    ptx::tma_load_3d(sbase + kQ + c * kChunk, &p.q_map, bar(kBarQ), c * 64, 0, q_tok0);
  const int layer_base = p.layer * p.n_pages;
  bool ok = true;
  int issued = 0;
  const int n_loc = min(max(w.n_a - w.t0, 0), w.t1 - w.t0);  // local tile j is global tile t0 + j
  // Pages of the runs of tiles j (cur), j + 1 (nxt) and j + 2 (nn, fetched
  // at the start of block j so the run-table loads are in flight a whole
  // block before their first TMA).  Past the last run the segment's first
  // page stands in (finite values, masked out).
  const int2 first = *reinterpret_cast<const int2*>(p.runs + seg.run_off);
  int ck[kMaxRuns], cv[kMaxRuns], xk[kMaxRuns], xv[kMaxRuns], nk[kMaxRuns], nv[kMaxRuns];
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
  // A tile whose runs sit on consecutive pages loads each chunk with one
  // copy (the tile map's box spans 128 / page pages).
  auto consecutive = [&](const int (&pg)[kMaxRuns]) {
    bool c = true;
#pragma unroll
    for (int g = 1; g < kMaxRuns; ++g) c = c && (g >= rpt || pg[g] == pg[0] + g);
    return c;
  };
  fetch(0, ck, cv);
  if (n_loc > 1) fetch(1, xk, xv);
  for (int ld = 0; ld < n_loc * kPerTile; ++ld) {
    int j, c;
    chunk_at(ld, n_loc, j, c);
    if (ld >= kQChunks && (ld - kQChunks) % kPerTile == 0) {  // start of block b: QK of b + 1, PV of b
      const int b = (ld - kQChunks) / kPerTile;
      if (b >= 1) {
#pragma unroll
        for (int g = 0; g < kMaxRuns; ++g) {
          ck[g] = xk[g];
          cv[g] = xv[g];
          xk[g] = nk[g];
          xv[g] = nv[g];
        }
      }
      if (b + 2 < n_loc) fetch(b + 2, nk, nv);
    }
    const int slot = ld % kRing, use = ld / kRing;
    if (use >= 1 && !ptx::mbar_wait(bar(kBarEmpty0 + slot), (use - 1) & 1, abort_flag, kWaitLimitNs)) {
      ok = false;
      break;
    }
    // chunk c < 8: latent columns 64c (QK); c == 8: K_pe; c > 8: latent columns of this half (PV)
    const bool pe = c == kLat / 64;
    const int col = c < kQChunks ? (pe ? 0 : 64 * c) : 256 * half + 64 * (c - kQChunks);
    const CUtensorMap* map = pe ? &p.k_map : &p.v_map;
    const uint32_t dst = sbase + kSlots + slot * kChunk;
    // tile j is the current block's tile (cur) or, for QK chunks after the first tile, the next (nxt)
    const bool use_next = ld >= kQChunks && c < kQChunks;
    ptx::mbar_arrive_expect_tx(bar(kBarFull0 + slot), kChunk);
    int pgs[kMaxRuns];
#pragma unroll
    for (int g = 0; g < kMaxRuns; ++g) pgs[g] = use_next ? (pe ? xk[g] : xv[g]) : (pe ? ck[g] : cv[g]);
    if (consecutive(pgs)) {
      ptx::tma_load_4d(dst, pe ? &p.k_tile_map : &p.v_tile_map, bar(kBarFull0 + slot), col, 0, 0, pgs[0]);
    } else {
#pragma unroll
      for (int g = 0; g < kMaxRuns; ++g) {
        if (g >= rpt) break;
        ptx::tma_load_4d(dst + g * p.page * 128, map, bar(kBarFull0 + slot), col, 0, 0, pgs[g]);
      }
    }
    issued = ld + 1;
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 10, 0);
    *abort_flag = 1;
  }
  ptx::mbar_wait(bar(kBarQ), 0, abort_flag, kDrainLimitNs);
#pragma unroll
  for (int s = 0; s < kRing; ++s) {
    const int uses = issued > s ? (issued - s + kRing - 1) / kRing : 0;
    if (uses) ptx::mbar_wait(bar(kBarFull0 + s), (uses - 1) & 1, abort_flag, kDrainLimitNs);
  }
}

// --------------------------------------------------------------------- MMA
__device__ __forceinline__ void issue_mma(const AttnParams& p, const AttnWork& w, uint32_t sbase, uint32_t tmem,
                                          volatile int* abort_flag) {
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  constexpr uint32_t idesc_qk = ptx::idesc_bf16(kRows, kKeys, false);
  constexpr uint32_t idesc_pv = ptx::idesc_bf16(kRows, 64, true);
  const uint32_t tO = tmem + 256;
  const int n = min(max(w.n_a - w.t0, 0), w.t1 - w.t0);
  int ld = 0;
  bool ok = ptx::mbar_wait(bar(kBarQ), 0, abort_flag, kWaitLimitNs);
  auto next_chunk = [&]() -> uint32_t {  // wait for the chunk at stream position ld; its slot address
    const int slot = ld % kRing;
    ok = ok && ptx::mbar_wait(bar(kBarFull0 + slot), (ld / kRing) & 1, abort_flag, kWaitLimitNs);
    ptx::tc_fence_after();
    return sbase + kSlots + slot * kChunk;
  };
  auto release = [&]() {
    ptx::mma_commit(bar(kBarEmpty0 + ld % kRing));
    ++ld;
  };
  // Descriptors are built once and advanced by constants (only the start
  // address changes); the MMA thread shares its sub-partition with softmax.
  const uint64_t qd0 = ptx::smem_desc(sbase + kQ, 16, 1024);
  auto qk = [&](int j) {
    const uint32_t tS = tmem + 128u * (j & 1);
#pragma unroll 1
    for (int c = 0; c < kQChunks && ok; ++c) {
      const uint32_t kt = next_chunk();
      if (!ok) break;
      const uint64_t kd = ptx::smem_desc(kt, 16, 1024), qd = ptx::desc_advance(qd0, c * kChunk);
      ptx::mma_bf16(tS, qd, kd, idesc_qk, c > 0);
#pragma unroll
      for (int ks = 1; ks < 4; ++ks)
        ptx::mma_bf16(tS, ptx::desc_advance(qd, ks * 32), ptx::desc_advance(kd, ks * 32), idesc_qk, 1);
      release();
    }
    if (ok) ptx::mma_commit(bar(kBarS0 + (j & 1)));
  };
  if (ok && n > 0) qk(0);
  for (int j = 0; j < n && ok; ++j) {
    if (j + 1 < n) qk(j + 1);
    if (!ok) break;
    if (!(ok = ptx::mbar_wait(bar(kBarP), j & 1, abort_flag, kWaitLimitNs))) break;
    ptx::tc_fence_after();
    const uint32_t tP = tmem + 128u * (j & 1);  // P of tile j, packed over S
#pragma unroll 1
    for (int i = 0; i < kVChunks && ok; ++i) {
      const uint32_t vt = next_chunk();
      if (!ok) break;
      const uint64_t vd = ptx::smem_desc(vt, kChunk, 1024);
      ptx::mma_bf16_tmem_a(tO + 64u * i, tP, vd, idesc_pv, j > 0);
#pragma unroll
      for (int ks = 1; ks < kKeys / 16; ++ks)
        ptx::mma_bf16_tmem_a(tO + 64u * i, tP + 8u * ks, ptx::desc_advance(vd, ks * 2048), idesc_pv, 1);
      release();
    }
    if (ok) ptx::mma_commit(bar(kBarO));
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 11, 0);
    *abort_flag = 1;
  }
  ptx::mma_commit(bar(kBarFin));
  ptx::mbar_wait(bar(kBarFin), 0, abort_flag, kDrainLimitNs);
}

// ----------------------------------------------------------------- softmax
__device__ __forceinline__ void softmax(const AttnParams& p, const AttnWork& w, const AttnSeg& seg, uint8_t* smem,
                                        uint32_t sbase, uint32_t tmem, volatile int* abort_flag) {
  const int n = min(max(w.n_a - w.t0, 0), w.t1 - w.t0);  // local tile j is global tile t0 + j
  const uint32_t bars = sbase + kBars;
  auto bar = [&](int i) { return bars + 8u * uint32_t(i); };
  const int quad = (threadIdx.x / 32) & 3;  // warps 2..5 -> TMEM lane quadrants 2, 3, 0, 1
  const int lane = threadIdx.x % 32;
  const int r = quad * 32 + lane;
  const uint32_t lane_addr = uint32_t(quad * 32) << 16;
  const uint32_t tO = tmem + 256;
  const int G = p.group, tpt = kRows / G, rpt = kKeys / p.page;
  const int t_loc = r / G, g = r % G;
  const int qi = w.qt0 * tpt + t_loc;
  const bool row_valid = qi < seg.q_len;
  const int lim = seg.kv_len - seg.q_len + (row_valid ? qi : seg.q_len - 1);
  const float sl2 = p.scale_log2;
  int* colE = reinterpret_cast<int*>(smem + kColE);
  int page_shift = 4;
  while ((1 << page_shift) < p.page) ++page_shift;
  const int sl_own = r & (p.page - 1);
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  // (lohi, es) of the run holding key column r of the current tile, fetched one tile ahead;
  // lo = hi = 0 past the segment's last run, so no slot matches
  const int2* run_le = reinterpret_cast<const int2*>(p.runs + seg.run_off);
  int2 run_cur = make_int2(0, 0);
  {
    const int ri0 = w.t0 * rpt + (r >> page_shift);
    if (ri0 < seg.n_runs) run_cur = run_le[2 * ri0 + 1];
  }
  for (int j = 0; j < n; ++j) {
    const uint32_t tS = tmem + 128u * (j & 1);
    ok = ptx::mbar_wait(bar(kBarS0 + (j & 1)), (j >> 1) & 1, abort_flag, kWaitLimitNs);
    if (!ptx::bar_red_and(1, 128, ok)) {
      ok = false;
      break;
    }
    int e = INT_MAX;  // entry index of key column r (INT_MAX: none)
    {
      const int lo = run_cur.x & 0xffff, hi = run_cur.x >> 16;
      if (sl_own >= lo && sl_own < hi) e = run_cur.y + (sl_own - lo);
      colE[r] = e;
      const int ri = (w.t0 + j + 1) * rpt + (r >> page_shift);
      run_cur = ri < seg.n_runs ? run_le[2 * ri + 1] : make_int2(0, 0);
    }
    const bool all_valid = ptx::bar_red_and(1, 128, e != INT_MAX);
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
    if (j > 0) {  // O stable (PV of tile j-1 done) before any rescale
      ok = ptx::mbar_wait(bar(kBarO), (j - 1) & 1, abort_flag, kWaitLimitNs);
      if (!ptx::bar_red_and(1, 128, ok)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c = 0; c < 256 / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_load32(tO + lane_addr + c * 32, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          ptx::tmem_store32(tO + lane_addr + c * 32, o);
        }
      }
    }
    l_run = l_run * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
    m_run = m_use;
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(kBarP));
  }
  if (ok && n > 0) {
    ok = ptx::mbar_wait(bar(kBarO), (n - 1) & 1, abort_flag, kWaitLimitNs);
    ok = ptx::bar_red_and(1, 128, ok);
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout, blockIdx.x, 12, 0);
    *abort_flag = 1;
    return;
  }
  ptx::tc_fence_after();
  const int half = w.n_b;
  if (w.part >= 0) {
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
    return;
  }
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

__global__ void __launch_bounds__(kThreads, 1) segment_attn_mla_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bars = sbase + kBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBars + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBars + 8 * kNumBars + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const AttnWork w = p.work[blockIdx.x];
  const AttnSeg seg = p.segs[w.seg];
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) ptx::mbar_init(bars + 8u * i, i == kBarP ? 128 : 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0) {
    if (lane == 0) produce(p, w, seg, sbase, abort_flag);
  } else if (warp == 1) {
    if (lane == 0) issue_mma(p, w, sbase, tmem, abort_flag);
  } else {
    softmax(p, w, seg, smem, sbase, tmem, abort_flag);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_segment_attn_mla(const AttnParams& p, cudaStream_t st) {
  if (p.n_work <= 0) return cudaSuccess;
  const int smem = int(kBytes) + 1024;
  cudaError_t e = cudaFuncSetAttribute(segment_attn_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  segment_attn_mla_kernel<<<p.n_work, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace akv
