// Internal interface between the host engine (engine.cpp) and the CUDA
// kernels.  Nothing here is part of the public C ABI.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace akv {

// Device error word, written by kernels with atomicCAS from 0 so the first
// failure wins.  code is an akv_status value; info holds where it happened.
struct DevErr {
  int32_t code;
  int32_t info[3];
};

#ifdef __CUDACC__
// Device-side descriptor checks of the -DAKV_CHECKED build: a failed check
// records AKV_ERR_DEVICE (8) with where it happened and the kernel skips the
// work the descriptor names (or, for attention, the whole CTA returns before
// touching memory).  Never a trap or an assert.  err may be null.
__device__ __forceinline__ void report_device_error(DevErr* err, int where, int a, int b) {
  if (err && atomicCAS(&err->code, 0, 8) == 0) {
    err->info[0] = where;
    err->info[1] = a;
    err->info[2] = b;
  }
}
#endif

// One flush run: rows [lo, hi) of K page src are rotated by the shift whose
// (cos, sin) table row is didx and written to the same rows of page dst
// (dst == src: in place; dst != src: copy-on-write).
struct RunDesc {
  int32_t src;
  int32_t dst;
  int32_t lohi;  // lo | hi << 16
  int32_t didx;
};

// One compaction copy run: n consecutive slots from (src_k, src_v) at src_lo
// to (dst_k, dst_v) at dst_lo; the key rows are rotated by shift table row
// didx (-1: copied as they are).
struct CopyRun {
  int32_t src_k;
  int32_t src_v;
  int32_t dst_k;
  int32_t dst_v;
  int32_t src_lo;
  int32_t dst_lo;
  int32_t n;
  int32_t didx;
};

// One attention run: rows [lo, hi) of K page kp / V page vp hold the
// segment's entries es .. es + (hi - lo) - 1.
struct AttnRun {
  int32_t kp;
  int32_t vp;
  int32_t lohi;  // lo | hi << 16
  int32_t es;
};

struct AttnSeg {
  int32_t run_off;  // first run in the run table
  int32_t n_runs;
  int32_t kv_len;
  int32_t q_len;
  int32_t q_row0;
  int32_t ent_off;   // attention mass: first entry of this segment in the entry -> token table
  int32_t mass_off;  // attention mass: first output element of this segment
  int32_t pad;
};

// One CTA's work: two consecutive 128-row query tiles (A = qt0, B = qt0 + 1)
// of segment seg for kv head kvh (GQA), or one query tile qt0 and output half
// n_b (MLA).  n_a / n_b: KV tiles each query tile reads in all (up to the causal
// limit of its last row); n_b = 0 when the segment has no tile B.  The CTA
// reads KV tiles [t0, t1) of those.  part < 0: it owns the whole range and
// writes the final output; part >= 0: it writes unnormalised partial results
// to partial slot `part`; the part that finishes last merges them all.
struct AttnWork {
  int32_t seg;
  int32_t kvh;   // GQA: kv head; MLA: flags (kShadow)
  int32_t qt0;
  int32_t n_a;
  int32_t n_b;
  int32_t t0;
  int32_t t1;
  int32_t part;  // partial slot of this split part, -1 when the item is not split
  int32_t comb;  // its CombineItem
};

// MLA work runs as CTA pairs (entries 2i, 2i + 1: two query tiles, one KV
// range, one output half).  A segment with an odd number of query tiles
// fills its last pair with a shadow: it repeats its partner's tile so the
// pair's MMAs have both row halves, and writes nothing.
constexpr int32_t kShadow = 1;

// One split work item: its parts own partial slots [part0, part0 + n_parts);
// count[t] is the ticket counter of query tile t, zero at launch (the host
// uploads it with the work list), taken by each part once its partial is
// written; the part that draws the last ticket merges.
struct CombineItem {
  int32_t part0;
  int32_t n_parts;
  int32_t count[2];
};

struct AttnParams {
  CUtensorMap q_map;  // Q [n_q_rows][Hq][d_qk], box {64, G, 128/G}
  CUtensorMap k_map;  // rotated pool, [L*P][H][page][d_rot], box {64, page, 1, 1}
  CUtensorMap v_map;  // value pool,  [L*P][H][page][d_v],   box {64, page, 1, 1}
  CUtensorMap k_tile_map;  // GQA: as k_map, box {64, page, 1, 128 / page}: a tile's consecutive pages at once;
                           // MLA: box {64, min(page, 64), 1, max(64 / page, 1)}: the pages of 64 keys
  CUtensorMap v_tile_map;  // as v_map, with k_tile_map's box
  const AttnRun* runs;
  const AttnSeg* segs;
  const AttnWork* work;
  void* o;            // bf16 [n_q_rows][Hq][d_v]
  float* lse;         // float [n_q_rows][Hq] or null
  float* partial;     // split-KV scratch: per part [tile][width + 2][128 rows] floats (O columns, m, l)
  CombineItem* comb;  // split items (ticket counters), null when nothing is split
  int32_t comb_tiles; // query tiles per partial slot (2 for GQA pairs, 1 under MLA)
  DevErr* err;
  float scale_log2;   // softmax scale * log2(e)
  int32_t n_work;
  const int32_t* cta_units;  // persistent schedule: CTA b runs units [cta_units[b], cta_units[b + 1]) of work;
                             // null: CTA b runs unit b
  int32_t n_cta;             // CTAs of the persistent schedule (grid size when cta_units is set)
  // Fused rotation: the kernel rotates each K row of run r by the shift of
  // table row run_didx[r] (-1: none) on its way to the tensor core.
  const int32_t* run_didx;   // per run, or null
  const float2* cs;          // (cos, sin)(delta * theta_j): [shifts][d_rot / 2], float64-evaluated
  int32_t rope_half;         // pair layout: 0 interleaved (2j, 2j+1), 1 half-split (j, j + d/2)
  int32_t fused;             // 1: launch the fused-rotation variant
  int32_t layer;
  int32_t n_pages;
  int32_t n_layers;
  int32_t hq;
  int32_t group;      // query heads per kv head
  int32_t page;
  int32_t width;      // output columns one CTA writes (d_v, or d_v / 2 under MLA)
  int32_t dv;         // output row width (d_v)
  uint64_t wait_ns;   // limit of every bounded wait (a wait that runs out reports AKV_ERR_DEVICE_TIMEOUT)
  int32_t load_cap;   // test hook (GQA): K/V tile copies the producer of a CTA issues at most; < 0: no cap
  int32_t n_segs;     // entries of segs (bounds of the checked build)
  int32_t n_runs;     // entries of runs
  int32_t n_q_rows;   // rows of Q, O and lse
};

// Attention-mass pass (GQA): one CTA per (segment, kv head, query tile);
// work[i].n_a = the KV tiles that query tile reads.
struct MassParams {
  CUtensorMap q_map;       // as AttnParams
  CUtensorMap k_map;
  CUtensorMap k_tile_map;
  const AttnRun* runs;
  const AttnSeg* segs;
  const AttnWork* work;
  const float* lse;        // natural-log softmax normaliser [n_q_rows][Hq] from the attention pass
  const int32_t* ent_tok;  // per segment entry: its logical token index
  float* mass;             // [sum of segments' kv_end], zeroed by the host, accumulated with atomics
  DevErr* err;
  float scale_log2;
  int32_t n_work;
  int32_t layer;
  int32_t n_pages;
  int32_t hq;
  int32_t group;
  int32_t page;
  int32_t n_segs;     // bounds of the checked build
  int32_t n_runs;
  int32_t n_q_rows;
  int32_t pad;
};

#if defined(__CUDACC__) && defined(AKV_CHECKED)
// Checked build: the descriptors one attention work item reads name a
// segment of the table, a run range inside the run table whose runs name
// existing pages and a non-empty row range of one page, and query rows inside
// Q.  Threads of a CTA split the run checks by `lane` of `lanes`.
__device__ __forceinline__ bool attn_item_ok(const AttnWork& w, const AttnSeg* segs, const AttnRun* runs, int n_segs,
                                             int n_runs, int n_q_rows, int n_pages, int page, int lane, int lanes) {
  if (w.seg < 0 || w.seg >= n_segs || w.t0 < 0 || w.t0 > w.t1 || w.qt0 < 0) return false;
  const AttnSeg sg = segs[w.seg];
  if (sg.run_off < 0 || sg.n_runs < 1 || sg.run_off + sg.n_runs > n_runs || sg.q_row0 < 0 || sg.q_len < 0 ||
      sg.q_row0 + sg.q_len > n_q_rows || sg.kv_len < sg.q_len)
    return false;
  bool ok = true;
  for (int i = lane; i < sg.n_runs && ok; i += lanes) {
    const AttnRun r = runs[sg.run_off + i];
    const int lo = r.lohi & 0xffff, hi = r.lohi >> 16;
    ok = r.kp >= 0 && r.kp < n_pages && r.vp >= 0 && r.vp < n_pages && lo < hi && hi <= page && r.es >= 0;
  }
  return ok;
}
#endif

// Floats of one partial slot: tiles x 128 rows x (width + 2).
__host__ __device__ inline int64_t partial_floats(int tiles, int width) { return int64_t(tiles) * 128 * (width + 2); }

// Launchers; each returns the launch's cudaError_t.
cudaError_t launch_kv_write(const void* src_k, void* pool_k, const int32_t* rows_k, int dim_k, const void* src_v,
                            void* pool_v, const int32_t* rows_v, int dim_v, int64_t n, int n_layers, int heads,
                            int page, int64_t n_pages, int n_sm, DevErr* err, cudaStream_t st);

cudaError_t launch_compact_copy(void* kpool, void* vpool, const CopyRun* runs, const float2* cs, int n_runs,
                                int n_layers, int heads, int d_rot, int d_v, int page, int64_t n_pages, bool half,
                                int n_sm, DevErr* err, cudaStream_t st);

cudaError_t launch_attn_mass(const MassParams& p, int dim, cudaStream_t st);

cudaError_t launch_repos_rotate(void* kpool, const RunDesc* runs, const float2* cs, int n_runs,
                                int n_layers, int heads, int d_rot, int page, int64_t n_pages,
                                bool half_layout, DevErr* err, cudaStream_t st);

// Float32 debug mode of repos_rotate: rotated rows of each run go to
// out[L][total_rows][H][d_rot] (rows of run r start at row_off[r]); the pool
// is only read.
cudaError_t launch_repos_rotate_f32(const void* kpool, const RunDesc* runs, const float2* cs, const int32_t* row_off,
                                    int64_t total_rows, float* out, int n_runs, int n_layers, int heads, int d_rot,
                                    int page, int64_t n_pages, bool half_layout, DevErr* err, cudaStream_t st);

// dim: d_rot = d_v (GQA, 64 or 128).
cudaError_t launch_segment_attn(const AttnParams& p, int dim, cudaStream_t st);

// MLA variant: 16 query heads over one latent (d_v 512) + K_pe (64) per token;
// work items carry the output half (0 or 1) in n_b.
cudaError_t launch_segment_attn_mla(const AttnParams& p, cudaStream_t st);
int segment_attn_mla_slots();

// Merge split-KV partials: items [n_items], tiles_per_item query tiles of 128
// rows each, `width` output columns per part.
// Shared-memory bytes the attention kernel needs for head dimension dim.
int segment_attn_smem_bytes(int dim);

}  // namespace akv
