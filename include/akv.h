/*
 * akv.h -- C ABI of the GB300 agentic KV-cache engine (libakv.so).
 *
 * The engine keeps a paged bf16 KV cache for agent trajectories and applies
 * the cache operations an agent harness issues instead of editing its prompt:
 *
 *   append  add the K/V of new tokens            ("Cache Engineering for Agents"
 *   drop    hide a span from later attention       reading notes, section 1
 *   repos   move retained keys to new positions    "Problem & Solution")
 *   splice  replace a span by a stub (Leyline AMORTIZE)
 *   attend  segment-batch attention of new queries over each segment's pages
 *
 * Sources, cited by page title and section:
 *   [AKV-blog]  "AKV: Cache Engineering for Autonomous Agents and
 *               State-Preserving Prefix Invalidation Bypass"
 *   [AKV-notes] "Cache Engineering for Agents" (reading notes on Fu et al.)
 *   [Leyline]   "Leyline: KV Cache Directives for Agentic Inference"
 *
 * Conventions (apply to every function):
 *   - Every function returns akv_status.  A call that fails with AKV_ERR_ARG,
 *     AKV_ERR_RANGE, AKV_ERR_NO_PAGES or AKV_ERR_OVERFLOW changes nothing.
 *     AKV_ERR_CUDA means a CUDA call failed; the context should then be
 *     destroyed.  akv_last_error() gives a message for the last failure.
 *   - Spans [s, e) are half-open logical token indices of a sequence as the
 *     harness sees it.  splice shifts the logical indices of later tokens.
 *   - Positions and shifts are int32; an operation that would take a
 *     position or a composed shift outside int32 fails with AKV_ERR_OVERFLOW.
 *     A shift delta moves a key from position p to p + delta.
 *   - The K/V pools are device memory owned by the caller and must stay
 *     allocated while the context lives.  Pool memory must hold finite values
 *     before first use (zero it): attention reads whole pages and masks the
 *     slots it does not need, and a NaN there would leak through 0 * NaN.
 *   - Data pointers passed to append / splice / attend may be device memory
 *     or host memory (pinned for asynchronous copies).  Host inputs are copied
 *     into library-owned device staging memory on the context's own copy
 *     stream, which does not wait for earlier work on the given stream (the
 *     copy overlaps the kernels of earlier calls); the given stream waits for
 *     the copy before the kernel that reads it.  So a host input must hold its
 *     final contents when the call is made, and stay unchanged until the given
 *     stream has passed the call.  A host output is copied back on the given
 *     stream, so synchronise it before reading the output.  (While the given
 *     stream is being captured into a graph, inputs are copied on it.)
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All device work of a call is enqueued on it asynchronously;
 *     host bookkeeping changes at call time.  Use one stream per context, or
 *     order the streams yourself.
 *   - A context is not thread-safe; one host thread at a time.
 *   - No C++ exception crosses this boundary.
 */
#ifndef AKV_H
#define AKV_H

#include <stdint.h>

#if defined(__GNUC__)
#define AKV_API __attribute__((visibility("default")))
#else
#define AKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum akv_status {
  AKV_OK = 0,
  AKV_ERR_ARG = 1,            /* bad argument (null pointer, dead sequence, bad config) */
  AKV_ERR_RANGE = 2,          /* a span or index outside the sequence or buffer */
  AKV_ERR_NO_PAGES = 4,       /* the page pool cannot supply the pages needed */
  AKV_ERR_OVERFLOW = 5,       /* a position or composed shift would leave int32 */
  AKV_ERR_CUDA = 6,           /* a CUDA runtime/driver call failed */
  AKV_ERR_DEVICE_TIMEOUT = 7, /* a kernel gave up a bounded wait (see akv_check_device_error) */
  AKV_ERR_DEVICE = 8          /* a kernel's own bounds check failed */
} akv_status;

typedef enum akv_layout {
  AKV_LAYOUT_GQA = 0, /* K and V per kv head; all of K is rotated */
  AKV_LAYOUT_MLA = 1  /* K_pe (rotated) + one latent shared as K_nope and V ([Leyline] "Method") */
} akv_layout;

typedef enum akv_rope_layout {
  AKV_ROPE_INTERLEAVED = 0, /* pairs (2j, 2j+1), as [AKV-blog] section 2 writes the rotation */
  AKV_ROPE_HALF = 1         /* pairs (j, j + d_rot/2) */
} akv_rope_layout;

/* Model and pool shape of one context. */
typedef struct akv_config {
  int32_t layout;       /* akv_layout */
  int32_t n_layers;     /* layers held in each pool */
  int32_t n_q_heads;    /* query heads; a multiple of n_kv_heads, n_q_heads/n_kv_heads divides 128 */
  int32_t n_kv_heads;   /* kv heads (GQA); must be 1 under MLA */
  int32_t d_rot;        /* rotated key width: head_dim (GQA) or K_pe width (MLA); even */
  int32_t d_v;          /* value width: head_dim (GQA, = d_rot) or latent width (MLA) */
  int32_t page_size;    /* tokens per page: 16, 32, 64 or 128 */
  int32_t n_pages;      /* pages in each pool */
  int32_t rope_layout;  /* akv_rope_layout */
  int32_t reserved;     /* must be 0 */
  double rope_base;     /* RoPE base: theta_j = rope_base^(-2j/d_rot) */
} akv_config;

/* Caller-owned device pools (bf16).  Row-major layouts:
 *   k_pool [n_layers][n_pages][n_kv_heads][page_size][d_rot]   (K, or K_pe under MLA)
 *   v_pool [n_layers][n_pages][n_kv_heads][page_size][d_v]     (V, or the latent under MLA)
 * Both base addresses must be 16-byte aligned (TMA). */
typedef struct akv_pools {
  void* k_pool;
  void* v_pool;
} akv_pools;

/* One attention segment ([AKV-notes] section 3 "Segment-Batch Attention").
 * The segment sees the visible (not dropped) tokens of sequence `seq` in
 * logical indices [0, kv_end), minus the `n_hide` extra spans in `hide`
 * (host array of [a, b) pairs), in logical order.  Its queries are tokens
 * [kv_end - q_len, kv_end), which must be visible, not hidden, and hence the
 * last q_len entries; query row i sees entries j <= kv_len - q_len + i
 * (causal, aligned bottom-right).  Their Q rows are q[q_row0 .. q_row0+q_len). */
typedef struct akv_segment {
  int32_t seq;
  int32_t q_len;
  int64_t kv_end;
  int64_t q_row0;
  const int64_t* hide;
  int32_t n_hide;
  int32_t reserved;   /* must be 0 */
} akv_segment;

/* Extended radix tree ([AKV-blog] section 3 "Resolving History Dependence via
 * Extended Radix Trees"; [AKV-notes] "Cache Reuse Matching Rules").  A path is
 * a list of items: a cached token (kind AKV_ITEM_TOKEN, a = token id, b = the
 * position its cached key encodes) or a cache-operation marker (kind >= 1 is
 * the caller's operation code, a, b, c its arguments), in the order they were
 * applied.  Tokens of a path are the logical tokens of the sequence that holds
 * it, in order. */
#define AKV_ITEM_TOKEN 0
typedef struct akv_item {
  int32_t kind;
  int32_t a;
  int32_t b;
  int32_t c;
} akv_item;

#define AKV_MATCH_NONE 0
#define AKV_MATCH_EXACT 1      /* same tokens, positions and operations: reuse as is */
#define AKV_MATCH_RETRIGGER 2  /* same tokens and operations, other positions: reuse after rotating keys */
typedef struct akv_match {
  int32_t kind;       /* AKV_MATCH_* */
  int32_t seq;        /* tree-held sequence with the matched prefix (-1: none) */
  int64_t n_items;    /* request items matched */
  int64_t n_tokens;   /* tokens among them */
} akv_match;

/* Per-kernel launch statistics collected while profiling is enabled. */
typedef struct akv_kernel_stats {
  int64_t launches[5];   /* [0] kv_write  [1] repos_rotate  [2] segment_attn  [3] compact_copy  [4] attn_mass */
  double ms[5];          /* summed CUDA-event time of those launches (events around each launch), milliseconds */
  double bytes[5];       /* algorithmic bytes moved (kv_write, repos_rotate, compact_copy) */
  double flops[5];       /* algorithmic FLOPs (segment_attn: QK^T and PV over the visible pairs; attn_mass:
                          * QK^T and the column-sum product, 2 x 128 FLOPs per visible pair and head) */
} akv_kernel_stats;

typedef struct akv_ctx akv_ctx;

/* Create a context.  pools == NULL gives a metadata-only context: every
 * bookkeeping rule runs, no CUDA call is made and data pointers are ignored
 * (for planning and for checking the bookkeeping on hosts without a GPU).
 * Otherwise the current CUDA device is used and TMA descriptors of the
 * pools are built once here.  *out receives the context. */
AKV_API akv_status akv_create(const akv_config* cfg, const akv_pools* pools, akv_ctx** out);

/* Destroy a context and free the library-owned device and host memory.
 * Synchronises the device work the context has enqueued. */
AKV_API akv_status akv_destroy(akv_ctx* ctx);

/* Message of the last failure on this context ("" if none).  Valid until the next call. */
AKV_API const char* akv_last_error(const akv_ctx* ctx);

/* "kv_alloc": a new empty sequence; ids are the lowest unused non-negative integers. */
AKV_API akv_status akv_seq_alloc(akv_ctx* ctx, int32_t* seq_out);

/* A new sequence sharing tokens [0, n_prefix) of `src` by page reference
 * (a shared radix prefix; [AKV-blog] section 3, copy-on-write page references).
 * Copies no data.  Pending shifts and drop marks are inherited. */
AKV_API akv_status akv_seq_fork(akv_ctx* ctx, int32_t src, int64_t n_prefix, int32_t* seq_out);

/* Release a sequence; pages no live sequence references return to the pool. */
AKV_API akv_status akv_seq_free(akv_ctx* ctx, int32_t seq);

/* Logical length of a sequence (tokens, including dropped ones). */
AKV_API akv_status akv_seq_len(akv_ctx* ctx, int32_t seq, int64_t* n_out);

/* "append" ([AKV-notes] section 1): add n tokens whose keys are already
 * RoPE-rotated at their positions.
 *   k: bf16 [n_layers][n][n_kv_heads][d_rot]   v: bf16 [n_layers][n][n_kv_heads][d_v]
 *   pos: host int32[n], or NULL = last position + 1 counting up (0 if empty).
 * The page of the last token is filled further when both its K and V page
 * are referenced by this sequence only; otherwise new pages are opened
 * (lowest free id first). */
AKV_API akv_status akv_append(akv_ctx* ctx, int32_t seq, int64_t n, const void* k, const void* v,
                      const int32_t* pos, void* stream);

/* "drop" ([AKV-blog] section 2 "The Drop Primitive"): tokens [s, e) become
 * invisible to later attention.  Frees nothing and writes no device memory. */
AKV_API akv_status akv_drop(akv_ctx* ctx, int32_t seq, int64_t s, int64_t e);

/* "repos" ([AKV-blog] section 2 "The Repos Primitive and Rotary Position
 * Embeddings"; [Leyline] "Method", composition R(a)R(b) = R(a+b)): record a
 * shift `delta` for tokens [s, e).  Shifts compose per token by addition; the
 * keys are rotated once, by the composed shift, at the next flush. */
AKV_API akv_status akv_repos(akv_ctx* ctx, int32_t seq, int64_t s, int64_t e, int32_t delta);

/* A turn's list of drop / repos directives for one sequence in one call
 * ([Leyline] "Method": directives arrive as a list and compose by addition).
 * Equivalent to calling akv_drop / akv_repos once per entry, in order, but
 * all or nothing: on an error (AKV_ERR_ARG for an unknown kind, AKV_ERR_RANGE
 * for a span outside the sequence, AKV_ERR_OVERFLOW) no entry is applied. */
#define AKV_EDIT_DROP 1
#define AKV_EDIT_REPOS 2
typedef struct akv_edit_op {
  int32_t kind;   /* AKV_EDIT_DROP or AKV_EDIT_REPOS */
  int32_t delta;  /* shift of a repos (ignored for a drop) */
  int64_t s;      /* span [s, e), logical token indices */
  int64_t e;
} akv_edit_op;
AKV_API akv_status akv_edit(akv_ctx* ctx, int32_t seq, const akv_edit_op* ops, int32_t n_ops);

/* Leyline AMORTIZE splice ([Leyline] "Method", D = (s, e, R, AMORTIZE)):
 * remove tokens [s, e) from the sequence, insert n_stub stub tokens at s
 * (written to fresh pages), and shift every later token by
 * n_stub - (e - s).  Under MLA only K_pe is rotated; the latent (K_nope and V)
 * is untouched.  k_stub / v_stub as in akv_append with n = n_stub; pos NULL =
 * the position of token s counting up. */
AKV_API akv_status akv_splice(akv_ctx* ctx, int32_t seq, int64_t s, int64_t e, int64_t n_stub,
                      const void* k_stub, const void* v_stub, const int32_t* pos, void* stream);

/* Materialise pending shifts (the repos_rotate kernel; [AKV-blog] section 2
 * "The Repos Primitive and Rotary Position Embeddings": a retained key moves
 * from position m to m + delta by one more rotation, K' = R(delta) K, since
 * R(a) R(b) = R(a + b); [Leyline] "Method": several directives collapse into
 * one composed shift per token, and under MLA only K_pe rotates).  Every
 * visible token with a pending shift is rotated once, K'[i] = R(delta_i) K[i],
 * in fp32 with one rounding to bf16.  A K page referenced by this sequence
 * only is rotated in place; a shared one is first copied (copy-on-write of
 * the K page only, [AKV-notes] section 3 "Cache Management").  seq = -1
 * flushes every live sequence in increasing id order. */
AKV_API akv_status akv_flush(akv_ctx* ctx, int32_t seq, void* stream);

/* Segment-batch attention for one layer (the segment_batch_attn kernel;
 * [AKV-notes] section 3 "Segment-Batch Attention": the incoming queries are
 * split into segments by the history they see, and each segment runs
 * ordinary causal attention over the KV pages it selects, with no dense
 * custom mask; [AKV-blog] section 4 "Segment-Batch Attention Kernel
 * Architecture": heterogeneous segments share one launch).  Flushes the
 * segments' sequences first, then one launch covers every segment.
 *   q:   bf16 [n_q_rows][n_q_heads][d_qk]  (d_qk = d_rot under GQA; d_v + d_rot
 *        under MLA, laid out [latent part | rope part]); already RoPE'd.
 *   o:   bf16 [n_q_rows][n_q_heads][d_v]; rows outside the segments are not written.
 *   lse: float [n_q_rows][n_q_heads] natural-log softmax normaliser, or NULL.
 *   scale: softmax scale (1/sqrt(d_k)).
 * Query head h reads kv head h / (n_q_heads / n_kv_heads). */
AKV_API akv_status akv_attend(akv_ctx* ctx, int32_t layer, const akv_segment* segs, int32_t n_segs,
                      const void* q, int64_t n_q_rows, void* o, float* lse, float scale,
                      void* stream);

/* Insert the path `items[0 .. n)` held by live sequence `seq` (its first
 * n_tokens(items) logical tokens).  When the path adds tree nodes the tree
 * forks `seq` (shared pages, reference-counted) and keeps that fork as the
 * holder of the new nodes; *tree_seq_out (nullable) receives it, or -1 when
 * the path was already present.  Items are compared exactly. */
AKV_API akv_status akv_tree_insert(akv_ctx* ctx, const akv_item* items, int64_t n, int32_t seq,
                           int32_t* tree_seq_out);

/* Match a request path: the longest exact-match prefix, replaced by the
 * longest history-compatible branch (same tokens and operations, positions
 * free) only if that is strictly longer; a walk stops at the first item that
 * differs.  Ties between equally long branches go to the earliest inserted
 * holder. */
AKV_API akv_status akv_tree_match(akv_ctx* ctx, const akv_item* items, int64_t n, akv_match* out);

/* Match, then give the request a new sequence holding the matched prefix:
 * a fork of the holder (copy-on-write page references); on a retrigger match
 * every token is also repositioned by (request position - cached position)
 * and flushed, i.e. the repos_rotate kernel rotates the keys into
 * copy-on-write pages.  *seq_out = -1 when nothing matches. */
AKV_API akv_status akv_tree_reuse(akv_ctx* ctx, const akv_item* items, int64_t n, akv_match* out, int32_t* seq_out,
                          void* stream);

/* Forget every path and free the tree's sequences. */
AKV_API akv_status akv_tree_clear(akv_ctx* ctx);

/* Fragmentation of a sequence's pages ([AKV-blog] "Dilemma 2: Memory
 * Fragmentation in Paged Pools"): 1 - visible tokens / (K pages * page_size),
 * the share of the slots of its K pages holding none of its visible tokens
 * (0 for an empty sequence).  The page's policy (compact above 40 %) is the
 * caller's. */
AKV_API akv_status akv_fragmentation(akv_ctx* ctx, int32_t seq, double* frac_out);

/* Compaction (same passage: surviving blocks copied into contiguous physical
 * spans; the compact_copy kernel).  The visible tokens of `seq`, in logical
 * order, are copied densely into fresh pages (lowest free ids, one K and one
 * V page per page_size tokens); a pending shift is applied to the copied key
 * in the same pass (position += shift, shift 0), the value is copied as is.
 * Dropped tokens leave the logical sequence, so later logical indices move
 * down as after a splice.  The old pages lose the sequence's reference (pages
 * shared with other sequences stay with them).  Needs ceil(visible /
 * page_size) free pages in each pool (AKV_ERR_NO_PAGES, state unchanged). */
AKV_API akv_status akv_compact(akv_ctx* ctx, int32_t seq, void* stream);

/* Attention mass (the attn_mass kernel, a second light pass after
 * akv_attend): for every segment and every logical token t < kv_end of its
 * sequence, the softmax probability the token's entry receives summed over
 * the segment's q_len query rows and all query heads,
 *   mass[off_s + t] = sum_rows sum_heads exp(scale * q . k_t - lse_row),
 * and 0 for tokens the segment does not see.  This is the cumulative attention
 * weight a serving engine watches to pick droppable blocks ([AKV-blog]
 * "Dilemma 1: Client-Side vs Server-Side Drop Policy"); the policy on top is
 * the caller's.  q, scale and the segments must be those of the attention
 * pass, lse its natural-log output [n_q_rows][n_q_heads].  mass: float
 * [sum over segments of kv_end], segment s at off_s = kv_end of segments
 * before it; host or device memory.  Values are sums of bf16-rounded
 * probabilities accumulated in float32 (atomics: the summation order varies
 * between runs).  GQA layout only. */
AKV_API akv_status akv_attention_mass(akv_ctx* ctx, int32_t layer, const akv_segment* segs, int32_t n_segs,
                              const void* q, int64_t n_q_rows, const float* lse, float scale, float* mass,
                              void* stream);

/* Segment-batch attention with the rotation fused in ([AKV-blog] section 4,
 * "Segment-Batch Attention Kernel Architecture": rotate keys in registers /
 * shared memory on the way to the tensor core, so transient position versions
 * cost no HBM writes).  Same arguments and results as akv_attend, but pending
 * shifts stay pending: no flush, no copy-on-write, the pools are only read.
 * Each key with a pending shift is rotated in shared memory by the same
 * float32 arithmetic and (cos, sin) table as akv_flush, so its bf16 bits equal
 * the materialised key's; runs then also break where the shift changes, so
 * tile composition (and float rounding order) can differ from akv_attend.
 * Under MLA only K_pe is rotated ([Leyline] "Method"); the latent is read as
 * stored.  Without pending shifts it is akv_attend without the flush. */
AKV_API akv_status akv_attend_fused(akv_ctx* ctx, int32_t layer, const akv_segment* segs, int32_t n_segs,
                            const void* q, int64_t n_q_rows, void* o, float* lse, float scale,
                            void* stream);

/* Float32 debug mode of the repos_rotate kernel: rotate rows of the K pool
 * (K_pe under MLA) by given shifts exactly as akv_flush would, but write the
 * unrounded float32 results to `out` instead of rounding them back into the
 * pool (the pool is only read).  Checks the rotation arithmetic against
 * float64 without the bf16 storage rounding ([Leyline] "Limitations": the
 * rotation runs in fp32; storage adds its own rounding).
 *   runs: host int32, 4 per run: K page, slot_lo, slot_hi, delta.
 *   out:  device float [n_layers][sum of (slot_hi - slot_lo)][n_kv_heads][d_rot],
 *         rows in run order. */
AKV_API akv_status akv_debug_rotate_f32(akv_ctx* ctx, const int32_t* runs, int32_t n_runs, float* out,
                                        void* stream);

/* The repos_rotate kernel for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers
 * such as a serving process that reserves nearly all of HBM for its KV pool
 * up front (no room for more cudaMalloc calls) or a latency-critical path
 * that must avoid cudaMalloc / cudaFree because they can synchronise the
 * whole device.  It needs no context and allocates nothing: the run list and
 * the (cos, sin) table are copied into a fixed 256 KiB array in the library's
 * own device memory (every GPU that loads the library holds it until exit).
 *   k_pool: device bf16 [n_layers][n_pages][n_kv_heads][page_size][d_rot],
 *           read and written (the same layout as akv_pools.k_pool).
 *   runs:   host int32, 5 per run: src page, dst page, slot_lo, slot_hi,
 *           delta -- rows [slot_lo, slot_hi) of page src, every layer and
 *           head, rotated by delta and stored to the same rows of page dst
 *           (the run format of akv_last_flush_runs).
 *   d_rot: 16, 32, 64, 128 or 256; page_size: 16, 32, 64 or 128.
 * Runs of one call execute concurrently, so they must write disjoint rows:
 * two runs writing the same (page, row), or a copy (src != dst) reading rows
 * that another copy writes, give AKV_ERR_ARG.  A copy may read rows that an
 * in-place run (src == dst) rotates, as a flush of two sequences sharing a
 * page lists them: those copies are made in a first launch, before the
 * in-place rotations.  Run lists from akv_last_flush_runs always qualify.
 * Returns AKV_ERR_RANGE when a run is outside the pool or when the runs plus
 * the table (16 B per run, rounded up to 256 B, plus 4 * d_rot B per distinct
 * delta) exceed 256 KiB, checked before any device work; AKV_ERR_ARG for a bad
 * shape, for overlapping runs, and while `stream` is being captured into a
 * graph (the run list and the table are copied from temporary host memory
 * during the call).  Every call overwrites the part of the array it uses, so
 * nothing needs clearing between calls, but calls that overlap on the GPU
 * (e.g. unordered streams) race on the array; calls on one stream are
 * ordered.  The first call on a device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress) and caches it: make that
 * first call before any stream capture. */
AKV_API akv_status akv_repos_rotate_noalloc(void* k_pool, int32_t n_layers, int32_t n_kv_heads,
                                            int32_t page_size, int32_t n_pages, int32_t d_rot,
                                            int32_t rope_layout, double rope_base, const int32_t* runs,
                                            int32_t n_runs, void* stream);

/* --- inspection (host memory only; used by the bookkeeping tests) -------- */

/* Per-token state of a sequence into caller arrays of akv_seq_len entries
 * (any may be NULL): K page, V page, slot, stored position, pending shift,
 * visibility (1 visible, 0 dropped). */
AKV_API akv_status akv_export_state(akv_ctx* ctx, int32_t seq, int32_t* k_page, int32_t* v_page,
                            int32_t* slot, int32_t* pos, int32_t* delta, uint8_t* visible);

/* Reference counts of every page: k_rc, v_rc int32[n_pages] (either may be NULL). */
AKV_API akv_status akv_refcounts(akv_ctx* ctx, int32_t* k_rc, int32_t* v_rc);

/* Run list of the last flush that had work: 5 int32 per run
 * (src K page, dst K page, slot_lo, slot_hi, delta), at most `cap` runs
 * written; *n_runs receives the full count. */
AKV_API akv_status akv_last_flush_runs(akv_ctx* ctx, int32_t* out, int64_t cap, int64_t* n_runs);

/* Run list a segment would attend over (after its sequence is flushed):
 * 4 int32 per run (K page, V page, slot_lo, slot_hi); *kv_len the entry count.
 * Fails with AKV_ERR_ARG if a visible token of the segment has a pending shift. */
AKV_API akv_status akv_segment_runs(akv_ctx* ctx, const akv_segment* seg, int32_t* out, int64_t cap,
                            int64_t* n_runs, int64_t* kv_len);

/* Schedule of the last akv_attend of a metadata-only context (pools NULL:
 * the planners run, nothing is launched), for checking the schedule on hosts
 * without a GPU.  units: 9 int32 per work entry (segment, kv head or MLA
 * flags, first query tile, KV tiles of query tile A, of tile B or the MLA
 * output half, first and end KV tile of the entry, partial slot or -1, merge
 * item or -1), at most `cap` entries; cta_units: the persistent schedule's
 * boundaries (CTA -- MLA: CTA pair -- b runs entries or pair units
 * [cta_units[b], cta_units[b + 1])), at most cta_cap values; *n_cta = 0 when
 * the launch has one unit per CTA.  n_sm > 0 sets the SM count later plans
 * assume (0 keeps it).  AKV_ERR_ARG on a context with pools. */
AKV_API akv_status akv_last_attention_plan(akv_ctx* ctx, int32_t* units, int64_t cap, int64_t* n_units,
                                           int32_t* cta_units, int64_t cta_cap, int64_t* n_cta, int32_t n_sm);

/* --- device status and measurement --------------------------------------- */

/* Synchronise `stream` and read the device error word of the context's
 * kernels: *code = 0, AKV_ERR_DEVICE_TIMEOUT or AKV_ERR_DEVICE.  The word
 * is cleared after reading.  Returns the same status as *code. */
AKV_API akv_status akv_check_device_error(akv_ctx* ctx, void* stream, int32_t* code);

/* Where results are copied to host memory.  By default (stream NULL) a host
 * output of akv_attend / akv_attend_fused (o, lse) or akv_attention_mass
 * (mass) is copied on the call's own stream, so synchronising that stream
 * covers it.  With an output stream set, the copy is enqueued on `stream`
 * (a cudaStream_t) after everything enqueued on the call's stream so far, so
 * it overlaps the kernels of later calls; the caller then synchronises the
 * output stream (or an event recorded on it) before reading a host output.
 * The device staging of a result is reused two calls later, after its copy
 * has completed.  While the call's stream is being captured into a graph,
 * results are copied on it.  The stream must stay valid while set. */
AKV_API akv_status akv_set_output_stream(akv_ctx* ctx, void* stream);

/* Split-KV control for akv_attend and akv_attention_mass.  0 (default): the
 * engine cuts long work items into chunks of KV tiles when that fills the
 * GPU's waves of SMs better; in akv_attend the CTA that finishes an item's
 * last chunk merges the chunks' partial softmax results (running maximum and
 * sum rescaled to a common maximum), akv_attention_mass needs no merge (its
 * lse is final; chunks add into the same outputs).  1..8: use exactly that
 * many chunks per item (1 = never split). */
AKV_API akv_status akv_set_attention_split(akv_ctx* ctx, int32_t split);

/* Test hook for the bounded waits of the attention kernels (no counterpart
 * on the pages: every device-side wait gives up after a time limit, records
 * AKV_ERR_DEVICE_TIMEOUT in the device error word, drains its copies and
 * tensor-core work, frees its TMEM and exits, so a stuck launch reports an
 * error instead of hanging the GPU).  wait_ns: the limit of every wait in
 * later akv_attend / akv_attend_fused launches (0 restores the default,
 * 4 s).  load_cap >= 0: each copy-issuing thread of a CTA issues at most
 * that many K/V copies (GQA: tiles; MLA: ring rounds) and then stops, so the
 * waits for the missing ones run out; -1 (default) removes the cap.  A test sets a
 * short limit and a cap, checks akv_check_device_error for
 * AKV_ERR_DEVICE_TIMEOUT and that the context still works after restoring
 * (0, -1).  AKV_ERR_ARG for load_cap < -1. */
AKV_API akv_status akv_debug_wait_limit(akv_ctx* ctx, uint64_t wait_ns, int32_t load_cap);

/* Test hook of the checked build (libakv_checked.so, compiled with
 * -DAKV_CHECKED; no counterpart on the pages).  That build adds device-side
 * descriptor checks to every kernel: a descriptor naming a page outside the
 * pool, a row range outside a page, a segment or run outside its table or
 * query rows outside Q makes the kernel record AKV_ERR_DEVICE in the device
 * error word and skip the work it names (attention: the CTA returns before
 * touching memory), never a trap.  Host validation normally keeps such
 * descriptors away from the device, so this call corrupts one after it:
 * what = 1, the next flush's first run gets a row range ending past its page;
 * what = 2, the next attention launch's first run gets a K page outside the
 * pool; 0 cancels.  The plain library returns AKV_ERR_ARG. */
AKV_API akv_status akv_debug_corrupt(akv_ctx* ctx, int32_t what);

/* Enable (1) or disable (0) per-launch CUDA-event timing of the context's
 * kernels; enabling clears the statistics. */
AKV_API akv_status akv_profile_enable(akv_ctx* ctx, int32_t on);

/* Synchronise the timed launches and return the statistics gathered since
 * profiling was enabled. */
AKV_API akv_status akv_profile_read(akv_ctx* ctx, akv_kernel_stats* out);

#ifdef __cplusplus
}
#endif

#endif /* AKV_H */
