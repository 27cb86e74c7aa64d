// Host engine of the agentic KV cache: page pools, sequences, the
// append / drop / repos / splice contract, composition of shifts, flush run
// lists and the (cos, sin) table, segment run lists and the attention work
// list, staging of host buffers, and the C ABI of include/akv.h.
//
// Sources, cited by page title and section:
//   [AKV-blog]  "AKV: Cache Engineering for Autonomous Agents and
//               State-Preserving Prefix Invalidation Bypass"
//   [AKV-notes] "Cache Engineering for Agents" (reading notes on Fu et al.)
//   [Leyline]   "Leyline: KV Cache Directives for Agentic Inference"
//
// Bookkeeping rules (the pages leave these open; the float64 oracle states
// the same rules independently and the tests compare the two bit for bit):
//   * two pools of equal size: "K" holds the rotated key part, "V" the rest;
//     each page has a reference count = live sequences with a token in it;
//     a fresh page is the lowest free id of its pool.
//   * append fills the last token's page at slot + 1 when its K and V pages
//     both have one reference; otherwise it opens a K page and a V page.
//   * drop only hides ([AKV-blog] section 2 "The Drop Primitive": no
//     deallocation).  repos only adds to a token's pending shift.
//   * flush rotates visible tokens with a pending shift once by the composed
//     shift ([Leyline] "Method": R(a)R(b) = R(a+b)).  A shared K page is
//     copied first with every visible token of the sequence in it ([AKV-notes]
//     section 3 "Cache Management": rotate copies that form a new branch).
//   * splice removes [s, e), writes the stub to fresh pages, inserts it at s
//     and shifts later tokens by n_stub - (e - s) ([Leyline] "Method").

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/akv.h"
#include "akv_internal.h"

namespace {

constexpr int64_t kI32Min = INT32_MIN;
constexpr int64_t kI32Max = INT32_MAX;

struct Fail {
  akv_status st;
  std::string msg;
};

[[noreturn]] void fail(akv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  throw Fail{st, buf};
}

void cuda_check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) fail(AKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct Tok {  // 20 bytes: every pass over a sequence streams these records
  int32_t kp, vp, pos, delta;
  int16_t slot;  // < page_size <= 128
  uint8_t vis;
  int64_t eff() const { return int64_t(pos) + delta; }
};

// Reference counts of one pool with lowest-free-id-first allocation.
class Pool {
 public:
  // Free pages are the set bits of a bitmap; the lowest set bit at or after
  // hint_ (no free page lies below it) is the lowest free id, so allocation
  // follows the lowest-free-id-first rule and a free is O(1).
  void init(int32_t n) {
    rc_.assign(n, 0);
    free_.assign((size_t(n) + 63) / 64, ~uint64_t(0));
    if (n % 64) free_.back() = (uint64_t(1) << (n % 64)) - 1;
    hint_ = 0;
    n_free_ = n;
  }
  int32_t alloc() {  // callers check n_free() first
    while (free_[hint_] == 0) ++hint_;
    const int b = __builtin_ctzll(free_[hint_]);
    free_[hint_] &= free_[hint_] - 1;
    const int32_t p = int32_t(hint_ * 64 + size_t(b));
    rc_[p] = 1;
    --n_free_;
    return p;
  }
  void inc(int32_t p) { ++rc_[p]; }
  void dec(int32_t p) {
    if (--rc_[p] == 0) {
      free_[size_t(p) / 64] |= uint64_t(1) << (p % 64);
      hint_ = std::min(hint_, size_t(p) / 64);
      ++n_free_;
    }
  }
  int32_t rc(int32_t p) const { return rc_[p]; }
  int32_t n_free() const { return n_free_; }
  const std::vector<int32_t>& counts() const { return rc_; }

 private:
  std::vector<int32_t> rc_;
  std::vector<uint64_t> free_;
  size_t hint_ = 0;
  int32_t n_free_ = 0;
};

// Epoch-stamped marks over page ids: distinct-page sets in O(tokens).
class Marks {
 public:
  void init(int32_t n) { m_.assign(n, 0); }
  void next() {
    if (++epoch_ == 0) {
      std::fill(m_.begin(), m_.end(), 0);
      epoch_ = 1;
    }
  }
  bool test_set(int32_t p) {
    if (m_[p] == epoch_) return false;
    m_[p] = epoch_;
    return true;
  }
  bool test(int32_t p) const { return m_[p] == epoch_; }

 private:
  std::vector<uint32_t> m_;
  uint32_t epoch_ = 0;
};

// A pinned-host + device buffer pair reused across calls.  acquire() waits
// for the event recorded by the previous user, so a buffer is never
// overwritten while a copy or kernel that reads it is still queued.
// Staging for host inputs / outputs (and device scratch): two buffers used in
// turn, so the host can stage the next call while the GPU still reads the
// previous one; acquire waits only for the use before last of its buffer.
struct Staging {
  void* host = nullptr;  // the current buffer (valid after acquire)
  void* dev = nullptr;
  bool want_host = true;
  struct Buf {
    void* host = nullptr;
    void* dev = nullptr;
    size_t cap = 0;
    cudaEvent_t ev = nullptr;
    cudaEvent_t copied = nullptr;
    bool pending = false;
  } buf[2];
  int cur = 1;

  void acquire(size_t bytes) {
    cur ^= 1;
    Buf& b = buf[cur];
    if (!b.ev) cuda_check(cudaEventCreateWithFlags(&b.ev, cudaEventDisableTiming), "cudaEventCreate");
    if (b.pending) {
      cuda_check(cudaEventSynchronize(b.ev), "cudaEventSynchronize");
      b.pending = false;
    }
    if (bytes > b.cap || (want_host && !b.host)) {
      const size_t want = std::max<size_t>(bytes + bytes / 2, 4096);
      if (b.host) cudaFreeHost(b.host);
      if (b.dev) cudaFree(b.dev);
      b.host = b.dev = nullptr;
      b.cap = 0;
      if (want_host) cuda_check(cudaMallocHost(&b.host, want), "cudaMallocHost");
      cuda_check(cudaMalloc(&b.dev, want), "cudaMalloc");
      b.cap = want;
    }
    host = b.host;
    dev = b.dev;
  }
  void release(cudaStream_t st) {
    cuda_check(cudaEventRecord(buf[cur].ev, st), "cudaEventRecord");
    buf[cur].pending = true;
  }
  // Copy `bytes` of host `src` into the current device buffer.  With a copy
  // stream `cp` the copy runs there, ahead of `st`'s earlier work, and `st`
  // waits for it; acquire() has already waited until `st` no longer reads
  // this buffer's previous contents.  Without one (or while `st` is being
  // captured into a graph) the copy is ordered on `st` itself.
  void copy_in(const void* src, size_t bytes, cudaStream_t st, cudaStream_t cp, const char* what) {
    if (cp) {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      cuda_check(cudaStreamIsCapturing(st, &cs), "cudaStreamIsCapturing");
      if (cs != cudaStreamCaptureStatusNone) cp = nullptr;
    }
    if (!cp) {
      cuda_check(cudaMemcpyAsync(dev, src, bytes, cudaMemcpyHostToDevice, st), what);
      return;
    }
    Buf& b = buf[cur];
    if (!b.copied) cuda_check(cudaEventCreateWithFlags(&b.copied, cudaEventDisableTiming), "cudaEventCreate");
    cuda_check(cudaMemcpyAsync(dev, src, bytes, cudaMemcpyHostToDevice, cp), what);
    cuda_check(cudaEventRecord(b.copied, cp), "cudaEventRecord");
    cuda_check(cudaStreamWaitEvent(st, b.copied, 0), "cudaStreamWaitEvent");
  }
  void destroy() {
    for (Buf& b : buf) {
      if (b.ev) {
        cudaEventSynchronize(b.ev);
        cudaEventDestroy(b.ev);
      }
      if (b.copied) {
        cudaEventSynchronize(b.copied);
        cudaEventDestroy(b.copied);
      }
      if (b.host) cudaFreeHost(b.host);
      if (b.dev) cudaFree(b.dev);
      b = Buf{};
    }
    host = dev = nullptr;
  }
};

// Uploads several host arrays to one device block through a ring of
// staging buffers; returns device pointers (16-byte aligned pieces).
class Uploader {
 public:
  static constexpr int kRing = 4;
  struct Piece {
    const void* src;
    size_t bytes;
    void** dst_dev;
  };
  void upload(std::initializer_list<Piece> pieces, cudaStream_t st) {
    // the tables are the library's own and final here, so they may go ahead on the copy stream
    size_t total = 0;
    for (auto& p : pieces) total += (p.bytes + 15) & ~size_t(15);
    Staging& s = ring_[next_];
    next_ = (next_ + 1) % kRing;
    s.acquire(std::max<size_t>(total, 16));
    size_t off = 0;
    for (auto& p : pieces) {
      if (p.bytes) std::memcpy(static_cast<char*>(s.host) + off, p.src, p.bytes);
      *p.dst_dev = static_cast<char*>(s.dev) + off;
      off += (p.bytes + 15) & ~size_t(15);
    }
    s.copy_in(s.host, std::max<size_t>(off, 16), st, copy_stream, "descriptor upload");
    last_ = &s;
  }
  cudaStream_t copy_stream = nullptr;
  // Record the event after the kernel that reads the last upload.
  void done(cudaStream_t st) {
    if (last_) last_->release(st);
    last_ = nullptr;
  }
  void destroy() {
    for (auto& s : ring_) s.destroy();
  }

 private:
  Staging ring_[kRing];
  int next_ = 0;
  Staging* last_ = nullptr;
};

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn) return fn;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  cuda_check(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q),
             "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
  if (q != cudaDriverEntryPointSuccess || !ptr) fail(AKV_ERR_CUDA, "cuTensorMapEncodeTiled not available");
  fn = reinterpret_cast<EncodeTiledFn>(ptr);
  return fn;
}

// Row-major bf16 tensor map; dims/strides innermost first, strides in bytes
// for dims 1.., box in elements, 128-byte swizzle, zero fill out of bounds.
void encode_map(CUtensorMap* m, void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                const uint32_t* box) {
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
  CUresult r = get_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, d, s, b, e,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) fail(AKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
}

enum KernelId { kKvWrite = 0, kRepos = 1, kAttn = 2, kCompact = 3, kMass = 4 };

// End of a launch whose CTAs (or CTA pairs) cost `cost` each, run longest
// first, each on the slot that frees first (the hardware hands out CTAs in
// launch order as slots free up).
double lpt_makespan(std::vector<double> cost, int64_t slots) {
  std::sort(cost.begin(), cost.end(), std::greater<double>());
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int64_t i = 0; i < std::max<int64_t>(1, slots); ++i) free_at.push(0.0);
  double end = 0.0;
  for (double c : cost) {
    const double t = free_at.top() + c;
    free_at.pop();
    free_at.push(t);
    end = std::max(end, t);
  }
  return end;
}

// The same estimate in linear time for integer costs, given as a histogram
// (count[c] = CTAs of cost c): the CTAs taken longest first in waves of
// `slots`, each wave as long as its longest CTA (within a wave of LPT on
// near-equal costs; an upper bound when costs are skewed).
int64_t wave_makespan(const std::vector<int64_t>& count, int64_t slots) {
  slots = std::max<int64_t>(1, slots);
  int64_t end = 0, in_wave = 0;
  for (size_t c = count.size(); c-- > 0;) {
    int64_t m = count[c];
    while (m > 0) {
      if (in_wave == 0) end += int64_t(c);  // a new wave starts with its longest CTA
      const int64_t take = std::min(m, slots - in_wave);
      m -= take;
      in_wave = (in_wave + take) % slots;
    }
  }
  return end;
}

}  // namespace

struct akv_ctx {
  akv_config cfg{};
  bool meta = false;
  void* kpool = nullptr;
  void* vpool = nullptr;
  Pool K, V;
  Marks mk, mv;
  std::vector<std::vector<Tok>> seqs;
  std::vector<uint8_t> live;
  struct Pend {  // a recorded reposition not yet folded into the tokens
    int64_t s, e;
    int32_t d;
  };
  std::vector<std::vector<Pend>> pend;  // per sequence
  // Per sequence: an upper bound on |position| and |pending shift| of its
  // tokens; while bound + |delta| fits in int32 no per-token overflow check is needed.
  std::vector<int64_t> bound;
  std::vector<int32_t> page_dst;  // flush scratch: destination of each moving K page
  std::vector<int32_t> sim_rc;    // flush scratch: simulated reference-count changes
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_ids;

  // extended radix tree: node 0 is the root
  struct TreeNode {
    akv_item item{};       // the item on the edge into this node
    int32_t parent = -1;
    int32_t owner = -1;    // tree-held sequence with this prefix
    int64_t order = -1;    // insertion number of the owner (ties: earliest)
    int64_t n_tok = 0;     // tokens on the path root .. this node
    std::vector<int32_t> kids;
  };
  std::vector<TreeNode> tree = std::vector<TreeNode>(1);
  std::vector<int32_t> tree_seqs;
  int64_t tree_inserts = 0;
  std::string err;
  std::vector<int32_t> last_runs;  // 5 per run

  // device side
  int device = -1;
  akv::DevErr* dev_err = nullptr;
  Uploader up;
  Staging st_k, st_v, st_q, st_o, st_lse;
  cudaStream_t out_st = nullptr;     // akv_set_output_stream: where results are copied to host memory
  cudaEvent_t out_ready = nullptr;
  cudaStream_t copy_st = nullptr;  // host-to-device copies of inputs and descriptor tables
  Staging partial;         // split-KV partial results (device only)
  std::vector<akv::AttnWork> last_work;  // metadata-only contexts: the last attention plan
  std::vector<int32_t> last_cta_units;
  int n_sm = 148;          // SMs of the device, for split decisions
  int mla_slots = 148;     // MLA kernel CTAs resident at once (CTA pairs x 2)
  int split_override = 0;  // 0: choose the split factor; n >= 1: use n
  int32_t corrupt_next = 0;           // checked-build test hook (akv_debug_corrupt)
  uint64_t wait_ns = 4000000000ull;  // limit of the attention kernels' bounded waits
  int32_t load_cap = -1;              // test hook: cap on a CTA's K/V copies (attention: GQA tiles, MLA rounds)
  CUtensorMap k_map{}, v_map{}, k_tile_map{}, v_tile_map{};
  bool maps_ok = false;

  // profiling
  bool prof = false;
  struct Timed {
    int kernel;
    int launches;
    cudaEvent_t a, b;
    double bytes, flops;
  };
  std::vector<Timed> timed;
  std::vector<cudaEvent_t> ev_pool;
  akv_kernel_stats stats{};

  int64_t row_elems_k() const { return int64_t(cfg.n_kv_heads) * cfg.page_size * cfg.d_rot; }

  // Token records of a live sequence as they are; repositions recorded since
  // the last settle are still in pend[id].
  std::vector<Tok>& seq_raw(int32_t id) {
    if (id < 0 || id >= int32_t(seqs.size()) || !live[id]) fail(AKV_ERR_ARG, "sequence %d is not live", id);
    return seqs[id];
  }

  // Token records with every recorded reposition folded into the per-token
  // pending shift (what every reader of shifts, positions or order sees).
  std::vector<Tok>& seq(int32_t id) {
    auto& toks = seq_raw(id);
    settle(id);
    return toks;
  }

  // repos records a shift for a span in O(1); the spans are folded into the
  // tokens here, all at once, with a difference array (O(tokens + spans)).
  void settle(int32_t id) {
    auto& p = pend[id];
    if (p.empty()) return;
    auto& toks = seqs[id];
    if (p.size() == 1) {
      for (int64_t i = p[0].s; i < p[0].e; ++i) toks[i].delta += p[0].d;
    } else {
      // Sweep over the spans' sorted end points: between two consecutive
      // points every token gets the same sum of shifts; only spans with a
      // nonzero sum are touched.
      std::vector<std::pair<int64_t, int64_t>> ev;
      ev.reserve(2 * p.size());
      for (const Pend& r : p) {
        ev.emplace_back(r.s, r.d);
        ev.emplace_back(r.e, -int64_t(r.d));
      }
      std::sort(ev.begin(), ev.end());
      int64_t acc = 0;
      for (size_t k = 0; k + 1 < ev.size(); ++k) {
        acc += ev[k].second;
        if (acc == 0) continue;
        const int32_t a = int32_t(acc);
        for (int64_t i = ev[k].first; i < ev[k + 1].first; ++i) toks[size_t(i)].delta += a;
      }
    }
    p.clear();
  }

  int32_t new_id() {
    if (!free_ids.empty()) {
      int32_t id = free_ids.top();
      free_ids.pop();
      live[id] = 1;
      bound[id] = 0;
      return id;
    }
    seqs.emplace_back();
    pend.emplace_back();
    live.push_back(1);
    bound.push_back(0);
    return int32_t(seqs.size() - 1);
  }

  // distinct K and V pages of toks[a, b)
  void pages_of(const std::vector<Tok>& toks, size_t a, size_t b, std::vector<int32_t>& kps,
                std::vector<int32_t>& vps) {
    mk.next();
    mv.next();
    kps.clear();
    vps.clear();
    for (size_t i = a; i < b; ++i) {
      if (mk.test_set(toks[i].kp)) kps.push_back(toks[i].kp);
      if (mv.test_set(toks[i].vp)) vps.push_back(toks[i].vp);
    }
  }

  // ------------------------------------------------------------ profiling
  cudaEvent_t take_event() {
    if (!ev_pool.empty()) {
      cudaEvent_t e = ev_pool.back();
      ev_pool.pop_back();
      return e;
    }
    cudaEvent_t e;
    cuda_check(cudaEventCreate(&e), "cudaEventCreate");
    return e;
  }
  void begin_timed(int kernel, double bytes, double flops, cudaStream_t st, Timed& t, int launches = 1) {
    t.kernel = kernel;
    t.launches = launches;
    t.bytes = bytes;
    t.flops = flops;
    t.a = t.b = nullptr;
    if (!prof) return;
    t.a = take_event();
    t.b = take_event();
    cuda_check(cudaEventRecord(t.a, st), "cudaEventRecord");
  }
  void end_timed(Timed& t, cudaStream_t st) {
    if (!prof) return;
    cuda_check(cudaEventRecord(t.b, st), "cudaEventRecord");
    timed.push_back(t);
  }
  void collect() {
    for (auto& t : timed) {
      cuda_check(cudaEventSynchronize(t.b), "cudaEventSynchronize");
      float ms = 0.f;
      cuda_check(cudaEventElapsedTime(&ms, t.a, t.b), "cudaEventElapsedTime");
      stats.launches[t.kernel] += t.launches;
      stats.ms[t.kernel] += ms;
      stats.bytes[t.kernel] += t.bytes;
      stats.flops[t.kernel] += t.flops;
      ev_pool.push_back(t.a);
      ev_pool.push_back(t.b);
    }
    timed.clear();
  }

  // ------------------------------------------------------------- device IO
  // Returns a device pointer holding `bytes` of `src` (device: as is; host: staged).
  // Host inputs are read on the context's copy stream when the call is made
  // (so they overlap the kernels of earlier calls still running on `st`).
  const void* device_input(const void* src, size_t bytes, Staging& s, cudaStream_t st) {
    if (is_device_ptr(src)) return src;
    s.want_host = false;
    s.acquire(bytes);
    s.copy_in(src, bytes, st, copy_st, "host input copy");
    return s.dev;
  }

  void write_rows(const std::vector<int32_t>& krow, const std::vector<int32_t>& vrow, const void* k,
                  const void* v, cudaStream_t st) {
    const int64_t n = int64_t(krow.size());
    if (meta || n == 0) return;
    if (!k || !v) fail(AKV_ERR_ARG, "null K/V data pointer");
    const size_t kbytes = size_t(cfg.n_layers) * n * cfg.n_kv_heads * cfg.d_rot * 2;
    const size_t vbytes = size_t(cfg.n_layers) * n * cfg.n_kv_heads * cfg.d_v * 2;
    const void* kd = device_input(k, kbytes, st_k, st);
    const void* vd = device_input(v, vbytes, st_v, st);
    void* dk = nullptr;
    void* dv = nullptr;
    up.upload({{krow.data(), krow.size() * 4, &dk}, {vrow.data(), vrow.size() * 4, &dv}}, st);
    Timed t;
    begin_timed(kKvWrite, double(kbytes + vbytes) * 2.0, 0.0, st, t, 1);
    cuda_check(akv::launch_kv_write(kd, kpool, static_cast<int32_t*>(dk), cfg.d_rot, vd, vpool,
                                    static_cast<int32_t*>(dv), cfg.d_v, n, cfg.n_layers, cfg.n_kv_heads,
                                    cfg.page_size, cfg.n_pages, n_sm, dev_err, st),
               "kv_write launch");
    end_timed(t, st);
    up.done(st);
    if (st_k.dev && !is_device_ptr(k)) st_k.release(st);
    if (st_v.dev && !is_device_ptr(v)) st_v.release(st);
  }

  // ---------------------------------------------------------- operations
  void append(int32_t sid, int64_t n, const void* k, const void* v, const int32_t* pos, cudaStream_t st) {
    auto& toks = seq(sid);
    if (n < 0) fail(AKV_ERR_ARG, "negative token count");
    if (n > kI32Max) fail(AKV_ERR_RANGE, "too many tokens");
    std::vector<int32_t> p(n);
    if (pos) {
      std::memcpy(p.data(), pos, size_t(n) * 4);
    } else {
      int64_t start = toks.empty() ? 0 : toks.back().eff() + 1;
      if (n && start + n - 1 > kI32Max) fail(AKV_ERR_OVERFLOW, "position %lld leaves int32", (long long)(start + n - 1));
      for (int64_t i = 0; i < n; ++i) p[i] = int32_t(start + i);
    }
    int64_t room = 0;
    int32_t kp = -1, vp = -1, slot = -1;
    if (!toks.empty()) {
      const Tok& last = toks.back();
      if (K.rc(last.kp) == 1 && V.rc(last.vp) == 1) {
        room = cfg.page_size - 1 - last.slot;
        kp = last.kp;
        vp = last.vp;
        slot = last.slot;
      }
    }
    int64_t need = n <= room ? 0 : (n - room + cfg.page_size - 1) / cfg.page_size;
    if (need > K.n_free() || need > V.n_free()) fail(AKV_ERR_NO_PAGES, "append needs %lld pages", (long long)need);
    if (int64_t(toks.size()) + n > kI32Max) fail(AKV_ERR_RANGE, "sequence too long");
    std::vector<int32_t> krow(n), vrow(n);
    if (toks.capacity() < toks.size() + size_t(n))  // geometric growth: repeated appends stay amortised O(n)
      toks.reserve(std::max(toks.size() + size_t(n), toks.capacity() + toks.capacity() / 2));
    for (int64_t i = 0; i < n; ++i) {
      if (room > 0) {
        ++slot;
        --room;
      } else {
        kp = K.alloc();
        vp = V.alloc();
        slot = 0;
        room = cfg.page_size - 1;
      }
      toks.push_back(Tok{kp, vp, p[i], 0, int16_t(slot), 1});
      bound[sid] = std::max<int64_t>(bound[sid], std::abs(int64_t(p[i])));
      krow[i] = kp * cfg.page_size + slot;
      vrow[i] = vp * cfg.page_size + slot;
    }
    write_rows(krow, vrow, k, v, st);
  }

  void check_span(const std::vector<Tok>& toks, int64_t s, int64_t e, const char* what) {
    if (s < 0 || s > e || e > int64_t(toks.size())) fail(AKV_ERR_RANGE, "%s span [%lld, %lld) outside the sequence", what, (long long)s, (long long)e);
  }

  void drop(int32_t sid, int64_t s, int64_t e) {
    auto& toks = seq_raw(sid);  // visibility only
    check_span(toks, s, e, "drop");
    for (int64_t i = s; i < e; ++i) toks[i].vis = 0;
  }

  void check_shift(const std::vector<Tok>& toks, int64_t a, int64_t b, int64_t delta, int64_t seq_bound) {
    if (seq_bound + std::abs(delta) <= kI32Max) return;  // cannot leave int32
    for (int64_t i = a; i < b; ++i) {
      const Tok& t = toks[i];
      if (int64_t(t.delta) + delta < kI32Min || int64_t(t.delta) + delta > kI32Max)
        fail(AKV_ERR_OVERFLOW, "composed shift of token %lld leaves int32", (long long)i);
      if (t.eff() + delta < kI32Min || t.eff() + delta > kI32Max)
        fail(AKV_ERR_OVERFLOW, "position of token %lld leaves int32", (long long)i);
    }
  }

  // Exact bound of a sequence (used when the running bound grew too loose).
  static int64_t exact_bound(const std::vector<Tok>& toks) {
    int64_t b = 0;
    for (const Tok& t : toks) b = std::max({b, std::abs(t.eff()), std::abs(int64_t(t.delta))});
    return b;
  }

  void grow_bound(int32_t sid, int64_t by) {
    bound[sid] += by;
    if (bound[sid] > kI32Max) bound[sid] = exact_bound(seq(sid));
  }

  void repos(int32_t sid, int64_t s, int64_t e, int32_t delta) {
    auto& toks = seq_raw(sid);
    check_span(toks, s, e, "repos");
    if (bound[sid] + std::abs(int64_t(delta)) <= kI32Max) {
      // no token can leave int32: record the span, fold it in when read
      if (s < e && delta != 0) pend[sid].push_back(Pend{s, e, delta});
    } else {
      settle(sid);
      check_shift(toks, s, e, delta, bound[sid]);
      for (int64_t i = s; i < e; ++i) toks[i].delta += delta;
    }
    grow_bound(sid, std::abs(int64_t(delta)));
  }

  // A list of drop / repos directives for one sequence, in order, all or
  // nothing: every span is checked first (drops and repositions do not change
  // the sequence's length); when the running bound shows no token can leave
  // int32 every reposition is an O(1) record and nothing else can fail;
  // otherwise the sequence's state is saved and restored if a later entry
  // fails its overflow check.
  void edit(int32_t sid, const akv_edit_op* ops, int32_t n) {
    if (n < 0 || (n > 0 && !ops)) fail(AKV_ERR_ARG, "bad edit list");
    auto& toks = seq_raw(sid);
    int64_t shift_sum = 0;
    for (int32_t i = 0; i < n; ++i) {
      const akv_edit_op& o = ops[i];
      if (o.kind != AKV_EDIT_DROP && o.kind != AKV_EDIT_REPOS) fail(AKV_ERR_ARG, "edit %d: unknown kind %d", i, o.kind);
      check_span(toks, o.s, o.e, o.kind == AKV_EDIT_DROP ? "drop" : "repos");
      if (o.kind == AKV_EDIT_REPOS) shift_sum += std::abs(int64_t(o.delta));
    }
    const bool safe = bound[sid] + shift_sum <= kI32Max;
    std::vector<Tok> saved_toks;
    std::vector<Pend> saved_pend;
    const int64_t saved_bound = bound[sid];
    if (!safe) {
      saved_toks = toks;
      saved_pend = pend[sid];
    }
    try {
      for (int32_t i = 0; i < n; ++i) {
        if (ops[i].kind == AKV_EDIT_DROP)
          drop(sid, ops[i].s, ops[i].e);
        else
          repos(sid, ops[i].s, ops[i].e, ops[i].delta);
      }
    } catch (...) {
      if (!safe) {
        seqs[sid] = std::move(saved_toks);
        pend[sid] = std::move(saved_pend);
        bound[sid] = saved_bound;
      }
      throw;
    }
  }

  void splice(int32_t sid, int64_t s, int64_t e, int64_t n_stub, const void* k, const void* v, const int32_t* pos,
              cudaStream_t st) {
    auto& toks = seq(sid);
    check_span(toks, s, e, "splice");
    if (n_stub < 0 || n_stub > kI32Max) fail(AKV_ERR_RANGE, "bad stub length");
    const int64_t delta = n_stub - (e - s);
    if (delta < kI32Min || delta > kI32Max) fail(AKV_ERR_OVERFLOW, "splice shift leaves int32");
    std::vector<int32_t> p(n_stub);
    if (pos) {
      std::memcpy(p.data(), pos, size_t(n_stub) * 4);
    } else {
      int64_t p0 = s < int64_t(toks.size()) ? toks[s].eff() : (toks.empty() ? 0 : toks.back().eff() + 1);
      if (n_stub && p0 + n_stub - 1 > kI32Max) fail(AKV_ERR_OVERFLOW, "stub position leaves int32");
      for (int64_t i = 0; i < n_stub; ++i) p[i] = int32_t(p0 + i);
    }
    check_shift(toks, e, int64_t(toks.size()), delta, bound[sid]);
    if (int64_t(toks.size()) - (e - s) + n_stub > kI32Max) fail(AKV_ERR_RANGE, "sequence too long");
    // pages referenced only by the removed tokens are released
    std::vector<int32_t> kk, vv, kr, vr;
    pages_of(toks, 0, size_t(s), kk, vv);
    for (size_t i = size_t(e); i < toks.size(); ++i) {
      mk.test_set(toks[i].kp);
      mv.test_set(toks[i].vp);
    }
    for (int64_t i = s; i < e; ++i) {
      const Tok& t = toks[i];
      if (mk.test_set(t.kp)) kr.push_back(t.kp);
      if (mv.test_set(t.vp)) vr.push_back(t.vp);
    }
    const int64_t need = (n_stub + cfg.page_size - 1) / cfg.page_size;
    int64_t kf = K.n_free(), vf = V.n_free();
    for (int32_t q : kr) kf += K.rc(q) == 1;
    for (int32_t q : vr) vf += V.rc(q) == 1;
    if (need > kf || need > vf) fail(AKV_ERR_NO_PAGES, "splice needs %lld pages", (long long)need);
    for (int32_t q : kr) K.dec(q);
    for (int32_t q : vr) V.dec(q);
    std::vector<Tok> stub(n_stub);
    std::vector<int32_t> krow(n_stub), vrow(n_stub);
    int32_t kp = -1, vp = -1;
    for (int64_t i = 0; i < n_stub; ++i) {
      const int32_t slot = int32_t(i % cfg.page_size);
      if (slot == 0) {
        kp = K.alloc();
        vp = V.alloc();
      }
      stub[i] = Tok{kp, vp, p[i], 0, int16_t(slot), 1};
      krow[i] = kp * cfg.page_size + slot;
      vrow[i] = vp * cfg.page_size + slot;
    }
    for (size_t i = size_t(e); i < toks.size(); ++i) toks[i].delta += int32_t(delta);
    std::vector<Tok> out;
    out.reserve(toks.size() - (e - s) + n_stub);
    out.insert(out.end(), toks.begin(), toks.begin() + s);
    out.insert(out.end(), stub.begin(), stub.end());
    out.insert(out.end(), toks.begin() + e, toks.end());
    toks.swap(out);
    int64_t pmax = 0;
    for (int32_t q : p) pmax = std::max<int64_t>(pmax, std::abs(int64_t(q)));
    bound[sid] = std::max(bound[sid], pmax);
    grow_bound(sid, std::abs(delta));
    write_rows(krow, vrow, k, v, st);
  }

  void fork(int32_t src, int64_t n_prefix, int32_t* out) {
    auto& toks = seq(src);
    if (n_prefix < 0 || n_prefix > int64_t(toks.size())) fail(AKV_ERR_RANGE, "fork prefix outside the sequence");
    // headroom, so the branch's first appends do not reallocate (and copy) every token record
    std::vector<Tok> child;
    child.reserve(size_t(n_prefix) + size_t(n_prefix) / 4 + 4096);
    child.assign(toks.begin(), toks.begin() + n_prefix);
    std::vector<int32_t> kps, vps;
    pages_of(child, 0, child.size(), kps, vps);
    for (int32_t q : kps) K.inc(q);
    for (int32_t q : vps) V.inc(q);
    const int64_t parent_bound = bound[src];
    int32_t id = new_id();
    seqs[id] = std::move(child);
    bound[id] = parent_bound;
    *out = id;
  }

  void free_seq(int32_t sid) {
    auto& toks = seq_raw(sid);
    pend[sid].clear();
    std::vector<int32_t> kps, vps;
    pages_of(toks, 0, toks.size(), kps, vps);
    for (int32_t q : kps) K.dec(q);
    for (int32_t q : vps) V.dec(q);
    std::vector<Tok>().swap(toks);
    live[sid] = 0;
    free_ids.push(sid);
  }

  // ------------------------------------------------------------ compaction
  // [AKV-blog] "Dilemma 2: Memory Fragmentation in Paged Pools".  The share
  // of the slots of the sequence's K pages that hold none of its visible tokens.
  double fragmentation(int32_t sid) {
    auto& toks = seq_raw(sid);  // visibility only
    std::vector<int32_t> kps, vps;
    pages_of(toks, 0, toks.size(), kps, vps);
    if (kps.empty()) return 0.0;
    int64_t vis = 0;
    for (const Tok& t : toks) vis += t.vis;
    return 1.0 - double(vis) / (double(kps.size()) * cfg.page_size);
  }

  // Visible tokens, in logical order, copied densely into fresh pages (any
  // pending shift applied to the copied key); dropped tokens leave the
  // sequence; the old pages lose its reference.
  void compact(int32_t sid, cudaStream_t st) {
    auto& toks = seq(sid);
    int64_t n_vis = 0;
    for (const Tok& t : toks) n_vis += t.vis;
    const int64_t need = (n_vis + cfg.page_size - 1) / cfg.page_size;
    if (need > K.n_free() || need > V.n_free()) fail(AKV_ERR_NO_PAGES, "compaction needs %lld pages", (long long)need);
    std::vector<int32_t> kps, vps;
    pages_of(toks, 0, toks.size(), kps, vps);
    std::vector<Tok> out;
    out.reserve(size_t(n_vis));
    std::vector<akv::CopyRun> runs;
    std::vector<int32_t> shifts;
    std::unordered_map<int32_t, int32_t> didx;
    int32_t dk = -1, dv = -1;
    int64_t b = 0;
    for (const Tok& t : toks) {
      if (!t.vis) continue;
      const int32_t ds = int32_t(out.size() % size_t(cfg.page_size));
      if (ds == 0) {
        dk = K.alloc();
        dv = V.alloc();
      }
      int32_t di = -1;
      if (t.delta != 0) {
        auto it = didx.find(t.delta);
        if (it == didx.end()) {
          it = didx.emplace(t.delta, int32_t(shifts.size())).first;
          shifts.push_back(t.delta);
        }
        di = it->second;
      }
      akv::CopyRun* last = runs.empty() ? nullptr : &runs.back();
      if (last && last->src_k == t.kp && last->src_v == t.vp && last->src_lo + last->n == t.slot && last->didx == di &&
          last->dst_k == dk && last->dst_lo + last->n == ds) {
        ++last->n;
      } else {
        runs.push_back(akv::CopyRun{t.kp, t.vp, dk, dv, t.slot, ds, 1, di});
      }
      const int32_t pos = int32_t(t.eff());
      out.push_back(Tok{dk, dv, pos, 0, int16_t(ds), 1});
      b = std::max<int64_t>(b, std::abs(int64_t(pos)));
    }
    for (int32_t q : kps) K.dec(q);
    for (int32_t q : vps) V.dec(q);
    toks.swap(out);
    bound[sid] = b;
    if (meta || runs.empty()) return;
    const std::vector<float2> cs = angle_table(shifts);
    void* druns = nullptr;
    void* dcs = nullptr;
    up.upload({{runs.data(), runs.size() * sizeof(akv::CopyRun), &druns}, {cs.data(), cs.size() * sizeof(float2), &dcs}},
              st);
    Timed tm;
    const double bytes = 2.0 * double(n_vis) * cfg.n_layers * cfg.n_kv_heads * (cfg.d_rot + cfg.d_v) * 2.0;
    begin_timed(kCompact, bytes, 0.0, st, tm, 2);  // key launch + value launch
    cuda_check(akv::launch_compact_copy(kpool, vpool, static_cast<akv::CopyRun*>(druns), static_cast<float2*>(dcs),
                                        int(runs.size()), cfg.n_layers, cfg.n_kv_heads, cfg.d_rot, cfg.d_v,
                                        cfg.page_size, cfg.n_pages, cfg.rope_layout == AKV_ROPE_HALF, n_sm, dev_err,
                                        st),
               "compact_copy launch");
    end_timed(tm, st);
    up.done(st);
  }

  // ----------------------------------------------------------------- flush
  // Pages holding visible tokens with a pending shift, first-appearance order.
  void moving_pages(const std::vector<Tok>& toks, std::vector<int32_t>& order) {
    mk.next();
    order.clear();
    int32_t last = -1;  // consecutive tokens mostly share their page
    for (const Tok& t : toks)
      if (t.vis && t.delta != 0 && t.kp != last) {
        last = t.kp;
        if (mk.test_set(t.kp)) order.push_back(t.kp);
      }
  }

  void flush(const std::vector<int32_t>& ids, cudaStream_t st) {
    for (int32_t sid : ids) settle(sid);
    // Budget check on simulated reference counts, so a failure changes nothing.
    // Each sequence's moving pages are computed once and reused by flush_seq.
    std::vector<std::vector<int32_t>> orders(ids.size());
    int64_t need = 0;
    if (ids.size() == 1) {  // one sequence: its copies are its shared moving pages
      moving_pages(seqs[ids[0]], orders[0]);
      for (int32_t q : orders[0]) need += K.rc(q) > 1;
    } else {
      std::vector<int32_t> touched;  // pages with a simulated change
      for (size_t k = 0; k < ids.size(); ++k) {
        auto& toks = seqs[ids[k]];
        moving_pages(toks, orders[k]);
        std::vector<int32_t> cow;
        for (int32_t q : orders[k])
          if (K.rc(q) + sim_rc[q] > 1) cow.push_back(q);
        need += int64_t(cow.size());
        if (cow.empty()) continue;
        mk.next();
        for (const Tok& t : toks)
          if (!t.vis) mk.test_set(t.kp);  // marked: a dropped token of this sequence sits in the page
        for (int32_t q : cow)
          if (!mk.test(q)) {
            if (sim_rc[q] == 0) touched.push_back(q);
            sim_rc[q] -= 1;
          }
      }
      for (int32_t q : touched) sim_rc[q] = 0;
    }
    if (need > K.n_free()) fail(AKV_ERR_NO_PAGES, "flush needs %lld copy-on-write pages", (long long)need);

    std::vector<akv::RunDesc> runs;
    std::vector<int32_t> deltas;          // distinct shifts, first-appearance order
    std::unordered_map<int32_t, int32_t> didx;
    std::vector<int32_t> flat;
    for (size_t k = 0; k < ids.size(); ++k) flush_seq(seqs[ids[k]], orders[k], runs, deltas, didx, flat);
    if (!runs.empty()) last_runs.swap(flat);
    if (meta || runs.empty()) return;

    // A page shared by two flushed sequences is copied out by the first
    // (copy-on-write) and, its reference gone, rotated in place by the second.
    // Runs execute concurrently within a launch, so when some page is both a
    // copy source and an in-place target the copies go in a first launch and
    // the in-place runs in a second (the bookkeeping applies them in order).
    std::stable_partition(runs.begin(), runs.end(), [](const akv::RunDesc& r) { return r.src != r.dst; });
    int n_copy = 0;
    while (n_copy < int(runs.size()) && runs[n_copy].src != runs[n_copy].dst) ++n_copy;
    bool conflict = false;
    if (n_copy > 0 && n_copy < int(runs.size())) {
      mk.next();
      for (int i = 0; i < n_copy; ++i) mk.test_set(runs[i].src);
      for (size_t i = n_copy; i < runs.size() && !conflict; ++i) conflict = mk.test(runs[i].dst);
    }
    std::vector<float2> cs = angle_table(deltas);
    if (corrupt_next == 1) {  // checked-build test hook: a row range past the page
      runs[0].lohi = (runs[0].lohi & 0xffff) | ((cfg.page_size + 1) << 16);
      corrupt_next = 0;
    }
    void* druns = nullptr;
    void* dcs = nullptr;
    up.upload({{runs.data(), runs.size() * sizeof(akv::RunDesc), &druns}, {cs.data(), cs.size() * sizeof(float2), &dcs}},
              st);
    int64_t rows = 0;
    for (auto& r : runs) rows += (r.lohi >> 16) - (r.lohi & 0xffff);
    Timed t;
    const double bytes = 2.0 * double(rows) * cfg.n_layers * cfg.n_kv_heads * cfg.d_rot * 2.0;
    begin_timed(kRepos, bytes, 0.0, st, t, conflict ? 2 : 1);
    auto launch = [&](int first, int n) {
      cuda_check(akv::launch_repos_rotate(kpool, static_cast<akv::RunDesc*>(druns) + first, static_cast<float2*>(dcs),
                                          n, cfg.n_layers, cfg.n_kv_heads, cfg.d_rot, cfg.page_size, cfg.n_pages,
                                          cfg.rope_layout == AKV_ROPE_HALF, dev_err, st),
                 "repos_rotate launch");
    };
    if (conflict) {
      launch(0, n_copy);
      launch(n_copy, int(runs.size()) - n_copy);
    } else {
      launch(0, int(runs.size()));
    }
    end_timed(t, st);
    up.done(st);
  }

  // (cos, sin)(delta * theta_j) for each distinct shift, evaluated in float64
  // and stored as float32: [deltas][d_rot / 2].
  std::vector<float2> angle_table(const std::vector<int32_t>& deltas) const {
    const int half = cfg.d_rot / 2;
    std::vector<double> th(half);  // theta_j, the same for every shift
    for (int j = 0; j < half; ++j) th[j] = std::pow(cfg.rope_base, -2.0 * j / cfg.d_rot);
    std::vector<float2> cs(deltas.size() * half);
    for (size_t d = 0; d < deltas.size(); ++d)
      for (int j = 0; j < half; ++j) {
        const double a = double(deltas[d]) * th[j];
        cs[d * half + j] = make_float2(float(std::cos(a)), float(std::sin(a)));
      }
    return cs;
  }

  void debug_rotate_f32(const int32_t* in, int32_t n_runs, float* out, cudaStream_t st) {
    if (meta) fail(AKV_ERR_ARG, "metadata-only context has no pools");
    if (n_runs < 0 || (n_runs > 0 && (!in || !out))) fail(AKV_ERR_ARG, "bad run list");
    std::vector<akv::RunDesc> runs(n_runs);
    std::vector<int32_t> row_off(n_runs), deltas;
    std::unordered_map<int32_t, int32_t> didx;
    int64_t rows = 0;
    for (int32_t r = 0; r < n_runs; ++r) {
      const int32_t pg = in[4 * r], lo = in[4 * r + 1], hi = in[4 * r + 2], d = in[4 * r + 3];
      if (pg < 0 || pg >= cfg.n_pages || lo < 0 || lo >= hi || hi > cfg.page_size)
        fail(AKV_ERR_RANGE, "run %d outside the pool", r);
      auto it = didx.find(d);
      if (it == didx.end()) {
        it = didx.emplace(d, int32_t(deltas.size())).first;
        deltas.push_back(d);
      }
      runs[r] = akv::RunDesc{pg, pg, lo | (hi << 16), it->second};
      row_off[r] = int32_t(rows);
      rows += hi - lo;
    }
    if (n_runs == 0) return;
    std::vector<float2> cs = angle_table(deltas);
    void* druns = nullptr;
    void* dcs = nullptr;
    void* doff = nullptr;
    up.upload({{runs.data(), runs.size() * sizeof(akv::RunDesc), &druns},
               {cs.data(), cs.size() * sizeof(float2), &dcs},
               {row_off.data(), row_off.size() * 4, &doff}},
              st);
    cuda_check(akv::launch_repos_rotate_f32(kpool, static_cast<akv::RunDesc*>(druns), static_cast<float2*>(dcs),
                                            static_cast<int32_t*>(doff), rows, out, n_runs, cfg.n_layers,
                                            cfg.n_kv_heads, cfg.d_rot, cfg.page_size, cfg.n_pages,
                                            cfg.rope_layout == AKV_ROPE_HALF, dev_err, st),
               "repos_rotate f32 launch");
    up.done(st);
  }

  // order: the sequence's moving pages in first-appearance order (moving_pages).
  void flush_seq(std::vector<Tok>& toks, const std::vector<int32_t>& order, std::vector<akv::RunDesc>& runs,
                 std::vector<int32_t>& deltas, std::unordered_map<int32_t, int32_t>& didx, std::vector<int32_t>& flat) {
    if (order.empty()) return;
    std::vector<int32_t> cow;
    for (int32_t q : order) {  // page_dst: source page -> destination page
      if (K.rc(q) > 1) {
        cow.push_back(q);
        page_dst[q] = K.alloc();
      } else {
        page_dst[q] = q;
      }
    }
    mk.next();
    for (int32_t q : cow) mk.test_set(q);  // marked = copied page
    mv.next();                             // marked = a copied page that keeps a token of this sequence
    // One pass: runs (maximal groups of consecutive emitted tokens with equal
    // source, destination and shift, consecutive slots), and each emitted
    // token moved to its destination with its shift folded into its position.
    bool open = false;
    int32_t c_src = 0, c_dst = 0, c_delta = 0, c_lo = 0, c_hi = 0;
    auto close = [&]() {
      if (!open) return;
      auto it = didx.find(c_delta);
      int32_t di;
      if (it == didx.end()) {
        di = int32_t(deltas.size());
        didx.emplace(c_delta, di);
        deltas.push_back(c_delta);
      } else {
        di = it->second;
      }
      runs.push_back(akv::RunDesc{c_src, c_dst, c_lo | (c_hi << 16), di});
      flat.insert(flat.end(), {c_src, c_dst, c_lo, c_hi, c_delta});
      open = false;
    };
    int32_t last = -1, last_dst = -1;  // page of the previous token, its destination
    bool last_copied = false;
    for (Tok& t : toks) {
      if (t.kp != last) {  // consecutive tokens mostly share their page
        last = t.kp;
        last_copied = mk.test(t.kp);
        last_dst = page_dst[t.kp];  // meaningful for moving pages only
      }
      const bool copied = last_copied;
      const bool emit = t.vis && (t.delta != 0 || copied);
      if (!emit) {
        if (copied) mv.test_set(t.kp);  // a dropped token stays behind in the copied page
        close();
        continue;
      }
      const int32_t d = last_dst;  // emitted tokens sit in moving pages
      if (open && c_src == t.kp && c_dst == d && c_delta == t.delta && t.slot == c_hi) {
        ++c_hi;
      } else {
        close();
        open = true;
        c_src = t.kp;
        c_dst = d;
        c_delta = t.delta;
        c_lo = t.slot;
        c_hi = t.slot + 1;
      }
      t.kp = d;
      t.pos += t.delta;
      t.delta = 0;
    }
    close();
    // A copied page loses this sequence's reference unless a dropped token stays in it.
    for (int32_t q : cow)
      if (!mv.test(q)) K.dec(q);
  }

  // -------------------------------------------------------------- segments
  struct SegPlan {
    std::vector<akv::AttnRun> runs;
    std::vector<int32_t> shift;  // fused plans: pending shift of each run's tokens
    std::vector<int32_t> tok;    // with want_tok: logical token index of each entry
    int64_t kv_len = 0;
  };

  void validate_segment(const akv_segment& g, int64_t n_q_rows) {
    auto& toks = seq(g.seq);
    if (g.reserved != 0) fail(AKV_ERR_ARG, "segment reserved field must be 0");
    if (g.q_len < 1 || g.kv_end < g.q_len || g.kv_end > int64_t(toks.size()))
      fail(AKV_ERR_RANGE, "segment outside the sequence");
    if (n_q_rows >= 0 && (g.q_row0 < 0 || g.q_row0 + g.q_len > n_q_rows)) fail(AKV_ERR_RANGE, "segment rows outside Q");
    if (g.n_hide < 0 || (g.n_hide > 0 && !g.hide)) fail(AKV_ERR_ARG, "bad hidden span list");
    for (int32_t h = 0; h < g.n_hide; ++h) {
      int64_t a = g.hide[2 * h], b = g.hide[2 * h + 1];
      if (a < 0 || a > b || b > g.kv_end) fail(AKV_ERR_RANGE, "hidden span outside the segment");
      if (b > g.kv_end - g.q_len && a < b) fail(AKV_ERR_ARG, "a query token of the segment is hidden");
    }
    for (int64_t i = g.kv_end - g.q_len; i < g.kv_end; ++i)
      if (!toks[i].vis) fail(AKV_ERR_ARG, "a query token of the segment is dropped");
  }

  // Runs of the segment's visible entries in logical order: maximal groups of
  // consecutive slots of one (K page, V page).  With `fused` the tokens may
  // carry pending shifts; runs then also break where the shift changes, and
  // each run records it (the attention kernel rotates those keys on the fly).
  SegPlan plan_segment(const akv_segment& g, bool fused = false, bool want_tok = false) {
    auto& toks = seq(g.seq);
    std::vector<uint8_t> hidden;
    if (g.n_hide > 0) {
      hidden.assign(size_t(g.kv_end), 0);
      for (int32_t h = 0; h < g.n_hide; ++h)
        for (int64_t i = g.hide[2 * h]; i < g.hide[2 * h + 1]; ++i) hidden[i] = 1;
    }
    SegPlan sp;
    bool open = false;
    akv::AttnRun cur{};
    int32_t lo = 0, hi = 0;
    for (int64_t i = 0; i < g.kv_end; ++i) {
      const Tok& t = toks[i];
      if (!t.vis || (!hidden.empty() && hidden[i])) continue;
      if (!fused && t.delta != 0) fail(AKV_ERR_ARG, "segment reads token %lld with a pending shift", (long long)i);
      if (open && cur.kp == t.kp && cur.vp == t.vp && t.slot == hi && (!fused || t.delta == sp.shift.back())) {
        ++hi;
      } else {
        if (open) {
          cur.lohi = lo | (hi << 16);
          sp.runs.push_back(cur);
        }
        if (fused) sp.shift.push_back(t.delta);
        open = true;
        cur.kp = t.kp;
        cur.vp = t.vp;
        cur.es = int32_t(sp.kv_len);
        lo = t.slot;
        hi = t.slot + 1;
      }
      if (want_tok) sp.tok.push_back(int32_t(i));
      ++sp.kv_len;
    }
    if (open) {
      cur.lohi = lo | (hi << 16);
      sp.runs.push_back(cur);
    }
    return sp;
  }

  // Split-KV for the MLA kernel (one CTA pair per pair of units): cut every
  // pair's KV-tile range into chunks so the launch ends as early as an
  // estimate of its schedule says; split chunks write partials and the chunk
  // that finishes last merges them.  Pairs run longest first (LPT), ties in
  // (segment, tile, half, chunk) order.
  static constexpr double kMlaUnitCost = 6.0;  // start + epilogue of a unit, in KV tiles (fitted to measured launches)
  static constexpr double kMlaPartCost = 8.0;  // the same for a split part (partial write, merge share)
  void plan_split(std::vector<akv::AttnWork>& work, std::vector<akv::CombineItem>& comb, int32_t& n_parts) {
    // work holds CTA pairs (2i, 2i + 1) sharing one KV range; a pair is cut
    // and scheduled as one.
    const int64_t pair_slots = std::max(1, mla_slots / 2);
    const size_t n_items = work.size() / 2;
    // Estimated makespan of a cut (chunks per item), in KV tiles: units run
    // longest first, each on the pair that frees first; a unit costs its
    // tiles plus a start and epilogue (more for a split part: its partial
    // write and a share of the merge).
    auto makespan = [&](const std::vector<int>& chunks) {
      std::vector<double> cost;
      for (size_t k = 0; k < n_items; ++k) {
        const int span = std::max(1, work[2 * k].n_a);
        for (int c = 0; c < chunks[k]; ++c)
          cost.push_back(double(span) / chunks[k] + (chunks[k] > 1 ? kMlaPartCost : kMlaUnitCost));
      }
      return lpt_makespan(std::move(cost), pair_slots);
    };
    // Candidates: every item in S chunks, or in S chunks with the smallest
    // number of items in S + 1 that fills the last wave of pairs.
    std::vector<int> best_chunks(n_items, 1);
    double best = -1.0;
    const int cands[] = {1, 2, 3, 4, 6, 8};
    for (int S : cands) {
      if (split_override > 0 && S != split_override) continue;
      for (int top = 0; top < 2; ++top) {
        std::vector<int> ch(n_items);
        int64_t units = 0;
        for (size_t k = 0; k < n_items; ++k) units += ch[k] = std::min(S, std::max(1, work[2 * k].n_a));
        if (top) {
          if (split_override > 0 || units % pair_slots == 0) continue;
          int64_t need = pair_slots - units % pair_slots;
          for (size_t k = n_items; k-- > 0 && need > 0;)
            if (ch[k] < 8 && ch[k] < work[2 * k].n_a) {
              ++ch[k];
              --need;
            }
        }
        const double m = makespan(ch);
        if (best < 0.0 || m < best - 1e-9) {
          best = m;
          best_chunks = ch;
        }
      }
    }
    if (split_override > 0)
      for (size_t k = 0; k < n_items; ++k) best_chunks[k] = std::min(std::min(split_override, 8), std::max(1, work[2 * k].n_a));
    std::vector<std::array<akv::AttnWork, 2>> pairs;
    for (size_t k = 0; k < work.size(); k += 2) {
      const int span = work[k].n_a;
      const int chunks = best_chunks[k / 2];
      int32_t base[2] = {-1, -1}, ci[2] = {-1, -1};
      if (chunks > 1) {
        for (int m = 0; m < 2; ++m) {
          if (work[k + m].kvh & akv::kShadow) continue;  // a shadow writes nothing, so owns no parts
          comb.push_back(akv::CombineItem{n_parts, chunks, {0, 0}});
          base[m] = n_parts;
          ci[m] = int32_t(comb.size()) - 1;
          n_parts += chunks;
        }
      }
      for (int c = 0; c < chunks; ++c) {
        std::array<akv::AttnWork, 2> pr = {work[k], work[k + 1]};
        for (int m = 0; m < 2; ++m) {
          pr[m].t0 = int32_t(int64_t(span) * c / chunks);
          pr[m].t1 = int32_t(int64_t(span) * (c + 1) / chunks);
          pr[m].part = base[m] >= 0 ? base[m] + c : -1;
          pr[m].comb = ci[m];
        }
        pairs.push_back(pr);
      }
    }
    auto cost = [](const std::array<akv::AttnWork, 2>& pr) {
      return std::max(0, std::min(pr[0].n_a, pr[0].t1) - pr[0].t0);
    };
    std::stable_sort(pairs.begin(), pairs.end(),
                     [&](const std::array<akv::AttnWork, 2>& a, const std::array<akv::AttnWork, 2>& b) {
                       return cost(a) > cost(b);
                     });
    work.clear();
    for (auto& pr : pairs) {
      work.push_back(pr[0]);
      work.push_back(pr[1]);
    }
  }

  // Persistent schedule for the MLA kernel (automatic split): the pair items
  // (work entries 2k, 2k + 1: one KV range, one output half) are laid end to
  // end in their order (consecutive items of one segment share its K/V in L2)
  // as sequences of KV tiles, each unit costing its tiles plus a start cost.
  // A pair's list takes units in that order until the next would exceed a
  // budget B, cutting the item at the budget (stream-K); the plan is the fill
  // with the smallest B that fits the resident CTA pairs, which minimises the
  // busiest pair's cost (the launch's length) among in-order fills.  An item
  // crossing a cut becomes several units whose partials the last to finish
  // merges; no piece is shorter than kMlaMinTiles (the cut moves back
  // instead) and no item is cut into more than 8 parts.  Pair b runs units
  // [cta_units[b], cta_units[b + 1]) (unit u = work entries 2u, 2u + 1).
  static constexpr int64_t kMlaMinTiles = 4;
  void plan_mla_persistent(std::vector<akv::AttnWork>& work, std::vector<akv::CombineItem>& comb, int32_t& n_parts,
                           std::vector<int32_t>& cta_units) {
    const int64_t pair_slots = std::max(1, mla_slots / 2);
    const size_t n_items = work.size() / 2;
    const int64_t unit_cost = int64_t(kMlaUnitCost);
    auto span_of = [&](size_t k) { return int64_t(std::max(1, work[2 * k].n_a)); };
    int64_t items_cost = 0;
    for (size_t k = 0; k < n_items; ++k) items_cost += unit_cost + span_of(k);
    struct Piece {
      size_t item;
      int32_t t0, t1;
    };
    std::vector<Piece> pieces;
    const int64_t n_pairs = std::max<int64_t>(1, std::min<int64_t>(pair_slots, items_cost / (4 * unit_cost)));
    // in-order fill under budget B; false when it needs more than n_pairs
    // pairs or an item more than 8 parts
    auto fill = [&](int64_t budget) {
      pieces.clear();
      cta_units.assign(1, 0);
      int64_t room = budget;
      for (size_t k = 0; k < n_items; ++k) {
        const int64_t span = span_of(k);
        int64_t start = 0;
        int32_t parts = 0;
        for (;;) {
          const int64_t rest = span - start;
          if (unit_cost + rest <= room) {
            pieces.push_back(Piece{k, int32_t(start), int32_t(span)});
            room -= unit_cost + rest;
            break;
          }
          int64_t take = room - unit_cost;
          if (rest - take < kMlaMinTiles) take = rest - kMlaMinTiles;
          const bool cut = take >= kMlaMinTiles && parts < 7;
          if (cut) {
            pieces.push_back(Piece{k, int32_t(start), int32_t(start + take)});
            start += take;
            ++parts;
          } else if (room == budget) {
            return false;  // a fresh pair can take nothing of this item
          }
          cta_units.push_back(int32_t(pieces.size()));
          if (int64_t(cta_units.size()) > n_pairs) return false;
          room = budget;
        }
      }
      if (cta_units.back() != int32_t(pieces.size())) cta_units.push_back(int32_t(pieces.size()));
      return int64_t(cta_units.size()) - 1 <= n_pairs;
    };
    int64_t lo = std::max<int64_t>(unit_cost + 1, items_cost / n_pairs), hi = items_cost;  // fill(hi) holds
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (fill(mid))
        hi = mid;
      else
        lo = mid + 1;
    }
    fill(hi);
    std::vector<int32_t> n_of(n_items, 0);
    for (const Piece& pc : pieces) ++n_of[pc.item];
    // partial slots and ticket counters of the items cut into several units
    // (a shadow writes nothing, so owns no parts)
    std::vector<int32_t> base_of(work.size(), -1), comb_of(work.size(), -1), next_of(n_items, 0);
    for (size_t k = 0; k < n_items; ++k) {
      if (n_of[k] < 2) continue;
      for (size_t m = 0; m < 2; ++m) {
        if (work[2 * k + m].kvh & akv::kShadow) continue;
        comb.push_back(akv::CombineItem{n_parts, n_of[k], {0, 0}});
        base_of[2 * k + m] = n_parts;
        comb_of[2 * k + m] = int32_t(comb.size()) - 1;
        n_parts += n_of[k];
      }
    }
    std::vector<akv::AttnWork> units;
    units.reserve(2 * pieces.size());
    for (const Piece& pc : pieces) {
      const int32_t idx = next_of[pc.item]++;
      for (size_t m = 0; m < 2; ++m) {
        akv::AttnWork e = work[2 * pc.item + m];
        e.t0 = pc.t0;
        e.t1 = pc.t1;
        e.part = base_of[2 * pc.item + m] >= 0 ? base_of[2 * pc.item + m] + idx : -1;
        e.comb = comb_of[2 * pc.item + m];
        units.push_back(e);
      }
    }
    work.swap(units);
  }

  // K-tile ranges of the attention-mass pass.  The lse is final, so a pair
  // item's K tiles can be cut into ranges that run as separate CTAs and add
  // into the same outputs, with no merge.  Every item is cut into S equal
  // ranges (or S + 1 for the fewest items that fill the last wave), S taken
  // from the estimated makespan over one CTA per SM; a range costs its
  // (K tile, query tile) steps plus a start (Q tiles, pipeline fill, drain).
  // CTAs run longest first.
  static constexpr int32_t kMassPartCost = 4;  // a CTA's start and drain, in (K tile, query tile) steps
  void plan_mass_split(std::vector<akv::AttnWork>& work) {
    const size_t n_items = work.size();
    auto tiles = [](const akv::AttnWork& w) { return std::max(w.n_a, w.n_b); };
    auto range = [&](const akv::AttnWork& w, int S, int c) {
      return std::make_pair(int32_t(int64_t(tiles(w)) * c / S), int32_t(int64_t(tiles(w)) * (c + 1) / S));
    };
    auto cost = [](const akv::AttnWork& w, int32_t t0, int32_t t1) {
      return std::max(0, std::min(w.n_a, t1) - t0) + std::max(0, std::min(w.n_b, t1) - t0) + kMassPartCost;
    };
    // largest items first: the extra range of a top-up goes to them
    std::stable_sort(work.begin(), work.end(),
                     [&](const akv::AttnWork& a, const akv::AttnWork& b) { return cost(a, 0, tiles(a)) > cost(b, 0, tiles(b)); });
    // costs as a histogram; items alike (the kv heads of one query-tile
    // pair, adjacent after the sort) are costed once
    int32_t max_cost = 0;
    for (const auto& w : work) max_cost = std::max(max_cost, cost(w, 0, tiles(w)));
    std::vector<int64_t> hist;
    auto makespan = [&](const std::vector<int>& ch) {
      hist.assign(size_t(max_cost) + 1, 0);
      for (size_t k = 0; k < n_items;) {
        size_t e = k + 1;
        while (e < n_items && ch[e] == ch[k] && work[e].n_a == work[k].n_a && work[e].n_b == work[k].n_b) ++e;
        for (int i = 0; i < ch[k]; ++i) {
          const auto r = range(work[k], ch[k], i);
          hist[size_t(cost(work[k], r.first, r.second))] += int64_t(e - k);
        }
        k = e;
      }
      return wave_makespan(hist, n_sm);
    };
    std::vector<int> best_ch(n_items, 1);
    int64_t best = -1;
    const int cands[] = {1, 2, 3, 4, 5, 6, 8};
    for (int S : cands) {
      if (split_override > 0 && S != std::min(split_override, 8)) continue;
      for (int top = 0; top < 2; ++top) {
        std::vector<int> ch(n_items);
        int64_t units = 0;
        for (size_t k = 0; k < n_items; ++k) units += ch[k] = std::min(S, std::max(1, tiles(work[k])));
        if (top) {
          if (split_override > 0 || units % n_sm == 0) continue;
          int64_t need = n_sm - units % n_sm;
          for (size_t k = 0; k < n_items && need > 0; ++k)
            if (ch[k] < 8 && ch[k] < tiles(work[k])) {
              ++ch[k];
              --need;
            }
        }
        const int64_t m = makespan(ch);
        if (best < 0 || m < best) {
          best = m;
          best_ch = ch;
        }
      }
    }
    std::vector<std::pair<int32_t, akv::AttnWork>> parts;
    for (size_t k = 0; k < n_items; ++k)
      for (int i = 0; i < best_ch[k]; ++i) {
        akv::AttnWork w = work[k];
        const auto r = range(w, best_ch[k], i);
        w.t0 = r.first;
        w.t1 = r.second;
        parts.emplace_back(cost(w, w.t0, w.t1), w);
      }
    std::stable_sort(parts.begin(), parts.end(),
                     [](const auto& a, const auto& b) { return a.first > b.first; });
    work.clear();
    for (const auto& pr : parts) work.push_back(pr.second);
  }

  // Persistent stream-K schedule for the GQA kernel: one CTA per SM, each
  // running an equal share of the work.  Items (query-tile pair x kv head)
  // are laid end to end as a sequence of KV-tile steps, each step costing
  // the query tiles it feeds (1 or 2), plus a fixed cost per unit for its
  // start and epilogue.  The sequence is cut into n_cta contiguous pieces of
  // equal cost; an item crossing a cut becomes several units (parts) whose
  // partial results the last one to finish merges.  A cut never leaves a
  // piece of an item shorter than kMinSteps steps.  akv_set_attention_split
  // (n >= 1) instead cuts every item into n equal parts, one CTA per unit.
  //
  // A launch with many items per CTA (many segments) is first laid out for L2
  // reuse: items are sorted by kv head, then sequence, segment and query tile
  // (items of one kv head of one sequence, or of forks sharing its pages, read
  // the same K/V), then dealt in that order, each to the CTA with the least
  // work so far, and the CTAs' lists are laid end to end before the cut.  The
  // CTAs running at the same time then all work on one or two such groups, so
  // each K/V tile is fetched from HBM about once per group instead of once per
  // item.  Units then run in that order inside each CTA.
  void plan_persistent(std::vector<akv::AttnWork>& work, std::vector<akv::CombineItem>& comb, int32_t& n_parts,
                       std::vector<int32_t>& cta_units, const std::vector<int32_t>& seg_seq) {
    if (split_override > 0) {
      std::vector<akv::AttnWork> units;
      for (auto& w : work) {
        const int span = w.t1;
        const int chunks = std::min(split_override, std::max(1, span));
        if (chunks > 1) comb.push_back(akv::CombineItem{n_parts, chunks, {0, 0}});
        for (int c = 0; c < chunks; ++c) {
          akv::AttnWork u = w;
          u.t0 = int32_t(int64_t(span) * c / chunks);
          u.t1 = int32_t(int64_t(span) * (c + 1) / chunks);
          if (chunks > 1) {
            u.part = n_parts++;
            u.comb = int32_t(comb.size()) - 1;
          }
          units.push_back(u);
        }
      }
      work.swap(units);
      cta_units.clear();
      return;
    }
    constexpr int64_t kUnitCost = 1;   // start + epilogue of a unit, in query-tile steps (measured: 1 to 14 within 0.6 %, 1 best)
    constexpr int64_t kMinSteps = 4;   // shortest piece of an item worth a unit
    constexpr int64_t kMinCtaCost = 48;
    constexpr int64_t kGroupedItemsPerCta = 4;  // from this many items per CTA on, lay items out by K/V group
    // cost of the first j steps of item w (O(1): each query tile feeds its first n steps)
    auto prefix = [](const akv::AttnWork& w, int64_t j) {
      return std::min<int64_t>(j, w.n_a) + std::min<int64_t>(j, w.n_b);
    };
    int64_t total = 0;
    for (auto& w : work) total += kUnitCost + prefix(w, w.t1);
    const int64_t n_cta = std::max<int64_t>(1, std::min<int64_t>(n_sm, total / kMinCtaCost));
    const bool grouped = int64_t(work.size()) >= kGroupedItemsPerCta * n_cta;
    if (grouped) {
      std::vector<size_t> idx(work.size());
      for (size_t i = 0; i < idx.size(); ++i) idx[i] = i;
      std::stable_sort(idx.begin(), idx.end(), [&](size_t a, size_t b) {
        const akv::AttnWork &x = work[a], &y = work[b];
        const int32_t sx = seg_seq[size_t(x.seg)], sy = seg_seq[size_t(y.seg)];
        if (x.kvh != y.kvh) return x.kvh < y.kvh;
        if (sx != sy) return sx < sy;
        if (x.seg != y.seg) return x.seg < y.seg;
        return x.qt0 < y.qt0;
      });
      std::vector<std::vector<size_t>> lists;
      lists.resize(static_cast<size_t>(n_cta));
      std::priority_queue<std::pair<int64_t, int64_t>, std::vector<std::pair<int64_t, int64_t>>, std::greater<>> load;
      for (int64_t c = 0; c < n_cta; ++c) load.emplace(0, c);
      for (size_t i : idx) {
        auto [l, c] = load.top();
        load.pop();
        lists[size_t(c)].push_back(i);
        load.emplace(l + kUnitCost + prefix(work[i], work[i].t1), c);
      }
      std::vector<akv::AttnWork> dealt;
      dealt.reserve(work.size());
      for (const auto& l : lists)
        for (size_t i : l) dealt.push_back(work[i]);
      work.swap(dealt);
    }
    std::vector<akv::AttnWork> units;
    std::vector<int32_t> item_of;  // unit -> item index
    total += (n_cta - 1) * kUnitCost;  // each cut starts one more unit
    units.reserve(work.size() + size_t(n_cta));
    item_of.reserve(work.size() + size_t(n_cta));
    cta_units.assign(1, 0);
    int64_t acc = 0, cta = 0;
    auto boundary = [&]() { return (cta + 1) * total / n_cta; };
    auto close_cta = [&]() {
      cta_units.push_back(int32_t(units.size()));
      ++cta;
    };
    for (size_t it = 0; it < work.size(); ++it) {
      const akv::AttnWork& w = work[it];
      const int64_t span = w.t1;
      int64_t start = 0;
      acc += kUnitCost;
      const int64_t base0 = acc;  // acc = base0 + prefix(j) after j steps of this item
      int64_t base = base0;
      bool close_at_end = false;
      while (cta < n_cta - 1 && base + prefix(w, span) >= boundary()) {
        // first step count j (> start) at which the running cost reaches the boundary
        const int64_t target = boundary() - base;
        int64_t lo = start + 1, hi = span;
        while (lo < hi) {
          const int64_t mid = (lo + hi) / 2;
          if (prefix(w, mid) >= target) hi = mid; else lo = mid + 1;
        }
        int64_t j = std::max(lo, start + kMinSteps);  // a piece is never shorter than kMinSteps
        if (span - j < kMinSteps) {
          close_at_end = true;  // finish the item in this CTA
          break;
        }
        akv::AttnWork u = w;
        u.t0 = int32_t(start);
        u.t1 = int32_t(j);
        units.push_back(u);
        item_of.push_back(int32_t(it));
        close_cta();
        start = j;
        base += kUnitCost;  // the next piece starts a unit
      }
      akv::AttnWork u = w;
      u.t0 = int32_t(start);
      u.t1 = int32_t(span);
      units.push_back(u);
      item_of.push_back(int32_t(it));
      acc = base + prefix(w, span);
      if (close_at_end && cta < n_cta - 1) close_cta();
    }
    if (cta_units.back() != int32_t(units.size())) close_cta();
    // Order inside each CTA (a few items per CTA): the piece that starts an
    // item (at KV step 0) first, then the piece that ends an item cut by the
    // previous CTA, then whole items.  With items of similar length every CTA
    // then reads the same KV step of its item at about the same time (three
    // phases in all), so the K/V tiles a step needs are fetched from HBM once
    // and served to the other CTAs from L2.
    if (!grouped) {
      std::vector<akv::AttnWork> ordered;
      std::vector<int32_t> ordered_item;
      ordered.reserve(units.size());
      ordered_item.reserve(units.size());
      for (size_t b = 0; b + 1 < cta_units.size(); ++b) {
        const size_t a0 = size_t(cta_units[b]), a1 = size_t(cta_units[b + 1]);
        auto is_head = [&](size_t u) { return units[u].t0 == 0 && units[u].t1 < work[size_t(item_of[u])].t1; };
        auto is_tail = [&](size_t u) { return units[u].t0 > 0; };
        for (int pass = 0; pass < 3; ++pass)
          for (size_t u = a0; u < a1; ++u) {
            const bool h = is_head(u), t = is_tail(u);
            if ((pass == 0 && h) || (pass == 1 && t && !h) || (pass == 2 && !h && !t)) {
              ordered.push_back(units[u]);
              ordered_item.push_back(item_of[u]);
            }
          }
      }
      units.swap(ordered);
      item_of.swap(ordered_item);
    }
    // Items cut into several units: consecutive partial slots per item and a
    // ticket counter.
    std::vector<int32_t> n_of(work.size(), 0), comb_of(work.size(), -1), next_of(work.size(), 0);
    for (int32_t i : item_of) ++n_of[size_t(i)];
    for (size_t it = 0; it < work.size(); ++it) {
      if (n_of[it] < 2) continue;
      comb_of[it] = int32_t(comb.size());
      comb.push_back(akv::CombineItem{n_parts, n_of[it], {0, 0}});
      next_of[it] = n_parts;
      n_parts += n_of[it];
    }
    for (size_t u = 0; u < units.size(); ++u) {
      const size_t it = size_t(item_of[u]);
      if (comb_of[it] < 0) continue;
      units[u].part = next_of[it]++;
      units[u].comb = comb_of[it];
    }
    work.swap(units);
  }

  // fused: leave pending shifts pending and rotate those keys inside the
  // attention kernel (no flush, no copy-on-write, no HBM writes of K).
  void attend(int32_t layer, const akv_segment* segs, int32_t n_segs, const void* q, int64_t n_q_rows, void* o,
              float* lse, float scale, cudaStream_t st, bool fused = false) {
    if (n_segs < 0 || (n_segs > 0 && !segs)) fail(AKV_ERR_ARG, "bad segment list");
    if (layer < 0 || layer >= cfg.n_layers) fail(AKV_ERR_RANGE, "layer outside the pools");
    if (n_q_rows < 0 || n_q_rows > kI32Max) fail(AKV_ERR_RANGE, "bad query row count");
    if (!meta && n_segs > 0 && (!q || !o)) fail(AKV_ERR_ARG, "null Q or O pointer");
    for (int32_t i = 0; i < n_segs; ++i) validate_segment(segs[i], n_q_rows);
    std::vector<int32_t> ids;
    for (int32_t i = 0; i < n_segs; ++i) ids.push_back(segs[i].seq);
    std::sort(ids.begin(), ids.end());
    ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
    if (!fused) flush(ids, st);
    if (n_segs == 0) return;

    const int G = cfg.n_q_heads / cfg.n_kv_heads;
    const int tpt = 128 / G;                   // query tokens per 128-row tile
    const int rpt = 128 / cfg.page_size;       // runs per 128-key tile
    std::vector<akv::AttnRun> runs;
    std::vector<int32_t> run_shift;  // fused: pending shift per run
    std::vector<akv::AttnSeg> tab;
    std::vector<akv::AttnWork> work;
    double flops = 0.0;
    const int dqk = cfg.layout == AKV_LAYOUT_MLA ? cfg.d_v + cfg.d_rot : cfg.d_rot;
    for (int32_t i = 0; i < n_segs; ++i) {
      SegPlan sp = plan_segment(segs[i], fused);
      if (fused) run_shift.insert(run_shift.end(), sp.shift.begin(), sp.shift.end());
      if (sp.kv_len > kI32Max) fail(AKV_ERR_RANGE, "segment too long");
      akv::AttnSeg s{};
      s.run_off = int32_t(runs.size());
      s.n_runs = int32_t(sp.runs.size());
      s.kv_len = int32_t(sp.kv_len);
      s.q_len = segs[i].q_len;
      s.q_row0 = int32_t(segs[i].q_row0);
      const int64_t ql = s.q_len, kl = s.kv_len;
      flops += double(cfg.n_q_heads) * 2.0 * (dqk + cfg.d_v) * double(ql * (kl - ql) + ql * (ql + 1) / 2);
      const int n_qt = (s.q_len + tpt - 1) / tpt;
      // KV tiles query tile qt reads: runs whose first entry is <= the
      // largest entry index its last row may see.
      auto tiles_of = [&](int qt) -> int32_t {
        if (qt >= n_qt) return 0;
        const int64_t last = std::min<int64_t>(ql, int64_t(qt + 1) * tpt) - 1;
        const int64_t limit = kl - ql + last;
        int64_t lo_r = 0, hi_r = int64_t(sp.runs.size());
        while (lo_r < hi_r) {
          int64_t mid = (lo_r + hi_r) / 2;
          if (sp.runs[mid].es <= limit) lo_r = mid + 1; else hi_r = mid;
        }
        return int32_t((lo_r + rpt - 1) / rpt);
      };
      if (cfg.layout == AKV_LAYOUT_MLA) {
        // CTA pairs: query tiles qt and qt + 1 over the KV tiles either reads,
        // one pair per half of the 512 output columns (n_b = half); a missing
        // second tile becomes a shadow of the first
        for (int qt = 0; qt < n_qt; qt += 2) {
          const int32_t nt = std::max(tiles_of(qt), tiles_of(qt + 1));
          const bool shadow = qt + 1 >= n_qt;
          for (int half = 0; half < 2; ++half) {
            work.push_back(akv::AttnWork{i, 0, qt, nt, half, 0, nt, -1, -1});
            work.push_back(akv::AttnWork{i, shadow ? akv::kShadow : 0, shadow ? qt : qt + 1, nt, half, 0, nt, -1, -1});
          }
        }
      } else {
        for (int qt = 0; qt < n_qt; qt += 2) {
          const int32_t na = tiles_of(qt), nb = tiles_of(qt + 1);
          for (int h = 0; h < cfg.n_kv_heads; ++h)
            work.push_back(akv::AttnWork{i, h, qt, na, nb, 0, std::max(na, nb), -1, -1});
        }
      }
      runs.insert(runs.end(), sp.runs.begin(), sp.runs.end());
      tab.push_back(s);
    }
    // Fused rotation: distinct pending shifts -> angle table rows; runs
    // without a shift keep -1 (their keys are read as stored).
    std::vector<int32_t> run_didx, shifts;
    bool rotate = false;
    if (fused) {
      std::unordered_map<int32_t, int32_t> didx;
      run_didx.resize(run_shift.size(), -1);
      for (size_t r = 0; r < run_shift.size(); ++r) {
        if (run_shift[r] == 0) continue;
        auto it = didx.find(run_shift[r]);
        if (it == didx.end()) {
          it = didx.emplace(run_shift[r], int32_t(shifts.size())).first;
          shifts.push_back(run_shift[r]);
        }
        run_didx[r] = it->second;
      }
      rotate = !shifts.empty();
    }
    const bool mla = cfg.layout == AKV_LAYOUT_MLA;
    std::vector<akv::CombineItem> comb;
    std::vector<int32_t> cta_units;  // persistent schedule: CTA (MLA: pair) b runs units [cta_units[b], cta_units[b+1])
    int32_t n_parts = 0;
    if (mla) {
      if (split_override > 0)
        plan_split(work, comb, n_parts);
      else
        plan_mla_persistent(work, comb, n_parts, cta_units);
    } else {
      std::vector<int32_t> seg_seq(static_cast<size_t>(n_segs));
      for (int32_t i = 0; i < n_segs; ++i) seg_seq[size_t(i)] = segs[i].seq;
      plan_persistent(work, comb, n_parts, cta_units, seg_seq);
    }
    if (meta) {  // the plan is kept for inspection (akv_last_attention_plan); no device work
      last_work = work;
      last_cta_units = cta_units;
      return;
    }
    if (mla) {
      if (cfg.d_v != 512 || cfg.d_rot != 64)
        fail(AKV_ERR_ARG, "MLA segment attention supports a 512-wide latent and a 64-wide K_pe");
    } else if (!(cfg.d_rot == 64 || cfg.d_rot == 128)) {
      fail(AKV_ERR_ARG, "GQA segment attention supports head_dim 64 or 128");
    }

    const size_t qbytes = size_t(n_q_rows) * cfg.n_q_heads * dqk * 2;
    const size_t obytes = size_t(n_q_rows) * cfg.n_q_heads * cfg.d_v * 2;
    const void* qd = device_input(q, qbytes, st_q, st);
    const bool o_host = !is_device_ptr(o);
    void* od = o;
    if (o_host) {
      st_o.want_host = false;
      st_o.acquire(obytes);
      od = st_o.dev;
    }
    float* lsed = lse;
    const bool lse_host = lse && !is_device_ptr(lse);
    if (lse_host) {
      st_lse.want_host = false;
      st_lse.acquire(size_t(n_q_rows) * cfg.n_q_heads * 4);
      lsed = static_cast<float*>(st_lse.dev);
    }
    if (reinterpret_cast<uintptr_t>(qd) % 16) fail(AKV_ERR_ARG, "Q must be 16-byte aligned");

    akv::AttnParams p{};
    {
      const uint64_t dims[3] = {uint64_t(dqk), uint64_t(cfg.n_q_heads), uint64_t(std::max<int64_t>(n_q_rows, 1))};
      const uint64_t strides[2] = {uint64_t(dqk) * 2, uint64_t(cfg.n_q_heads) * dqk * 2};
      const uint32_t box[3] = {64, uint32_t(G), uint32_t(tpt)};
      encode_map(&p.q_map, const_cast<void*>(qd), 3, dims, strides, box);
    }
    p.k_map = k_map;
    p.v_map = v_map;
    p.k_tile_map = k_tile_map;
    p.v_tile_map = v_tile_map;
    void* druns = nullptr;
    void* dsegs = nullptr;
    void* dwork = nullptr;
    void* dcomb = nullptr;
    void* dcta = nullptr;
    void* ddidx = nullptr;
    void* dcs = nullptr;
    const std::vector<float2> cs = rotate ? angle_table(shifts) : std::vector<float2>();
    if (!rotate) run_didx.clear();
    if (corrupt_next == 2) {  // checked-build test hook: a K page outside the pool
      runs[0].kp = cfg.n_pages;
      corrupt_next = 0;
    }
    up.upload({{runs.data(), runs.size() * sizeof(akv::AttnRun), &druns},
               {tab.data(), tab.size() * sizeof(akv::AttnSeg), &dsegs},
               {work.data(), work.size() * sizeof(akv::AttnWork), &dwork},
               {comb.data(), comb.size() * sizeof(akv::CombineItem), &dcomb},
               {cta_units.data(), cta_units.size() * sizeof(int32_t), &dcta},
               {run_didx.data(), run_didx.size() * sizeof(int32_t), &ddidx},
               {cs.data(), cs.size() * sizeof(float2), &dcs}},
              st);
    p.runs = static_cast<akv::AttnRun*>(druns);
    p.segs = static_cast<akv::AttnSeg*>(dsegs);
    p.work = static_cast<akv::AttnWork*>(dwork);
    p.o = od;
    p.lse = lsed;
    p.err = dev_err;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.n_work = int32_t(work.size());
    p.cta_units = cta_units.empty() ? nullptr : static_cast<const int32_t*>(dcta);
    p.n_cta = cta_units.empty() ? 0 : int32_t(cta_units.size()) - 1;
    p.layer = layer;
    p.n_pages = cfg.n_pages;
    p.n_layers = cfg.n_layers;
    p.hq = cfg.n_q_heads;
    p.group = G;
    p.page = cfg.page_size;
    p.width = mla ? cfg.d_v / 2 : cfg.d_v;
    p.dv = cfg.d_v;
    p.wait_ns = wait_ns;
    p.load_cap = load_cap;
    p.n_segs = int32_t(tab.size());
    p.n_runs = int32_t(runs.size());
    p.n_q_rows = int32_t(n_q_rows);
    p.fused = rotate ? 1 : 0;
    p.run_didx = rotate ? static_cast<const int32_t*>(ddidx) : nullptr;
    p.cs = rotate ? static_cast<const float2*>(dcs) : nullptr;
    p.rope_half = cfg.rope_layout == AKV_ROPE_HALF ? 1 : 0;
    const int tiles_per_item = mla ? 1 : 2;
    p.comb = static_cast<akv::CombineItem*>(dcomb);
    p.comb_tiles = tiles_per_item;
    if (n_parts > 0) {
      const size_t need = size_t(n_parts) * size_t(akv::partial_floats(tiles_per_item, p.width)) * 4;
      partial.want_host = false;
      partial.acquire(need);
      p.partial = static_cast<float*>(partial.dev);
    }
    Timed t;
    begin_timed(kAttn, 0.0, flops, st, t, 1);
    cuda_check(mla ? akv::launch_segment_attn_mla(p, st) : akv::launch_segment_attn(p, cfg.d_rot, st),
               "segment_attn launch");
    end_timed(t, st);
    up.done(st);
    if (n_parts > 0) partial.release(st);
    if (st_q.dev && !is_device_ptr(q)) st_q.release(st);
    const cudaStream_t ost = output_stream(st);
    if (o_host) {
      cuda_check(cudaMemcpyAsync(o, od, obytes, cudaMemcpyDeviceToHost, ost), "O copy to host");
      st_o.release(ost);
    }
    if (lse_host) {
      cuda_check(cudaMemcpyAsync(lse, lsed, size_t(n_q_rows) * cfg.n_q_heads * 4, cudaMemcpyDeviceToHost, ost),
                 "LSE copy to host");
      st_lse.release(ost);
    }
  }

  // Stream for copies of results to host memory: the caller's stream, or the
  // output stream set by akv_set_output_stream, which first waits for
  // everything enqueued on the caller's stream so far (the kernel that wrote
  // the result).  Then a result copy overlaps the caller's next kernels.
  cudaStream_t output_stream(cudaStream_t st) {
    if (!out_st || out_st == st) return st;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cuda_check(cudaStreamIsCapturing(st, &cs), "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone) return st;
    if (!out_ready) cuda_check(cudaEventCreateWithFlags(&out_ready, cudaEventDisableTiming), "cudaEventCreate");
    cuda_check(cudaEventRecord(out_ready, st), "cudaEventRecord");
    cuda_check(cudaStreamWaitEvent(out_st, out_ready, 0), "cudaStreamWaitEvent");
    return out_st;
  }

  // ---------------------------------------------------------- radix tree
  static bool same_item(const akv_item& x, const akv_item& y) {
    return x.kind == y.kind && x.a == y.a && x.b == y.b && x.c == y.c;
  }
  // what a retrigger match compares: a token without its position
  static bool same_key(const akv_item& x, const akv_item& y) {
    if (x.kind != y.kind) return false;
    if (x.kind == AKV_ITEM_TOKEN) return x.a == y.a;
    return x.a == y.a && x.b == y.b && x.c == y.c;
  }
  static void check_items(const akv_item* items, int64_t n) {
    if (n < 0 || (n > 0 && !items)) fail(AKV_ERR_ARG, "bad item list");
    for (int64_t i = 0; i < n; ++i)
      if (items[i].kind < 0) fail(AKV_ERR_ARG, "item %lld has a negative kind", (long long)i);
  }

  int32_t tree_insert(const akv_item* items, int64_t n, int32_t sid) {
    check_items(items, n);
    auto& toks = seq(sid);
    int64_t n_tok = 0;
    for (int64_t i = 0; i < n; ++i) n_tok += items[i].kind == AKV_ITEM_TOKEN;
    if (n_tok > int64_t(toks.size())) fail(AKV_ERR_RANGE, "path has more tokens than the sequence");
    int32_t at = 0;
    int64_t i = 0;
    for (; i < n; ++i) {  // existing prefix
      int32_t next = -1;
      for (int32_t k : tree[at].kids)
        if (same_item(tree[k].item, items[i])) {
          next = k;
          break;
        }
      if (next < 0) break;
      at = next;
    }
    if (i == n) return -1;  // already present
    int32_t holder = -1;
    fork(sid, n_tok, &holder);
    tree_seqs.push_back(holder);
    const int64_t order = tree_inserts++;
    for (; i < n; ++i) {
      TreeNode nd;
      nd.item = items[i];
      nd.parent = at;
      nd.owner = holder;
      nd.order = order;
      nd.n_tok = tree[at].n_tok + (items[i].kind == AKV_ITEM_TOKEN);
      tree.push_back(nd);
      const int32_t id = int32_t(tree.size()) - 1;
      tree[at].kids.push_back(id);
      at = id;
    }
    return holder;
  }

  // Deepest node (and its depth) reachable under the exact rule, and under the
  // compatible rule (a depth-first walk over every branch whose key matches).
  void tree_walk(const akv_item* items, int64_t n, int32_t& exact_node, int64_t& exact_len, int32_t& comp_node,
                 int64_t& comp_len) {
    exact_node = 0;
    exact_len = 0;
    for (int64_t i = 0; i < n; ++i) {
      int32_t next = -1;
      for (int32_t k : tree[exact_node].kids)
        if (same_item(tree[k].item, items[i])) {
          next = k;
          break;
        }
      if (next < 0) break;
      exact_node = next;
      exact_len = i + 1;
    }
    comp_node = 0;
    comp_len = 0;
    std::vector<std::pair<int32_t, int64_t>> stack{{0, 0}};
    while (!stack.empty()) {
      auto [nd, d] = stack.back();
      stack.pop_back();
      if (d > comp_len || (d == comp_len && d > 0 && tree[nd].order < tree[comp_node].order)) {
        comp_node = nd;
        comp_len = d;
      }
      if (d == n) continue;
      for (int32_t k : tree[nd].kids)
        if (same_key(tree[k].item, items[d])) stack.push_back({k, d + 1});
    }
  }

  akv_match tree_match(const akv_item* items, int64_t n, int32_t* node_out = nullptr) {
    check_items(items, n);
    int32_t en, cn;
    int64_t el, cl;
    tree_walk(items, n, en, el, cn, cl);
    akv_match m{AKV_MATCH_NONE, -1, 0, 0};
    int32_t node = 0;
    if (cl > el) {
      m.kind = AKV_MATCH_RETRIGGER;
      node = cn;
      m.n_items = cl;
    } else if (el > 0) {
      m.kind = AKV_MATCH_EXACT;
      node = en;
      m.n_items = el;
    }
    if (node > 0) {
      m.seq = tree[node].owner;
      m.n_tokens = tree[node].n_tok;
    }
    if (node_out) *node_out = node;
    return m;
  }

  int32_t tree_reuse(const akv_item* items, int64_t n, akv_match* out, cudaStream_t st) {
    int32_t node = 0;
    const akv_match m = tree_match(items, n, &node);
    if (out) *out = m;
    if (m.kind == AKV_MATCH_NONE) return -1;
    // shifts: request position - cached position, per token of the matched path
    std::vector<int32_t> shift;
    if (m.kind == AKV_MATCH_RETRIGGER) {
      std::vector<const akv_item*> path;
      for (int32_t k = node; k > 0; k = tree[k].parent) path.push_back(&tree[k].item);
      std::reverse(path.begin(), path.end());
      for (size_t i = 0; i < path.size(); ++i)
        if (path[i]->kind == AKV_ITEM_TOKEN) {
          const int64_t d = int64_t(items[i].b) - path[i]->b;
          if (d < kI32Min || d > kI32Max) fail(AKV_ERR_OVERFLOW, "position shift of token %zu leaves int32", i);
          shift.push_back(int32_t(d));
        }
    }
    int32_t sid = -1;
    fork(m.seq, m.n_tokens, &sid);
    try {
      for (size_t a = 0; a < shift.size();) {
        size_t b = a + 1;
        while (b < shift.size() && shift[b] == shift[a]) ++b;
        if (shift[a] != 0) repos(sid, int64_t(a), int64_t(b), shift[a]);
        a = b;
      }
      if (!shift.empty()) flush(std::vector<int32_t>{sid}, st);
    } catch (...) {
      free_seq(sid);  // leave nothing behind on failure
      throw;
    }
    return sid;
  }

  void tree_clear() {
    for (int32_t q : tree_seqs)
      if (q >= 0 && q < int32_t(seqs.size()) && live[q]) free_seq(q);
    tree_seqs.clear();
    tree.assign(1, TreeNode{});
    tree_inserts = 0;
  }

  // ------------------------------------------------------- attention mass
  // Per segment and logical token: the softmax probability the token's entry
  // receives, summed over the segment's query rows and heads, from the Q and
  // the lse of a finished attention pass ([AKV-blog] "Dilemma 1").
  void attention_mass(int32_t layer, const akv_segment* segs, int32_t n_segs, const void* q, int64_t n_q_rows,
                      const float* lse, float scale, float* mass, cudaStream_t st) {
    if (n_segs < 0 || (n_segs > 0 && !segs)) fail(AKV_ERR_ARG, "bad segment list");
    if (layer < 0 || layer >= cfg.n_layers) fail(AKV_ERR_RANGE, "layer outside the pools");
    if (n_q_rows < 0 || n_q_rows > kI32Max) fail(AKV_ERR_RANGE, "bad query row count");
    if (cfg.layout != AKV_LAYOUT_GQA) fail(AKV_ERR_ARG, "attention mass is implemented for the GQA layout");
    if (!meta && n_segs > 0 && (!q || !lse || !mass)) fail(AKV_ERR_ARG, "null Q, lse or mass pointer");
    for (int32_t i = 0; i < n_segs; ++i) validate_segment(segs[i], n_q_rows);
    std::vector<int32_t> ids;
    for (int32_t i = 0; i < n_segs; ++i) ids.push_back(segs[i].seq);
    std::sort(ids.begin(), ids.end());
    ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
    flush(ids, st);
    if (n_segs == 0) return;
    const int G = cfg.n_q_heads / cfg.n_kv_heads, tpt = 128 / G, rpt = 128 / cfg.page_size;
    std::vector<akv::AttnRun> runs;
    std::vector<akv::AttnSeg> tab;
    std::vector<akv::AttnWork> work;
    std::vector<int32_t> ent_tok;
    int64_t mass_len = 0;
    double flops = 0.0;  // QK^T and the column-sum product (ones(128 x 128) P) over the visible pairs
    for (int32_t i = 0; i < n_segs; ++i) {
      SegPlan sp = plan_segment(segs[i], false, true);
      akv::AttnSeg sg{};
      sg.run_off = int32_t(runs.size());
      sg.n_runs = int32_t(sp.runs.size());
      sg.kv_len = int32_t(sp.kv_len);
      sg.q_len = segs[i].q_len;
      sg.q_row0 = int32_t(segs[i].q_row0);
      sg.ent_off = int32_t(ent_tok.size());
      sg.mass_off = int32_t(mass_len);
      if (mass_len + segs[i].kv_end > kI32Max) fail(AKV_ERR_RANGE, "mass output too long");
      mass_len += segs[i].kv_end;
      const int64_t ql = sg.q_len, kl = sg.kv_len;
      flops += double(cfg.n_q_heads) * 2.0 * (cfg.d_rot + 128) * double(ql * (kl - ql) + ql * (ql + 1) / 2);
      const int n_qt = int((ql + tpt - 1) / tpt);
      // KV tiles query tile qt reads: runs whose first entry is <= its last row's limit
      auto tiles_of = [&](int qt) -> int32_t {
        if (qt >= n_qt) return 0;
        const int64_t limit = kl - ql + std::min<int64_t>(ql, int64_t(qt + 1) * tpt) - 1;
        int64_t lo_r = 0, hi_r = int64_t(sp.runs.size());
        while (lo_r < hi_r) {
          const int64_t mid = (lo_r + hi_r) / 2;
          if (sp.runs[mid].es <= limit) lo_r = mid + 1; else hi_r = mid;
        }
        return int32_t((lo_r + rpt - 1) / rpt);
      };
      // one item per pair of query tiles (the second absent: n_b = 0) and kv head
      for (int qt = 0; qt < n_qt; qt += 2) {
        const int32_t na = tiles_of(qt), nb = tiles_of(qt + 1);
        for (int h = 0; h < cfg.n_kv_heads; ++h)
          work.push_back(akv::AttnWork{i, h, qt, na, nb, 0, std::max(na, nb), -1, -1});
      }
      runs.insert(runs.end(), sp.runs.begin(), sp.runs.end());
      ent_tok.insert(ent_tok.end(), sp.tok.begin(), sp.tok.end());
      tab.push_back(sg);
    }
    plan_mass_split(work);
    if (meta) return;
    if (!(cfg.d_rot == 64 || cfg.d_rot == 128)) fail(AKV_ERR_ARG, "attention mass supports head_dim 64 or 128");
    const size_t qbytes = size_t(n_q_rows) * cfg.n_q_heads * cfg.d_rot * 2;
    const void* qd = device_input(q, qbytes, st_q, st);
    const float* lsed = static_cast<const float*>(device_input(lse, size_t(n_q_rows) * cfg.n_q_heads * 4, st_lse, st));
    if (reinterpret_cast<uintptr_t>(qd) % 16) fail(AKV_ERR_ARG, "Q must be 16-byte aligned");
    const bool m_host = !is_device_ptr(mass);
    float* md = mass;
    if (m_host) {
      st_o.want_host = false;
      st_o.acquire(size_t(mass_len) * 4);
      md = static_cast<float*>(st_o.dev);
    }
    cuda_check(cudaMemsetAsync(md, 0, size_t(mass_len) * 4, st), "mass zeroing");
    akv::MassParams p{};
    {
      const uint64_t dims[3] = {uint64_t(cfg.d_rot), uint64_t(cfg.n_q_heads), uint64_t(std::max<int64_t>(n_q_rows, 1))};
      const uint64_t strides[2] = {uint64_t(cfg.d_rot) * 2, uint64_t(cfg.n_q_heads) * cfg.d_rot * 2};
      const uint32_t box[3] = {64, uint32_t(G), uint32_t(tpt)};
      encode_map(&p.q_map, const_cast<void*>(qd), 3, dims, strides, box);
    }
    p.k_map = k_map;
    p.k_tile_map = k_tile_map;
    void *druns = nullptr, *dsegs = nullptr, *dwork = nullptr, *dtok = nullptr;
    up.upload({{runs.data(), runs.size() * sizeof(akv::AttnRun), &druns},
               {tab.data(), tab.size() * sizeof(akv::AttnSeg), &dsegs},
               {work.data(), work.size() * sizeof(akv::AttnWork), &dwork},
               {ent_tok.data(), ent_tok.size() * sizeof(int32_t), &dtok}},
              st);
    p.runs = static_cast<akv::AttnRun*>(druns);
    p.segs = static_cast<akv::AttnSeg*>(dsegs);
    p.work = static_cast<akv::AttnWork*>(dwork);
    p.ent_tok = static_cast<const int32_t*>(dtok);
    p.lse = lsed;
    p.mass = md;
    p.err = dev_err;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.n_work = int32_t(work.size());
    p.n_segs = int32_t(tab.size());
    p.n_runs = int32_t(runs.size());
    p.n_q_rows = int32_t(n_q_rows);
    p.layer = layer;
    p.n_pages = cfg.n_pages;
    p.hq = cfg.n_q_heads;
    p.group = G;
    p.page = cfg.page_size;
    Timed t;
    begin_timed(kMass, 0.0, flops, st, t, 1);
    cuda_check(akv::launch_attn_mass(p, cfg.d_rot, st), "attn_mass launch");
    end_timed(t, st);
    up.done(st);
    if (st_q.dev && !is_device_ptr(q)) st_q.release(st);
    if (st_lse.dev && !is_device_ptr(lse)) st_lse.release(st);
    if (m_host) {
      const cudaStream_t ost = output_stream(st);
      cuda_check(cudaMemcpyAsync(mass, md, size_t(mass_len) * 4, cudaMemcpyDeviceToHost, ost), "mass copy to host");
      st_o.release(ost);
    }
  }

  // ------------------------------------------------------------ lifecycle  // ------------------------------------------------------------ lifecycle
  void create(const akv_config& c, const akv_pools* pools) {
    cfg = c;
    if (c.n_layers <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.n_pages <= 0 || c.reserved != 0)
      fail(AKV_ERR_ARG, "bad config sizes");
    if (c.page_size != 16 && c.page_size != 32 && c.page_size != 64 && c.page_size != 128)
      fail(AKV_ERR_ARG, "page_size must be 16, 32, 64 or 128");
    if (c.d_rot <= 0 || c.d_rot % 8 || c.d_v <= 0 || c.d_v % 8) fail(AKV_ERR_ARG, "d_rot and d_v must be multiples of 8");
    if (c.n_q_heads % c.n_kv_heads) fail(AKV_ERR_ARG, "n_q_heads must be a multiple of n_kv_heads");
    const int G = c.n_q_heads / c.n_kv_heads;
    if (G > 128 || 128 % G) fail(AKV_ERR_ARG, "n_q_heads / n_kv_heads must divide 128");
    if (c.layout != AKV_LAYOUT_GQA && c.layout != AKV_LAYOUT_MLA) fail(AKV_ERR_ARG, "bad layout");
    if (c.layout == AKV_LAYOUT_MLA && c.n_kv_heads != 1) fail(AKV_ERR_ARG, "MLA needs n_kv_heads = 1");
    if (c.layout == AKV_LAYOUT_GQA && c.d_v != c.d_rot) fail(AKV_ERR_ARG, "GQA needs d_v = d_rot");
    if (c.rope_layout != AKV_ROPE_INTERLEAVED && c.rope_layout != AKV_ROPE_HALF) fail(AKV_ERR_ARG, "bad rope layout");
    if (c.rope_layout == AKV_ROPE_HALF && c.d_rot % 16) fail(AKV_ERR_ARG, "half layout needs d_rot % 16 == 0");
    if (!(c.rope_base > 0.0)) fail(AKV_ERR_ARG, "rope_base must be positive");
    if (int64_t(c.n_pages) * c.page_size > kI32Max) fail(AKV_ERR_ARG, "pool too large for int32 rows");
    K.init(c.n_pages);
    V.init(c.n_pages);
    mk.init(c.n_pages);
    mv.init(c.n_pages);
    page_dst.assign(c.n_pages, -1);
    sim_rc.assign(c.n_pages, 0);
    if (!pools) {
      meta = true;
      return;
    }
    if (!pools->k_pool || !pools->v_pool) fail(AKV_ERR_ARG, "null pool pointer");
    if (reinterpret_cast<uintptr_t>(pools->k_pool) % 16 || reinterpret_cast<uintptr_t>(pools->v_pool) % 16)
      fail(AKV_ERR_ARG, "pools must be 16-byte aligned");
    kpool = pools->k_pool;
    vpool = pools->v_pool;
    cuda_check(cudaGetDevice(&device), "cudaGetDevice");
    cuda_check(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, device), "cudaDeviceGetAttribute");
    cuda_check(cudaMalloc(&dev_err, sizeof(akv::DevErr)), "cudaMalloc");
    cuda_check(cudaMemset(dev_err, 0, sizeof(akv::DevErr)), "cudaMemset");
    cuda_check(cudaStreamCreateWithFlags(&copy_st, cudaStreamNonBlocking), "cudaStreamCreate");
    up.copy_stream = copy_st;
    if (c.d_rot % 64 == 0 && c.d_v % 64 == 0) {
      const uint64_t lp = uint64_t(c.n_layers) * c.n_pages;
      const uint32_t box[4] = {64, uint32_t(c.page_size), 1, 1};
      const uint64_t kd[4] = {uint64_t(c.d_rot), uint64_t(c.page_size), uint64_t(c.n_kv_heads), lp};
      const uint64_t ks[3] = {uint64_t(c.d_rot) * 2, uint64_t(c.page_size) * c.d_rot * 2,
                              uint64_t(c.n_kv_heads) * c.page_size * c.d_rot * 2};
      encode_map(&k_map, kpool, 4, kd, ks, box);
      const uint64_t vd[4] = {uint64_t(c.d_v), uint64_t(c.page_size), uint64_t(c.n_kv_heads), lp};
      const uint64_t vs[3] = {uint64_t(c.d_v) * 2, uint64_t(c.page_size) * c.d_v * 2,
                              uint64_t(c.n_kv_heads) * c.page_size * c.d_v * 2};
      encode_map(&v_map, vpool, 4, vd, vs, box);
      // GQA loads a 128-key tile's consecutive pages at once, MLA a 64-key unit
      // (a 128-slot page is then two units).
      const bool mla_units = c.layout == AKV_LAYOUT_MLA;
      const uint32_t tbox[4] = {64, uint32_t(mla_units ? std::min(c.page_size, 64) : c.page_size), 1,
                                uint32_t(mla_units ? std::max(1, 64 / c.page_size) : 128 / c.page_size)};
      encode_map(&k_tile_map, kpool, 4, kd, ks, tbox);
      encode_map(&v_tile_map, vpool, 4, vd, vs, tbox);
      maps_ok = true;
    }
    if (c.layout == AKV_LAYOUT_MLA) {
      mla_slots = akv::segment_attn_mla_slots();
      if (mla_slots <= 0) mla_slots = n_sm & ~1;
    }
  }

  void destroy() {
    if (meta) return;
    cudaDeviceSynchronize();
    up.destroy();
    st_k.destroy();
    st_v.destroy();
    st_q.destroy();
    st_o.destroy();
    st_lse.destroy();
    if (out_ready) {
      cudaEventDestroy(out_ready);
      out_ready = nullptr;
    }
    partial.destroy();
    for (auto& t : timed) {
      cudaEventDestroy(t.a);
      cudaEventDestroy(t.b);
    }
    for (auto e : ev_pool) cudaEventDestroy(e);
    if (copy_st) cudaStreamDestroy(copy_st);
    if (dev_err) cudaFree(dev_err);
  }
};

namespace {

template <typename F>
akv_status guard(akv_ctx* ctx, F&& f) {
  if (!ctx) return AKV_ERR_ARG;
  try {
    ctx->err.clear();
    f();
    return AKV_OK;
  } catch (const Fail& e) {
    ctx->err = e.msg;
    return e.st;
  } catch (const std::bad_alloc&) {
    ctx->err = "host out of memory";
    return AKV_ERR_NO_PAGES;
  } catch (...) {
    ctx->err = "internal error";
    return AKV_ERR_ARG;
  }
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

akv_status akv_create(const akv_config* cfg, const akv_pools* pools, akv_ctx** out) {
  if (!cfg || !out) return AKV_ERR_ARG;
  *out = nullptr;
  akv_ctx* ctx = new (std::nothrow) akv_ctx();
  if (!ctx) return AKV_ERR_ARG;
  akv_status s = guard(ctx, [&] { ctx->create(*cfg, pools); });
  if (s != AKV_OK) {
    ctx->destroy();
    delete ctx;
    return s;
  }
  *out = ctx;
  return AKV_OK;
}

akv_status akv_destroy(akv_ctx* ctx) {
  if (!ctx) return AKV_ERR_ARG;
  ctx->destroy();
  delete ctx;
  return AKV_OK;
}

const char* akv_last_error(const akv_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

akv_status akv_seq_alloc(akv_ctx* ctx, int32_t* seq_out) {
  return guard(ctx, [&] {
    if (!seq_out) fail(AKV_ERR_ARG, "null output");
    *seq_out = ctx->new_id();
    ctx->seqs[*seq_out].clear();
  });
}

akv_status akv_seq_fork(akv_ctx* ctx, int32_t src, int64_t n_prefix, int32_t* seq_out) {
  return guard(ctx, [&] {
    if (!seq_out) fail(AKV_ERR_ARG, "null output");
    ctx->fork(src, n_prefix, seq_out);
  });
}

akv_status akv_seq_free(akv_ctx* ctx, int32_t seq) {
  return guard(ctx, [&] { ctx->free_seq(seq); });
}

akv_status akv_seq_len(akv_ctx* ctx, int32_t seq, int64_t* n_out) {
  return guard(ctx, [&] {
    if (!n_out) fail(AKV_ERR_ARG, "null output");
    *n_out = int64_t(ctx->seq_raw(seq).size());
  });
}

akv_status akv_append(akv_ctx* ctx, int32_t seq, int64_t n, const void* k, const void* v, const int32_t* pos,
                      void* stream) {
  return guard(ctx, [&] { ctx->append(seq, n, k, v, pos, as_stream(stream)); });
}

akv_status akv_drop(akv_ctx* ctx, int32_t seq, int64_t s, int64_t e) {
  return guard(ctx, [&] { ctx->drop(seq, s, e); });
}

akv_status akv_repos(akv_ctx* ctx, int32_t seq, int64_t s, int64_t e, int32_t delta) {
  return guard(ctx, [&] { ctx->repos(seq, s, e, delta); });
}

akv_status akv_edit(akv_ctx* ctx, int32_t seq, const akv_edit_op* ops, int32_t n_ops) {
  return guard(ctx, [&] { ctx->edit(seq, ops, n_ops); });
}

akv_status akv_splice(akv_ctx* ctx, int32_t seq, int64_t s, int64_t e, int64_t n_stub, const void* k_stub,
                      const void* v_stub, const int32_t* pos, void* stream) {
  return guard(ctx, [&] { ctx->splice(seq, s, e, n_stub, k_stub, v_stub, pos, as_stream(stream)); });
}

akv_status akv_flush(akv_ctx* ctx, int32_t seq, void* stream) {
  return guard(ctx, [&] {
    std::vector<int32_t> ids;
    if (seq == -1) {
      for (int32_t i = 0; i < int32_t(ctx->seqs.size()); ++i)
        if (ctx->live[i]) ids.push_back(i);
    } else {
      ctx->seq(seq);
      ids.push_back(seq);
    }
    ctx->flush(ids, as_stream(stream));
  });
}

akv_status akv_attend(akv_ctx* ctx, int32_t layer, const akv_segment* segs, int32_t n_segs, const void* q,
                      int64_t n_q_rows, void* o, float* lse, float scale, void* stream) {
  return guard(ctx, [&] { ctx->attend(layer, segs, n_segs, q, n_q_rows, o, lse, scale, as_stream(stream)); });
}

akv_status akv_tree_insert(akv_ctx* ctx, const akv_item* items, int64_t n, int32_t seq, int32_t* tree_seq_out) {
  return guard(ctx, [&] {
    const int32_t t = ctx->tree_insert(items, n, seq);
    if (tree_seq_out) *tree_seq_out = t;
  });
}

akv_status akv_tree_match(akv_ctx* ctx, const akv_item* items, int64_t n, akv_match* out) {
  return guard(ctx, [&] {
    if (!out) fail(AKV_ERR_ARG, "null output");
    *out = ctx->tree_match(items, n);
  });
}

akv_status akv_tree_reuse(akv_ctx* ctx, const akv_item* items, int64_t n, akv_match* out, int32_t* seq_out,
                          void* stream) {
  return guard(ctx, [&] {
    if (!seq_out) fail(AKV_ERR_ARG, "null output");
    *seq_out = ctx->tree_reuse(items, n, out, as_stream(stream));
  });
}

akv_status akv_tree_clear(akv_ctx* ctx) {
  return guard(ctx, [&] { ctx->tree_clear(); });
}

akv_status akv_fragmentation(akv_ctx* ctx, int32_t seq, double* frac_out) {
  return guard(ctx, [&] {
    if (!frac_out) fail(AKV_ERR_ARG, "null output");
    *frac_out = ctx->fragmentation(seq);
  });
}

akv_status akv_compact(akv_ctx* ctx, int32_t seq, void* stream) {
  return guard(ctx, [&] { ctx->compact(seq, as_stream(stream)); });
}

akv_status akv_attention_mass(akv_ctx* ctx, int32_t layer, const akv_segment* segs, int32_t n_segs, const void* q,
                              int64_t n_q_rows, const float* lse, float scale, float* mass, void* stream) {
  return guard(ctx, [&] { ctx->attention_mass(layer, segs, n_segs, q, n_q_rows, lse, scale, mass, as_stream(stream)); });
}

akv_status akv_attend_fused(akv_ctx* ctx, int32_t layer, const akv_segment* segs, int32_t n_segs, const void* q,
                            int64_t n_q_rows, void* o, float* lse, float scale, void* stream) {
  return guard(ctx, [&] { ctx->attend(layer, segs, n_segs, q, n_q_rows, o, lse, scale, as_stream(stream), true); });
}

akv_status akv_debug_rotate_f32(akv_ctx* ctx, const int32_t* runs, int32_t n_runs, float* out, void* stream) {
  return guard(ctx, [&] { ctx->debug_rotate_f32(runs, n_runs, out, as_stream(stream)); });
}

akv_status akv_export_state(akv_ctx* ctx, int32_t seq, int32_t* k_page, int32_t* v_page, int32_t* slot,
                            int32_t* pos, int32_t* delta, uint8_t* visible) {
  return guard(ctx, [&] {
    const auto& toks = ctx->seq(seq);
    for (size_t i = 0; i < toks.size(); ++i) {
      if (k_page) k_page[i] = toks[i].kp;
      if (v_page) v_page[i] = toks[i].vp;
      if (slot) slot[i] = toks[i].slot;
      if (pos) pos[i] = toks[i].pos;
      if (delta) delta[i] = toks[i].delta;
      if (visible) visible[i] = toks[i].vis;
    }
  });
}

akv_status akv_refcounts(akv_ctx* ctx, int32_t* k_rc, int32_t* v_rc) {
  return guard(ctx, [&] {
    if (k_rc) std::memcpy(k_rc, ctx->K.counts().data(), ctx->K.counts().size() * 4);
    if (v_rc) std::memcpy(v_rc, ctx->V.counts().data(), ctx->V.counts().size() * 4);
  });
}

akv_status akv_last_flush_runs(akv_ctx* ctx, int32_t* out, int64_t cap, int64_t* n_runs) {
  return guard(ctx, [&] {
    const int64_t n = int64_t(ctx->last_runs.size() / 5);
    if (n_runs) *n_runs = n;
    if (out && cap > 0) std::memcpy(out, ctx->last_runs.data(), size_t(std::min(n, cap)) * 5 * 4);
  });
}

akv_status akv_segment_runs(akv_ctx* ctx, const akv_segment* seg, int32_t* out, int64_t cap, int64_t* n_runs,
                            int64_t* kv_len) {
  return guard(ctx, [&] {
    if (!seg) fail(AKV_ERR_ARG, "null segment");
    ctx->validate_segment(*seg, -1);
    auto sp = ctx->plan_segment(*seg);
    if (n_runs) *n_runs = int64_t(sp.runs.size());
    if (kv_len) *kv_len = sp.kv_len;
    for (int64_t i = 0; out && i < std::min<int64_t>(cap, int64_t(sp.runs.size())); ++i) {
      const auto& r = sp.runs[i];
      out[4 * i + 0] = r.kp;
      out[4 * i + 1] = r.vp;
      out[4 * i + 2] = r.lohi & 0xffff;
      out[4 * i + 3] = r.lohi >> 16;
    }
  });
}

akv_status akv_check_device_error(akv_ctx* ctx, void* stream, int32_t* code) {
  akv_status inner = AKV_OK;
  akv_status s = guard(ctx, [&] {
    int32_t c = 0;
    if (!ctx->meta) {
      akv::DevErr e{};
      cuda_check(cudaStreamSynchronize(as_stream(stream)), "cudaStreamSynchronize");
      cuda_check(cudaMemcpy(&e, ctx->dev_err, sizeof e, cudaMemcpyDeviceToHost), "error word read");
      cuda_check(cudaMemset(ctx->dev_err, 0, sizeof e), "error word clear");
      c = e.code;
      if (c) {
        char buf[160];
        snprintf(buf, sizeof buf, "device error %d (info %d %d %d)", e.code, e.info[0], e.info[1], e.info[2]);
        ctx->err = buf;
      }
    }
    if (code) *code = c;
    inner = akv_status(c);
  });
  return s != AKV_OK ? s : inner;
}

akv_status akv_set_attention_split(akv_ctx* ctx, int32_t split) {
  return guard(ctx, [&] {
    if (split < 0 || split > 8) fail(AKV_ERR_ARG, "split must be 0 (automatic) or 1..8");
    ctx->split_override = split;
  });
}

akv_status akv_debug_wait_limit(akv_ctx* ctx, uint64_t wait_ns, int32_t load_cap) {
  return guard(ctx, [&] {
    if (load_cap < -1) fail(AKV_ERR_ARG, "load_cap must be -1 (no cap) or >= 0");
    ctx->wait_ns = wait_ns ? wait_ns : 4000000000ull;
    ctx->load_cap = load_cap;
  });
}

akv_status akv_last_attention_plan(akv_ctx* ctx, int32_t* units, int64_t cap, int64_t* n_units, int32_t* cta_units,
                                   int64_t cta_cap, int64_t* n_cta, int32_t n_sm) {
  return guard(ctx, [&] {
    if (!ctx->meta) fail(AKV_ERR_ARG, "the plan is kept by metadata-only contexts");
    if (n_sm > 0) {  // the device size later plans assume
      ctx->n_sm = n_sm;
      ctx->mla_slots = n_sm & ~1;
    }
    const int64_t n = int64_t(ctx->last_work.size());
    if (n_units) *n_units = n;
    for (int64_t i = 0; i < std::min(n, cap) && units; ++i) {
      const akv::AttnWork& w = ctx->last_work[size_t(i)];
      const int32_t row[9] = {w.seg, w.kvh, w.qt0, w.n_a, w.n_b, w.t0, w.t1, w.part, w.comb};
      std::memcpy(units + 9 * i, row, sizeof row);
    }
    const int64_t nc = ctx->last_cta_units.empty() ? 0 : int64_t(ctx->last_cta_units.size()) - 1;
    if (n_cta) *n_cta = nc;
    for (int64_t i = 0; i <= nc && i < cta_cap && cta_units; ++i) cta_units[i] = ctx->last_cta_units[size_t(i)];
  });
}

akv_status akv_set_output_stream(akv_ctx* ctx, void* stream) {
  return guard(ctx, [&] { ctx->out_st = static_cast<cudaStream_t>(stream); });
}

akv_status akv_debug_corrupt(akv_ctx* ctx, int32_t what) {
  return guard(ctx, [&] {
#ifdef AKV_CHECKED
    if (what < 0 || what > 2) fail(AKV_ERR_ARG, "what must be 0, 1 (flush) or 2 (attend)");
    ctx->corrupt_next = what;
#else
    (void)what;
    fail(AKV_ERR_ARG, "descriptor corruption needs the checked build (libakv_checked.so)");
#endif
  });
}

akv_status akv_profile_enable(akv_ctx* ctx, int32_t on) {
  return guard(ctx, [&] {
    if (ctx->meta) return;
    ctx->collect();
    ctx->stats = akv_kernel_stats{};
    ctx->prof = on != 0;
  });
}

akv_status akv_profile_read(akv_ctx* ctx, akv_kernel_stats* out) {
  return guard(ctx, [&] {
    if (!out) fail(AKV_ERR_ARG, "null output");
    if (!ctx->meta) ctx->collect();
    *out = ctx->stats;
  });
}

}  // extern "C"
