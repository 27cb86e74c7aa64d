"""ctypes binding of libakv.so (include/akv.h): argument marshalling only.

Every computation runs in the library: the host bookkeeping in its C++ engine
and every step of the data path in its CUDA kernels.  Tensors are passed as
raw pointers (``tensor.data_ptr()``); torch only provides device memory and
streams.  There is no fallback: if the library is missing, loading fails.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# AKV_CHECKED=1 selects the build with device-side descriptor checks (see build.py)
LIB_PATH = os.path.join(_HERE, "libakv_checked.so" if os.environ.get("AKV_CHECKED", "") == "1" else "libakv.so")

OK, ERR_ARG, ERR_RANGE, ERR_NO_PAGES, ERR_OVERFLOW, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_DEVICE = 0, 1, 2, 4, 5, 6, 7, 8
STATUS_NAMES = {0: "OK", 1: "ARG", 2: "RANGE", 4: "NO_PAGES", 5: "OVERFLOW", 6: "CUDA", 7: "DEVICE_TIMEOUT",
                8: "DEVICE"}
LAYOUT_GQA, LAYOUT_MLA = 0, 1
ROPE_INTERLEAVED, ROPE_HALF = 0, 1


class AKVError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status
        self.code = STATUS_NAMES.get(status, str(status))


EDIT_DROP, EDIT_REPOS = 1, 2


class EditOp(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("delta", ctypes.c_int32), ("s", ctypes.c_int64), ("e", ctypes.c_int64)]


class Config(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("d_rot", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("n_pages", ctypes.c_int32), ("rope_layout", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("rope_base", ctypes.c_double)]


class Pools(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p)]


class Segment(ctypes.Structure):
    _fields_ = [("seq", ctypes.c_int32), ("q_len", ctypes.c_int32), ("kv_end", ctypes.c_int64),
                ("q_row0", ctypes.c_int64), ("hide", ctypes.POINTER(ctypes.c_int64)), ("n_hide", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class Match(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("seq", ctypes.c_int32), ("n_items", ctypes.c_int64),
                ("n_tokens", ctypes.c_int64)]


MATCH_KINDS = {0: "none", 1: "exact", 2: "retrigger"}


def items_array(items):
    """Path items as int32 [n, 4] (kind, a, b, c): ("tok", x, p) -> (0, x, p, 0); ("op", code, a, b, c)
    -> (code, a, b, c)."""
    rows = []
    for it in items:
        if it[0] == "tok":
            rows.append((0, it[1], it[2], 0))
        else:
            rows.append((it[1], it[2], it[3], it[4]))
    return np.ascontiguousarray(np.asarray(rows, np.int32).reshape(-1, 4))


class KernelStats(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * 5), ("ms", ctypes.c_double * 5), ("bytes", ctypes.c_double * 5),
                ("flops", ctypes.c_double * 5)]


KERNEL_NAMES = ("kv_write", "repos_rotate", "segment_attn", "compact_copy", "attn_mass")

_lib = None


def load(path=LIB_PATH):
    """Load libakv.so (build it first with agentic_kv_cache_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m agentic_kv_cache_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I32, I64, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    pi32, pi64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
    sig = {
        "akv_create": [ctypes.POINTER(Config), ctypes.POINTER(Pools), ctypes.POINTER(P)],
        "akv_destroy": [P],
        "akv_seq_alloc": [P, pi32],
        "akv_seq_fork": [P, I32, I64, pi32],
        "akv_seq_free": [P, I32],
        "akv_seq_len": [P, I32, pi64],
        "akv_append": [P, I32, I64, P, P, P, P],
        "akv_drop": [P, I32, I64, I64],
        "akv_repos": [P, I32, I64, I64, I32],
        "akv_edit": [P, I32, ctypes.POINTER(EditOp), I32],
        "akv_splice": [P, I32, I64, I64, I64, P, P, P, P],
        "akv_flush": [P, I32, P],
        "akv_attend": [P, I32, ctypes.POINTER(Segment), I32, P, I64, P, P, F32, P],
        "akv_attend_fused": [P, I32, ctypes.POINTER(Segment), I32, P, I64, P, P, F32, P],
        "akv_fragmentation": [P, I32, ctypes.POINTER(ctypes.c_double)],
        "akv_tree_insert": [P, P, I64, I32, pi32],
        "akv_tree_match": [P, P, I64, ctypes.POINTER(Match)],
        "akv_tree_reuse": [P, P, I64, ctypes.POINTER(Match), pi32, P],
        "akv_tree_clear": [P],
        "akv_attention_mass": [P, I32, ctypes.POINTER(Segment), I32, P, I64, P, F32, P, P],
        "akv_compact": [P, I32, P],
        "akv_debug_rotate_f32": [P, P, I32, P, P],
        "akv_export_state": [P, I32, P, P, P, P, P, P],
        "akv_refcounts": [P, P, P],
        "akv_last_flush_runs": [P, P, I64, pi64],
        "akv_segment_runs": [P, ctypes.POINTER(Segment), P, I64, pi64, pi64],
        "akv_check_device_error": [P, P, pi32],
        "akv_profile_enable": [P, I32],
        "akv_set_attention_split": [P, I32],
        "akv_debug_wait_limit": [P, ctypes.c_uint64, I32],
        "akv_debug_corrupt": [P, I32],
        "akv_set_output_stream": [P, P],
        "akv_last_attention_plan": [P, P, I64, pi64, P, I64, pi64, I32],
        "akv_profile_read": [P, ctypes.POINTER(KernelStats)],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.akv_repos_rotate_noalloc.argtypes = [P, I32, I32, I32, I32, I32, I32, ctypes.c_double, P, I32, P]
    lib.akv_repos_rotate_noalloc.restype = ctypes.c_int
    lib.akv_last_error.argtypes = [P]
    lib.akv_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x):
    """Raw address of a torch tensor / numpy array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _i32_array(x, n):
    if x is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.int32))
    if a.size != n:
        raise ValueError("position array has the wrong length")
    return a, a.ctypes.data


class Engine:
    """One akv_ctx.  cfg: dict of akv_config fields; pools: (k_pool, v_pool) or None (metadata only)."""

    def __init__(self, cfg, pools=None):
        self.lib = load()
        self.cfg = Config(**{k: cfg[k] for k in ("layout", "n_layers", "n_q_heads", "n_kv_heads", "d_rot", "d_v",
                                                  "page_size", "n_pages", "rope_layout")},
                          reserved=0, rope_base=float(cfg["rope_base"]))
        self._pools = pools  # keep the tensors alive
        pp = None if pools is None else ctypes.byref(Pools(_ptr(pools[0]), _ptr(pools[1])))
        h = ctypes.c_void_p()
        st = self.lib.akv_create(ctypes.byref(self.cfg), pp, ctypes.byref(h))
        if st != OK:
            raise AKVError(st, "akv_create failed")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            self.lib.akv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st):
        if st != OK:
            raise AKVError(st, self.lib.akv_last_error(self.h).decode())

    # ------------------------------------------------------------ sequences
    def seq_alloc(self):
        out = ctypes.c_int32()
        self._check(self.lib.akv_seq_alloc(self.h, ctypes.byref(out)))
        return out.value

    def seq_fork(self, src, n_prefix):
        out = ctypes.c_int32()
        self._check(self.lib.akv_seq_fork(self.h, src, n_prefix, ctypes.byref(out)))
        return out.value

    def seq_free(self, seq):
        self._check(self.lib.akv_seq_free(self.h, seq))

    def seq_len(self, seq):
        out = ctypes.c_int64()
        self._check(self.lib.akv_seq_len(self.h, seq, ctypes.byref(out)))
        return out.value

    # ----------------------------------------------------------- operations
    def append(self, seq, n, k=None, v=None, pos=None, stream=None):
        keep, pp = _i32_array(pos, n)
        self._check(self.lib.akv_append(self.h, seq, n, _ptr(k), _ptr(v), pp, _stream(stream)))

    def drop(self, seq, s, e):
        self._check(self.lib.akv_drop(self.h, seq, s, e))

    def repos(self, seq, s, e, delta):
        self._check(self.lib.akv_repos(self.h, seq, s, e, delta))

    def edit(self, seq, ops):
        """A list of ("drop", s, e) / ("repos", s, e, delta) directives in one call, all or nothing."""
        arr = (EditOp * max(len(ops), 1))()
        for i, op in enumerate(ops):
            if op[0] == "drop":
                arr[i] = EditOp(EDIT_DROP, 0, op[1], op[2])
            elif op[0] == "repos":
                arr[i] = EditOp(EDIT_REPOS, op[3], op[1], op[2])
            else:
                arr[i] = EditOp(0, 0, op[1], op[2])  # rejected by the library
        self._check(self.lib.akv_edit(self.h, seq, arr, len(ops)))

    def splice(self, seq, s, e, n_stub, k=None, v=None, pos=None, stream=None):
        keep, pp = _i32_array(pos, n_stub)
        self._check(self.lib.akv_splice(self.h, seq, s, e, n_stub, _ptr(k), _ptr(v), pp, _stream(stream)))

    def flush(self, seq=-1, stream=None):
        self._check(self.lib.akv_flush(self.h, seq, _stream(stream)))

    @staticmethod
    def make_segments(segs):
        arr = (Segment * max(len(segs), 1))()
        keep = []
        for i, s in enumerate(segs):
            hide = np.ascontiguousarray(np.asarray(s.get("hide", []), dtype=np.int64).reshape(-1))
            keep.append(hide)
            arr[i].seq = s["seq"]
            arr[i].q_len = s["q_len"]
            arr[i].kv_end = s["kv_end"]
            arr[i].q_row0 = s.get("q_row0", 0)
            arr[i].hide = hide.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if hide.size else None
            arr[i].n_hide = hide.size // 2
            arr[i].reserved = 0
        return arr, keep

    def attention_mass(self, layer, segs, q, n_q_rows, lse, mass, scale=1.0, stream=None):
        """akv_attention_mass: mass [sum of kv_end] per segment and logical token (see include/akv.h)."""
        arr, keep = self.make_segments(segs)
        self._check(self.lib.akv_attention_mass(self.h, layer, arr, len(segs), _ptr(q), n_q_rows, _ptr(lse),
                                                float(scale), _ptr(mass), _stream(stream)))

    # --------------------------------------------------------- radix tree
    def tree_insert(self, items, seq):
        a = items_array(items)
        out = ctypes.c_int32()
        self._check(self.lib.akv_tree_insert(self.h, a.ctypes.data, a.shape[0], seq, ctypes.byref(out)))
        return out.value

    @staticmethod
    def _match(m):
        return dict(kind=MATCH_KINDS[m.kind], seq=m.seq, n_items=m.n_items, n_tokens=m.n_tokens)

    def tree_match(self, items):
        a = items_array(items)
        m = Match()
        self._check(self.lib.akv_tree_match(self.h, a.ctypes.data, a.shape[0], ctypes.byref(m)))
        return self._match(m)

    def tree_reuse(self, items, stream=None):
        a = items_array(items)
        m = Match()
        sid = ctypes.c_int32()
        self._check(self.lib.akv_tree_reuse(self.h, a.ctypes.data, a.shape[0], ctypes.byref(m), ctypes.byref(sid),
                                            _stream(stream)))
        return self._match(m), sid.value

    def tree_clear(self):
        self._check(self.lib.akv_tree_clear(self.h))

    def fragmentation(self, seq):
        out = ctypes.c_double()
        self._check(self.lib.akv_fragmentation(self.h, seq, ctypes.byref(out)))
        return out.value

    def compact(self, seq, stream=None):
        self._check(self.lib.akv_compact(self.h, seq, _stream(stream)))

    def attend(self, layer, segs, q, n_q_rows, o, lse=None, scale=1.0, stream=None, fused=False):
        """akv_attend (flush, then attention), or with fused=True akv_attend_fused (pending shifts
        applied to K inside the attention kernel; nothing is written to the pools)."""
        arr, keep = self.make_segments(segs)
        fn = self.lib.akv_attend_fused if fused else self.lib.akv_attend
        self._check(fn(self.h, layer, arr, len(segs), _ptr(q), n_q_rows, _ptr(o), _ptr(lse), float(scale),
                       _stream(stream)))

    def debug_rotate_f32(self, runs, out, stream=None):
        """runs: int array [n, 4] (K page, lo, hi, delta); out: device float32 tensor
        [n_layers][sum(hi - lo)][n_kv_heads][d_rot]."""
        r = np.ascontiguousarray(np.asarray(runs, dtype=np.int32).reshape(-1, 4))
        self._check(self.lib.akv_debug_rotate_f32(self.h, r.ctypes.data, r.shape[0], _ptr(out), _stream(stream)))

    # ----------------------------------------------------------- inspection
    def export_state(self, seq):
        n = self.seq_len(seq)
        out = {k: np.zeros(n, np.int32) for k in ("k_page", "v_page", "slot", "pos", "delta")}
        vis = np.zeros(n, np.uint8)
        self._check(self.lib.akv_export_state(self.h, seq, *(out[k].ctypes.data for k in
                                                             ("k_page", "v_page", "slot", "pos", "delta")),
                                              vis.ctypes.data))
        out["visible"] = vis.astype(np.int32)
        return out

    def refcounts(self):
        k = np.zeros(self.cfg.n_pages, np.int32)
        v = np.zeros(self.cfg.n_pages, np.int32)
        self._check(self.lib.akv_refcounts(self.h, k.ctypes.data, v.ctypes.data))
        return k, v

    def last_flush_runs(self):
        n = ctypes.c_int64()
        self._check(self.lib.akv_last_flush_runs(self.h, None, 0, ctypes.byref(n)))
        out = np.zeros((max(n.value, 1), 5), np.int32)
        self._check(self.lib.akv_last_flush_runs(self.h, out.ctypes.data, n.value, ctypes.byref(n)))
        return out[:n.value]

    def segment_runs(self, seg):
        arr, keep = self.make_segments([seg])
        n, kv = ctypes.c_int64(), ctypes.c_int64()
        self._check(self.lib.akv_segment_runs(self.h, arr, None, 0, ctypes.byref(n), ctypes.byref(kv)))
        out = np.zeros((max(n.value, 1), 4), np.int32)
        self._check(self.lib.akv_segment_runs(self.h, arr, out.ctypes.data, n.value, ctypes.byref(n),
                                              ctypes.byref(kv)))
        return out[:n.value], kv.value

    # ---------------------------------------------------------------- device
    def check_device_error(self, stream=None):
        code = ctypes.c_int32()
        st = self.lib.akv_check_device_error(self.h, _stream(stream), ctypes.byref(code))
        if st not in (OK, ERR_DEVICE_TIMEOUT, ERR_DEVICE):
            self._check(st)
        return code.value

    def set_attention_split(self, split):
        """0: automatic split-KV; n >= 1: exactly n KV chunks per work item (1 = never split).
        Applies to attend and attention_mass."""
        self._check(self.lib.akv_set_attention_split(self.h, int(split)))

    def last_attention_plan(self, n_sm=0):
        """Metadata-only contexts: (units [n, 9] int32, cta_units int32[n_cta + 1] or empty) of the
        last attend; n_sm > 0 sets the SM count later plans assume."""
        n, nc = ctypes.c_int64(), ctypes.c_int64()
        self._check(self.lib.akv_last_attention_plan(self.h, None, 0, ctypes.byref(n), None, 0, ctypes.byref(nc),
                                                     int(n_sm)))
        units = np.zeros((n.value, 9), np.int32)
        cta = np.zeros((nc.value + 1 if nc.value else 0,), np.int32)
        self._check(self.lib.akv_last_attention_plan(self.h, units.ctypes.data, n.value, ctypes.byref(n),
                                                     cta.ctypes.data if cta.size else None, cta.size,
                                                     ctypes.byref(nc), 0))
        return units, cta

    def set_output_stream(self, stream=None):
        """Copy host results (o, lse, mass) on `stream` (a torch stream or raw handle) after the
        call's kernels, so they overlap later calls; None: on the call's own stream."""
        self._check(self.lib.akv_set_output_stream(self.h, _stream(stream) if stream is not None else None))

    def debug_corrupt(self, what):
        """Checked-build test hook: 1 corrupts the next flush's first run, 2 the next attention
        launch's first run (after host validation); the plain library raises AKVError(ARG)."""
        self._check(self.lib.akv_debug_corrupt(self.h, int(what)))

    def debug_wait_limit(self, wait_ns=0, load_cap=-1):
        """Test hook: limit of the attention kernels' bounded waits (0: the default 4 s) and a cap
        on the K/V tile copies each CTA issues (-1: none)."""
        self._check(self.lib.akv_debug_wait_limit(self.h, int(wait_ns), int(load_cap)))

    def profile_enable(self, on=True):
        self._check(self.lib.akv_profile_enable(self.h, int(on)))

    def profile_read(self):
        s = KernelStats()
        self._check(self.lib.akv_profile_read(self.h, ctypes.byref(s)))
        return {name: dict(launches=s.launches[i], ms=s.ms[i], bytes=s.bytes[i], flops=s.flops[i])
                for i, name in enumerate(KERNEL_NAMES)}


def repos_rotate_noalloc(k_pool, cfg, runs, stream=None):
    """akv_repos_rotate_noalloc: rotate runs [n, 5] (src, dst, lo, hi, delta) of k_pool in the
    library's fixed device scratch array, without a context and without allocating."""
    lib = load()
    r = np.ascontiguousarray(np.asarray(runs, dtype=np.int32).reshape(-1, 5))
    st = lib.akv_repos_rotate_noalloc(_ptr(k_pool), cfg["n_layers"], cfg["n_kv_heads"], cfg["page_size"],
                                      cfg["n_pages"], cfg["d_rot"], cfg["rope_layout"], float(cfg["rope_base"]),
                                      r.ctypes.data, r.shape[0], _stream(stream))
    if st != OK:
        raise AKVError(st, "akv_repos_rotate_noalloc failed")


def config_from_shape(shape, n_pages):
    """akv_config fields for a synth.Shape."""
    return dict(layout=LAYOUT_MLA if shape.mla else LAYOUT_GQA, n_layers=shape.n_layers,
                n_q_heads=shape.n_q_heads, n_kv_heads=shape.n_kv_heads, d_rot=shape.d_rot, d_v=shape.d_v,
                page_size=shape.page_size, n_pages=n_pages,
                rope_layout=ROPE_HALF if shape.rope_layout == "half" else ROPE_INTERLEAVED,
                rope_base=shape.rope_base)


def make_pools(cfg, device="cuda"):
    """Zeroed bf16 pools for a config (torch only allocates here)."""
    import torch
    L, P, H, S = cfg["n_layers"], cfg["n_pages"], cfg["n_kv_heads"], cfg["page_size"]
    k = torch.zeros((L, P, H, S, cfg["d_rot"]), dtype=torch.bfloat16, device=device)
    v = torch.zeros((L, P, H, S, cfg["d_v"]), dtype=torch.bfloat16, device=device)
    return k, v
