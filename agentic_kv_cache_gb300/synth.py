"""Seeded synthetic workloads for tests and benchmarks.

This module only *describes* workloads: model shapes, the order of cache
operations an agent harness issues (append / fork / drop / repos / splice),
the attention segments, and seeded bf16 N(0,1) tensors.  It contains none of
the method's arithmetic (no RoPE, no composition of shifts, no attention); the
engine and the float64 oracle both consume its output.

Workload shapes follow the agent trajectories the pages describe (40-turn
trajectories growing past 64K tokens with large tool outputs; ~17K-token
prompts under MLA) and the model shapes they name (Llama-3.1-8B / 70B KV
heads, DeepSeek-V2-Lite MLA).  The pages' benchmarks (SWE-bench Lite,
WebArena, AgentBench, debug-gym) are not used: synthetic tensors of these
shapes stand in for them.

Operation tuples (sequence operands are symbolic names):
    ("alloc", name)
    ("fork", name, src, n_prefix)
    ("append", name, n, key)            K/V tensors drawn under ``key``
    ("drop", name, s, e)
    ("repos", name, s, e, delta)
    ("splice", name, s, e, n_stub, key) stub K/V drawn under ``key``
    ("flush", name)                     materialise pending shifts now
Segments: dict(seq=name, kv_end, q_len, hide=[(a, b), ...], q_row0).
"""
import dataclasses
import zlib

import numpy as np


@dataclasses.dataclass
class Shape:
    n_layers: int
    n_q_heads: int
    n_kv_heads: int       # 1 under MLA (the latent is shared by all heads)
    d_rot: int            # rotated key part: head_dim (GQA) or K_pe dim (MLA)
    d_v: int              # value / latent width
    rope_base: float
    page_size: int
    mla: bool = False
    rope_layout: str = "interleaved"

    @property
    def d_qk(self):
        return self.d_v + self.d_rot if self.mla else self.d_rot

    @property
    def scale(self):
        # 1/sqrt(d_k); under MLA the DeepSeek qk head dim (128 nope + 64 rope).
        return 1.0 / np.sqrt(192.0 if self.mla else float(self.d_rot))


@dataclasses.dataclass
class Workload:
    name: str
    shape: Shape
    n_pages: int
    ops: list
    segments: list
    seed: int = 0
    meta: dict = dataclasses.field(default_factory=dict)

    @property
    def n_queries(self):
        return sum(s["q_len"] for s in self.segments)


# ----------------------------------------------------------------- tensors
def _rng(seed, key, part):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, zlib.crc32(key.encode()), part])))


def normal_f32(seed, key, part, shape):
    """Seeded N(0,1) float32 array (the caller rounds it to bf16)."""
    return _rng(seed, key, part).standard_normal(shape, dtype=np.float32)


def kv_arrays(w, key, n):
    """(K-part, V-part) float32 for n new tokens: [L][n][H][d_rot], [L][n][H][d_v]."""
    s = w.shape
    k = normal_f32(w.seed, key, 0, (s.n_layers, n, s.n_kv_heads, s.d_rot))
    v = normal_f32(w.seed, key, 1, (s.n_layers, n, s.n_kv_heads, s.d_v))
    return k, v


def q_array(w, layer=0):
    """Queries of every segment of one layer, float32 [n_queries][Hq][d_qk]."""
    s = w.shape
    return normal_f32(w.seed, f"q{layer}", 2, (w.n_queries, s.n_q_heads, s.d_qk))


# --------------------------------------------------------------- helpers
def _split_exact(weights, total):
    """Integers proportional to weights summing exactly to total (largest remainder)."""
    weights = np.asarray(weights, np.float64)
    raw = weights * (total / weights.sum())
    base = np.floor(raw).astype(np.int64)
    rem = int(total - base.sum())
    order = np.argsort(-(raw - base), kind="stable")
    base[order[:rem]] += 1
    return base


def _disjoint_spans(rng, lo, hi, count, min_len, max_len):
    """count non-overlapping sorted spans [s, e) inside [lo, hi)."""
    for _ in range(1000):
        lens = rng.integers(min_len, max_len + 1, size=count)
        slack = (hi - lo) - int(lens.sum())
        if slack < count:
            continue
        gaps = np.sort(rng.choice(slack, size=count, replace=False))
        spans, cur, prev_gap = [], lo, 0
        for g, ln in zip(gaps, lens):
            cur += int(g - prev_gap)
            spans.append((cur, cur + int(ln)))
            cur += int(ln)
            prev_gap = g
        return spans
    raise ValueError("cannot place spans")


# ----------------------------------------------------------- the workloads
def tiny(seed=0):
    """1 layer, 4 query / 1 kv head, d 64, theta 1e4, page 16, 256 cached tokens.

    Branch B (forked, so its repositioned keys are a copy-on-write copy): drop
    [64, 128), repos [128, 256) by -64.  Two segments of 16 new queries in one
    launch: A over the unedited 256 tokens, B over its edited history.
    """
    shape = Shape(1, 4, 1, 64, 64, 1.0e4, 16)
    ops = [
        ("alloc", "A"),
        ("append", "A", 256, "ctx"),
        ("fork", "B", "A", 256),
        ("drop", "B", 64, 128),
        ("repos", "B", 128, 256, -64),
        ("append", "A", 16, "newA"),
        ("append", "B", 16, "newB"),
    ]
    segs = [dict(seq="A", kv_end=272, q_len=16, hide=[], q_row0=0),
            dict(seq="B", kv_end=272, q_len=16, hide=[], q_row0=16)]
    return Workload("tiny", shape, 64, ops, segs, seed)


def trajectory_lengths(seed, n_turns=40, total=32768, system=1024, schema=1024,
                       reason=(100, 400), tool=(200, 2048)):
    """Turn lengths of one agent trajectory of exactly ``total`` tokens.

    Reasoning turns are uniform in ``reason``.  Tool responses are
    ``tool[0] + u_i`` with u_i uniform in [0, tool[1] - tool[0]], then the u_i
    are scaled so that the whole trajectory has ``total`` tokens (40 responses
    of up to 2K cannot otherwise fit in 32K); every response stays in ``tool``.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1])))
    r = rng.integers(reason[0], reason[1] + 1, size=n_turns)
    u = rng.integers(0, tool[1] - tool[0] + 1, size=n_turns)
    target = total - system - schema - int(r.sum()) - n_turns * tool[0]
    if target < 0:
        raise ValueError("trajectory too short for its turns")
    u = _split_exact(u + 1e-9, target)
    t = tool[0] + u
    if t.max() > tool[1]:
        raise ValueError("tool responses do not fit the trajectory length")
    return r, t


def llama8b_32k(seed=0, n_layers=1, total=32768, n_new=2048, n_dropped=20, n_turns=40, fork=False):
    """A Llama-3.1-8B-shaped layer (32 q / 8 kv heads, d 128, theta 5e5, page 16).

    32K-token trajectory: 1K system prompt, 1K tool schema, then 40 turns of
    (reasoning, tool response).  The oldest ``n_dropped`` tool responses are
    dropped; each drop [s, e) comes with repos of everything after it by
    -(e - s), so retained suffix tokens carry the composed shift.  Then
    ``n_new`` new tokens are appended and attend as one segment.  With
    ``fork`` the edits go to a fork of the trajectory (a new branch).
    """
    shape = Shape(n_layers, 32, 8, 128, 128, 5.0e5, 16)
    scale = total / 32768.0
    r, t = trajectory_lengths(seed, n_turns=n_turns, total=total,
                              system=int(1024 * scale), schema=int(1024 * scale),
                              reason=(max(1, int(100 * scale)), max(1, int(400 * scale))),
                              tool=(max(1, int(200 * scale)), max(2, int(2048 * scale))))
    pos = int(1024 * scale) * 2
    tool_spans = []
    for ri, ti in zip(r, t):
        pos += int(ri)
        tool_spans.append((pos, pos + int(ti)))
        pos += int(ti)
    assert pos == total
    seq = "S"
    ops = [("alloc", "S"), ("append", "S", total, "hist")]
    if fork:
        ops.append(("fork", "F", "S", total))
        seq = "F"
    for s, e in tool_spans[:n_dropped]:
        ops.append(("drop", seq, s, e))
        ops.append(("repos", seq, e, total, -(e - s)))
    ops.append(("append", seq, n_new, "new"))
    segs = [dict(seq=seq, kv_end=total + n_new, q_len=n_new, hide=[], q_row0=0)]
    n_pages = 2 * (-(-(total + n_new) // 16)) + 64
    meta = dict(tool_spans=tool_spans, reasoning=r.tolist())
    return Workload("llama8b_32k", shape, n_pages, ops, segs, seed, meta)


def sessions_64k(seed=0, n_layers=32, n_sessions=8, prefix=4096, per_session=65536,
                 q_per_seg=512, seg_range=(4, 16), max_directives=4, span_len=(256, 4096)):
    """Eight sessions of a Llama-3.1-8B-shaped cache sharing a 4K radix prefix.

    Each session is a 64K-token trajectory (the shared prefix plus its own
    history), gets 1..4 non-overlapping directives after the prefix (drop a
    span [s, e) and repos everything after it by a shift in [-(e-s), e-s], so
    shifts of either sign compose per token), then 4..16 sequential segments of
    ``q_per_seg`` new queries.  Segment k additionally hides the first m_k of a
    list of drop-only spans, m_0 <= m_1 <= ... (nested visibility sets).
    """
    shape = Shape(n_layers, 32, 8, 128, 128, 5.0e5, 16)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 2])))
    ops = [("alloc", "P"), ("append", "P", prefix, "prefix")]
    segs, row = [], 0
    total_pages = -(-prefix // 16)
    for i in range(n_sessions):
        name = f"S{i}"
        ops.append(("fork", name, "P", prefix))
        ops.append(("append", name, per_session - prefix, f"hist{i}"))
        nd = int(rng.integers(1, max_directives + 1))
        spans = _disjoint_spans(rng, prefix, per_session, nd, *span_len)
        for s, e in spans:
            ln = e - s
            ops.append(("drop", name, s, e))
            ops.append(("repos", name, e, per_session, int(rng.integers(-ln, ln + 1))))
        n_seg = int(rng.integers(seg_range[0], seg_range[1] + 1))
        ops.append(("append", name, n_seg * q_per_seg, f"new{i}"))
        extra = _disjoint_spans(rng, prefix, per_session, 6, 64, 1024)
        counts = np.sort(rng.integers(0, len(extra) + 1, size=n_seg))
        for k in range(n_seg):
            kv_end = per_session + (k + 1) * q_per_seg
            segs.append(dict(seq=name, kv_end=kv_end, q_len=q_per_seg,
                             hide=[tuple(x) for x in extra[:int(counts[k])]], q_row0=row))
            row += q_per_seg
        total_pages += -(-(per_session - prefix + n_seg * q_per_seg) // 16) + 4
    return Workload("sessions_64k", shape, total_pages + 64, ops, segs, seed)


def mla_dsv2lite(seed=0, n_layers=27, concurrency=1, prompt=17408, span=2016, stub=32, n_new=256):
    """DeepSeek-V2-Lite MLA shape: latent 512 (unrotated), K_pe 64 (rotated), 16 heads, page 64.

    ``concurrency`` independent ~17K-token sessions.  Each gets a Leyline
    AMORTIZE splice replacing a 2,016-token span with a 32-token stub
    (Delta = 32 - 2016 = -1984 on every downstream K_pe), then 256 new tokens
    attend as one segment.
    """
    shape = Shape(n_layers, 16, 1, 64, 512, 1.0e4, 64, mla=True)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 3])))
    ops, segs = [], []
    for c in range(concurrency):
        name = f"C{c}"
        # the span starts after a kept prefix and leaves a downstream suffix to rotate
        lo, tail = min(1024, prompt // 4), min(1056, prompt // 4)
        s = int(rng.integers(lo, prompt - span - tail + 1))
        ops += [("alloc", name), ("append", name, prompt, f"prompt{c}"),
                ("splice", name, s, s + span, stub, f"stub{c}"),
                ("append", name, n_new, f"new{c}")]
        kv_end = prompt - span + stub + n_new
        segs.append(dict(seq=name, kv_end=kv_end, q_len=n_new, hide=[], q_row0=c * n_new))
    n_pages = concurrency * (-(-(prompt + stub + n_new) // 64) + 4) + 8
    return Workload("mla_dsv2lite", shape, n_pages, ops, segs, seed)


def llama70b_128k(seed=0, n_layers=80, total=131072, n_spans=64, n_branches=32, q_per_branch=1024,
                  p_hide=0.25, max_shift=65536):
    """Llama-3.1-70B KV shape (8 kv heads, 64 query heads, d 128, theta 5e5, page 16).

    128K retained tokens cut into 64 equal spans; a full-cache repos sweep moves
    each span by its own shift, uniform in [-64K, 64K].  Then 32 branches
    (forks sharing every page) each append 1K new tokens and attend as one
    segment that hides a seeded random subset of the spans (p = 0.25).
    """
    shape = Shape(n_layers, 64, 8, 128, 128, 5.0e5, 16)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 4])))
    ln = total // n_spans
    ops = [("alloc", "M"), ("append", "M", total, "ctx")]
    for k in range(n_spans):
        ops.append(("repos", "M", k * ln, (k + 1) * ln, int(rng.integers(-max_shift, max_shift + 1))))
    ops.append(("flush", "M"))  # the sweep is in place, before any branch shares the pages
    segs = []
    for b in range(n_branches):
        name = f"B{b}"
        ops.append(("fork", name, "M", total))
        ops.append(("append", name, q_per_branch, f"new{b}"))
        hide = [(k * ln, (k + 1) * ln) for k in range(n_spans) if rng.random() < p_hide]
        segs.append(dict(seq=name, kv_end=total + q_per_branch, q_len=q_per_branch, hide=hide,
                         q_row0=b * q_per_branch))
    n_pages = -(-total // 16) + n_branches * (-(-q_per_branch // 16) + 1) + 64
    return Workload("llama70b_128k", shape, n_pages, ops, segs, seed)


WORKLOADS = {
    "tiny": tiny,
    "llama8b_32k": llama8b_32k,
    "sessions_64k": sessions_64k,
    "mla_dsv2lite": mla_dsv2lite,
    "llama70b_128k": llama70b_128k,
}
