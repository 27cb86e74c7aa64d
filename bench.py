"""Benchmark: one post-drop agent turn on a Llama-3.1-8B-shaped layer at 32K context.

A step is one pass of the whole hot path over one turn of synthetic input:
fork the 32K-token trajectory (a new branch), drop the oldest 20 tool
responses and reposition every retained suffix token by its composed shift
(host bookkeeping), append the 2,048 new tokens' K/V (kv_write), flush the
shifts (repos_rotate, copy-on-write into the branch), and run segment-batch
attention of the 2,048 new queries over the edited history
(segment_batch_attn); the branch is then released.  Inputs are resident in HBM
when the timed region starts; L2 is flushed (a 512 MiB write) between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own
independent sessions (weak scaling, no data-path collective); the time is the
max over ranks.
"""
import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "repos rotated tokens/s (HBM GB/s) + segment-batch attn TFLOP/s at 32K ctx"
UNIT = "post-drop turns/s"
WORKLOAD = ("llama8b_32k: Llama-3.1-8B-shaped layer (32 q / 8 kv heads, d 128, RoPE theta 5e5, page 16), "
            "32K-token 40-turn trajectory, drop oldest 20 tool responses + repos of the retained suffix "
            "(copy-on-write branch), 2,048 new query tokens in one segment")
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def measured_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel's source
    has changed since those counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", [rec.get("source")]):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != rec["source_sha256_16"]:
        return None
    return rec


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings over the process group (the slowest rank sets
    the whole job's time); the values unchanged when no group is initialised."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()):
        return list(values)
    x = torch.tensor(list(values), dtype=torch.float64, device=device)
    tdist.all_reduce(x, op=tdist.ReduceOp.MAX)
    return x.tolist()


class ClockSampler:
    """nvidia-smi clock / throttle samples (every 20 ms) over the loaded stretch that holds the timed
    region.  A reader thread collects the lines as they come; start() waits until nvidia-smi is up,
    mark() is called just before the warm-up and stop() after the end-to-end loop, and the summary
    keeps the samples taken in between (the device-timed steps alone last only milliseconds)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.thread = None
        self.lines = []
        self.first = 0

    def start(self, wait_s=3.0):
        import threading
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t_end = time.time() + wait_s
        while not self.lines and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line)

    def mark(self):
        self.first = len(self.lines)

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines[self.first:]:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": "warm-up through the end-to-end loop, every 20 ms"}


# --------------------------------------------------------------------------- GPU arm
class Turn:
    """The engine, the resident 32K-token trajectory and the per-step inputs."""

    def __init__(self, seed=0, host_inputs=False, attn_split=0, n_new=2048, n_layers=1):
        import torch
        from agentic_kv_cache_gb300 import akv, build, runner, synth
        build.build()
        self.torch, self.akv, self.runner = torch, akv, runner
        self.w = w = synth.llama8b_32k(seed=seed, fork=True, n_new=n_new, n_layers=n_layers)
        s = w.shape
        self.cfg = akv.config_from_shape(s, w.n_pages)
        self.pools = akv.make_pools(self.cfg)
        self.eng = akv.Engine(self.cfg, self.pools)
        self.eng.set_attention_split(attn_split)
        self.stream = torch.cuda.current_stream()
        fork_at = next(i for i, op in enumerate(w.ops) if op[0] == "fork")
        self.setup_ops, self.step_ops = w.ops[:fork_at], w.ops[fork_at:]
        src = runner.torch_kv_source(w)
        self.names = runner.run_ops(self.eng, w, kv_source=src, ops=self.setup_ops, stream=self.stream)
        new_op = next(op for op in self.step_ops if op[0] == "append")
        self.new_k, self.new_v = src(new_op[3], new_op[2])
        q32 = synth.q_array(w, 0)
        self.q = torch.from_numpy(q32).cuda().to(torch.bfloat16)
        self.nq = q32.shape[0]
        self.o = torch.empty((self.nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
        if host_inputs:
            self.h_k = self.new_k.cpu().pin_memory()
            self.h_v = self.new_v.cpu().pin_memory()
            self.h_q = self.q.cpu().pin_memory()
            self.h_o = torch.empty(self.o.shape, dtype=torch.bfloat16).pin_memory()
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()

    def step(self, host=False, fused=False):
        k, v = (self.h_k, self.h_v) if host else (self.new_k, self.new_v)
        names = dict(self.names)
        self.runner.run_ops(self.eng, self.w, kv_source=lambda *_: (k, v), ops=self.step_ops, names=names,
                            stream=self.stream)
        segs = self.runner.engine_segments(self.w, names)
        q, o = (self.h_q, self.h_o) if host else (self.q, self.o)
        for layer in range(self.w.shape.n_layers):
            self.eng.attend(layer, segs, q, self.nq, o, None, self.w.shape.scale, stream=self.stream, fused=fused)
        self.eng.seq_free(names["F"])

    def flush_l2(self):
        self.flush_buf.zero_()

    def io_bytes(self):
        b = lambda t: t.numel() * t.element_size()
        return b(self.new_k) + b(self.new_v) + b(self.q), b(self.o)


def repos_sweep(steps, warmup=2, n_layers=80):
    """repos_rotate on the Llama-3.1-70B-shaped 128K cache: 80 layers, 64 spans with shifts in
    +-64K, flushed in place (42.95 GB of algorithmic traffic per flush; the launch large enough for
    HBM to be the bound).  Steps alternate the sign of every shift so the work repeats exactly."""
    import torch
    from agentic_kv_cache_gb300 import akv, runner, synth
    w = synth.llama70b_128k(n_branches=0, n_layers=n_layers)
    cfg = akv.config_from_shape(w.shape, w.n_pages)
    pools = akv.make_pools(cfg)
    eng = akv.Engine(cfg, pools)
    st = torch.cuda.current_stream()
    names = runner.run_ops(eng, w, kv_source=runner.torch_device_kv_source(w),
                           ops=[op for op in w.ops if op[0] in ("alloc", "append")], stream=st)
    spans = [op for op in w.ops if op[0] == "repos"]
    torch.cuda.synchronize()

    def sweep(sign):
        for op in spans:
            eng.repos(names[op[1]], op[2], op[3], sign * op[4])
        eng.flush(names["M"], stream=st)

    for i in range(warmup):
        sweep(1 if i % 2 == 0 else -1)
    torch.cuda.synchronize()
    eng.profile_enable(True)
    for i in range(steps):
        sweep(1 if (warmup + i) % 2 == 0 else -1)
    stats = eng.profile_read()["repos_rotate"]
    eng.profile_enable(False)
    assert eng.check_device_error(st) == 0
    hbm = load_peaks()[0]
    ms = stats["ms"] / stats["launches"]
    gbs = stats["bytes"] / stats["launches"] / (ms * 1e-3) / 1e9
    tokens = stats["bytes"] / stats["launches"] / (2 * 8 * 128 * 2)
    del eng, pools
    torch.cuda.empty_cache()
    tr = measured_traffic("repos_rotate")
    traffic = None
    if tr:  # the capture's bytes scaled to this launch by the rotated token-layers (traffic grows in proportion)
        traffic = tr["dram_bytes_per_launch"] * (131072 * n_layers) / tr["units_per_launch"]
    return {"traffic_per_launch": traffic,
            "workload": f"llama70b_128k full-cache sweep: {n_layers} layers x 131,072 tokens x 8 kv heads x d 128, "
                        "64 spans, shifts in +-64K, in place", "launches": stats["launches"],
            "ms_per_launch": ms, "bytes_per_launch": stats["bytes"] / stats["launches"], "GB/s": gbs,
            "frac_of_hbm": gbs / hbm, "frac_of_8TBs": gbs / 8000.0,
            "rotated_token_layers_per_s": tokens / (ms * 1e-3),
            "rotated_tokens_per_s": tokens / n_layers / (ms * 1e-3)}


def reprefill_equiv(t, reps=3):
    """Re-prefill attention-equivalent of the 32K turn: the retained tokens of the post-drop branch
    re-entered as a fresh, fully visible sequence (what rebuilding the cache from compacted text
    costs in attention) and attended causally with every token as a query, on the same kernel."""
    torch = t.torch
    names = dict(t.names)
    t.runner.run_ops(t.eng, t.w, kv_source=lambda *_: (t.new_k, t.new_v), ops=t.step_ops, names=names,
                     stream=t.stream)
    n = int(t.eng.export_state(names["F"])["visible"].sum())
    t.eng.seq_free(names["F"])
    s = t.w.shape
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    k = torch.randn((s.n_layers, n, s.n_kv_heads, s.d_rot), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((s.n_layers, n, s.n_kv_heads, s.d_v), generator=gen, device="cuda").to(torch.bfloat16)
    sid = t.eng.seq_alloc()
    t.eng.append(sid, n, k, v, stream=t.stream)
    q = torch.randn((n, s.n_q_heads, s.d_rot), generator=gen, device="cuda").to(torch.bfloat16)
    o = torch.empty((n, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
    seg = [dict(seq=sid, kv_end=n, q_len=n, hide=np.zeros(0, np.int64), q_row0=0)]
    t.eng.attend(0, seg, q, n, o, None, s.scale, stream=t.stream)
    torch.cuda.synchronize()
    t.eng.profile_enable(True)
    for _ in range(reps):
        t.eng.attend(0, seg, q, n, o, None, s.scale, stream=t.stream)
    stats = t.eng.profile_read()["segment_attn"]
    t.eng.profile_enable(False)
    assert t.eng.check_device_error(t.stream) == 0
    t.eng.seq_free(sid)
    ms = stats["ms"] / stats["launches"]
    flops = stats["flops"] / stats["launches"]
    del q, o, k, v
    torch.cuda.empty_cache()
    return {"queries": n, "ms_per_layer": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12, "flops": flops}


def fused_vs_materialised(t, steps=10, warmup=3):
    """The same turn two ways: flush (repos_rotate into copy-on-write pages) then attend, or
    akv_attend_fused (keys rotated in shared memory inside the attention kernel, no HBM writes,
    no copy-on-write).  GPU time per turn from CUDA events on the stream, plus the attention
    kernel's own time."""
    torch = t.torch
    out = {}
    for fused in (False, True):
        for _ in range(warmup):
            t.step(fused=fused)
            t.flush_l2()
        torch.cuda.synchronize()
        t.eng.profile_enable(True)
        ms = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(t.stream)
            t.step(fused=fused)
            b.record(t.stream)
            t.flush_l2()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        stats = t.eng.profile_read()
        t.eng.profile_enable(False)
        assert t.eng.check_device_error(t.stream) == 0
        att, rep = stats["segment_attn"], stats["repos_rotate"]
        out["fused" if fused else "materialised"] = {
            "ms_per_turn": sum(ms) / steps,
            "attn_ms": att["ms"] / max(att["launches"], 1),
            "attn_TFLOP/s": att["flops"] / max(att["ms"], 1e-9) / 1e9,
            "repos_ms": rep["ms"] / steps,
            "repos_bytes_per_turn": rep["bytes"] / steps,
        }
    return out


def mla_fused_rotation(concurrencies=(1, 8), n_news=(16, 256), steps=4, warmup=2):
    """The DeepSeek-V2-Lite MLA turn (27 layers) two ways: flush (K_pe of every token after the
    splice rotated into copy-on-write pages) then attend, or akv_attend_fused (K_pe rotated in
    shared memory inside the pair kernel, the shift left pending).  Per concurrency C and new-token
    count: GPU time per turn from CUDA events on the stream, the attention kernel's own time and
    algorithmic TFLOP/s."""
    import torch
    from agentic_kv_cache_gb300 import akv, runner, synth
    out = {}
    for C in concurrencies:
        for n_new in n_news:
            w = synth.mla_dsv2lite(concurrency=C, n_new=n_new)
            s = w.shape
            cfg = akv.config_from_shape(s, w.n_pages + C * (17408 // 64 + 8))
            pools = akv.make_pools(cfg)
            eng = akv.Engine(cfg, pools)
            st = torch.cuda.current_stream()
            src = runner.torch_device_kv_source(w)
            setup = [op for op in w.ops if op[0] == "alloc" or (op[0] == "append" and op[3].startswith("prompt"))]
            names = runner.run_ops(eng, w, kv_source=src, ops=setup, stream=st)
            turn = [op for op in w.ops if op[0] == "splice" or (op[0] == "append" and op[3].startswith("new"))]
            kv = {op[5] if op[0] == "splice" else op[3]: src(op[5] if op[0] == "splice" else op[3],
                                                             op[4] if op[0] == "splice" else op[2]) for op in turn}
            q = torch.from_numpy(synth.q_array(w)).cuda().to(torch.bfloat16)
            o = torch.empty((q.shape[0], s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
            prompt = next(op for op in w.ops if op[0] == "append")[2]

            def step(fused):
                br = {f"C{c}": eng.seq_fork(names[f"C{c}"], prompt) for c in range(C)}
                runner.run_ops(eng, w, kv_source=lambda key, n: kv[key], ops=turn, names=br, stream=st)
                if not fused:
                    for c in range(C):
                        eng.flush(br[f"C{c}"], stream=st)
                segs = runner.engine_segments(w, br)
                for layer in range(s.n_layers):
                    eng.attend(layer, segs, q, q.shape[0], o, None, s.scale, stream=st, fused=fused)
                for c in range(C):
                    eng.seq_free(br[f"C{c}"])

            res = {}
            for fused in (False, True):
                for _ in range(warmup):
                    step(fused)
                torch.cuda.synchronize()
                eng.profile_enable(True)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                for _ in range(steps):
                    step(fused)
                b.record(st)
                torch.cuda.synchronize()
                stats = eng.profile_read()
                eng.profile_enable(False)
                assert eng.check_device_error(st) == 0
                att, rep = stats["segment_attn"], stats["repos_rotate"]
                res["fused" if fused else "materialised"] = {
                    "ms_per_turn": a.elapsed_time(b) / steps,
                    "attn_ms_per_layer": att["ms"] / max(att["launches"], 1),
                    "attn_TFLOP/s": att["flops"] / max(att["ms"], 1e-9) / 1e9,
                    "repos_ms_per_turn": rep["ms"] / steps,
                }
            out[f"C{C}_q{n_new}"] = res
            del eng, pools
            torch.cuda.empty_cache()
    return out


def compaction(steps=4, warmup=1, n_layers=32):
    """akv_compact on the post-drop branch of the 32K trajectory with every layer of a
    Llama-3.1-8B-shaped model (32 layers): ~24.5K visible tokens copied into dense pages, the
    pending suffix shift applied to the keys on the way.  HBM-bound copy: algorithmic bytes =
    read + write of every kept K and V row."""
    import torch
    from agentic_kv_cache_gb300 import akv, runner, synth
    w = synth.llama8b_32k(fork=True, n_layers=n_layers)
    w.n_pages += 2 * (32768 // 16)
    cfg = akv.config_from_shape(w.shape, w.n_pages)
    pools = akv.make_pools(cfg)
    eng = akv.Engine(cfg, pools)
    st = torch.cuda.current_stream()
    src = runner.torch_device_kv_source(w)
    fork_at = next(i for i, op in enumerate(w.ops) if op[0] == "fork")
    names = runner.run_ops(eng, w, kv_source=src, ops=w.ops[:fork_at], stream=st)
    new_op = next(op for op in w.ops[fork_at:] if op[0] == "append")
    kv = src(new_op[3], new_op[2])
    frag = None
    for i in range(warmup + steps):
        if i == warmup:
            torch.cuda.synchronize()
            eng.profile_enable(True)
        nm = runner.run_ops(eng, w, kv_source=lambda *_: kv, ops=w.ops[fork_at:], names=dict(names), stream=st)
        frag = eng.fragmentation(nm["F"])
        eng.compact(nm["F"], stream=st)
        eng.seq_free(nm["F"])
    stats = eng.profile_read()["compact_copy"]
    eng.profile_enable(False)
    assert eng.check_device_error(st) == 0
    del eng, pools, kv
    torch.cuda.empty_cache()
    calls = stats["launches"] // 2  # one compaction = a key launch and a value launch
    ms = stats["ms"] / calls
    gbs = stats["bytes"] / calls / (ms * 1e-3) / 1e9
    return {"workload": f"llama8b_32k post-drop branch, {n_layers} layers", "fragmentation_before": frag,
            "ms_per_compaction": ms, "bytes_per_compaction": stats["bytes"] / calls, "GB/s": gbs,
            "frac_of_hbm": gbs / load_peaks()[0]}


def turn_all_layers(steps=5, warmup=3, n_layers=32):
    """The headline turn with every layer of the Llama-3.1-8B shape (32 layers): the same fork,
    20 drops + composed suffix repos, append of 2,048 tokens, one flush (all 32 layers) and segment
    attention of the 2,048 queries in each of the 32 layers (one Q reused per layer).  This is the
    TTFT-equivalent of the post-drop turn over the whole model's cache."""
    import torch
    t = Turn(n_layers=n_layers)
    for _ in range(warmup):
        t.step()
        t.flush_l2()
    torch.cuda.synchronize()
    t.eng.profile_enable(True)
    ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(t.stream)
        t.step()
        b.record(t.stream)
        t.flush_l2()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    stats = t.eng.profile_read()
    t.eng.profile_enable(False)
    assert t.eng.check_device_error(t.stream) == 0
    del t
    torch.cuda.empty_cache()
    hbm, bf16_peak, _, _ = load_peaks()
    att, rep = stats["segment_attn"], stats["repos_rotate"]
    att_tf = att["flops"] / max(att["ms"], 1e-9) / 1e9
    rep_gbs = rep["bytes"] / max(rep["ms"], 1e-9) / 1e6
    return {"workload": f"llama8b_32k post-drop turn, {n_layers} layers", "ttft_equiv_ms": statistics.median(ms),
            "attn_ms_per_layer": att["ms"] / max(att["launches"], 1), "attn_TFLOP/s": att_tf,
            "attn_frac_of_bf16_dense": att_tf / bf16_peak, "flush_ms": rep["ms"] / steps,
            "flush_bytes": rep["bytes"] / steps, "repos_GB/s": rep_gbs, "repos_frac_of_hbm": rep_gbs / hbm,
            "kv_write_ms": stats["kv_write"]["ms"] / steps}


def sessions_turn(steps=2, warmup=1, n_layers=32):
    """Eight 64K-token sessions sharing a 4K prefix, 32 layers of the Llama-3.1-8B shape.  A step is
    one turn of all eight: each session gets a branch (a fork sharing its pages), its 1-4 drop +
    repos directives (shifts of either sign, composed per token) and its 4-16 x 512 new tokens
    (kv_write, all layers); one flush rotates every shifted retained key of every branch in all 32
    layers into copy-on-write pages (repos_rotate); then one segment-batch attention launch per layer
    covers all 4-16 segments of all eight sessions (512 queries each, nested hidden spans), 32
    layers; the branches are released.  Inputs (new K/V, one Q reused per layer) are resident."""
    import torch
    from agentic_kv_cache_gb300 import akv, runner, synth
    w = synth.sessions_64k(n_layers=n_layers)
    s = w.shape
    per = {}
    for op in w.ops:
        if op[0] == "append" and op[3].startswith("hist"):
            per[op[1]] = op[2]
    extra = sum(-(-n // s.page_size) + 1 for n in per.values())   # copy-on-write K pages of the branches
    cfg = akv.config_from_shape(s, w.n_pages + extra + 64)
    pools = akv.make_pools(cfg)
    eng = akv.Engine(cfg, pools)
    st = torch.cuda.current_stream()
    src = runner.torch_device_kv_source(w)
    setup, turn = [], []
    for op in w.ops:
        if op[0] in ("drop", "repos") or (op[0] == "append" and op[3].startswith("new")):
            turn.append(op)
        else:
            setup.append(op)
    names = runner.run_ops(eng, w, kv_source=src, ops=setup, stream=st)
    kv = {op[3]: src(op[3], op[2]) for op in turn if op[0] == "append"}
    nq = w.n_queries
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    q = torch.randn((nq, s.n_q_heads, s.d_rot), generator=gen, device="cuda").to(torch.bfloat16)
    o = torch.empty((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
    seq_len = {n: eng.seq_len(names[n]) for n in per}
    torch.cuda.synchronize()

    def step():
        br = {n: eng.seq_fork(names[n], seq_len[n]) for n in per}
        runner.run_ops(eng, w, kv_source=lambda key, n: kv[key], ops=turn, names=br, stream=st)
        eng.flush(-1, stream=st)
        segs = runner.engine_segments(w, br)
        for layer in range(s.n_layers):
            eng.attend(layer, segs, q, nq, o, None, s.scale, stream=st)
        for n in per:
            eng.seq_free(br[n])

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    eng.profile_enable(True)
    ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        step()
        b.record(st)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    stats = eng.profile_read()
    eng.profile_enable(False)
    assert eng.check_device_error(st) == 0
    del eng, pools, kv, q, o
    torch.cuda.empty_cache()
    hbm, bf16_peak, bf16_sus, _ = load_peaks()
    att, rep, kvw = stats["segment_attn"], stats["repos_rotate"], stats["kv_write"]
    att_tf = att["flops"] / max(att["ms"], 1e-9) / 1e9
    rep_gbs = rep["bytes"] / max(rep["ms"], 1e-9) / 1e6
    return {"workload": f"sessions_64k: 8 sessions x 64K tokens sharing a 4K prefix, {n_layers} layers, 32 q / 8 kv heads, "
                        f"d 128; {len(w.segments)} segments x 512 queries; directives per session 1-4",
            "segments": len(w.segments), "queries": nq, "ms_per_turn": statistics.median(ms),
            "attn_ms_per_layer": att["ms"] / max(att["launches"], 1),
            "attn_flops_per_layer": att["flops"] / max(att["launches"], 1), "attn_TFLOP/s": att_tf,
            "attn_frac_of_bf16_dense": att_tf / bf16_peak,
            "attn_frac_of_bf16_sustained": att_tf / bf16_sus if bf16_sus else None,
            "flush_ms": rep["ms"] / steps, "flush_bytes": rep["bytes"] / steps, "repos_GB/s": rep_gbs,
            "repos_frac_of_hbm": rep_gbs / hbm, "rotated_token_layers_per_s": rep["bytes"] / 4096 / max(rep["ms"], 1e-9) * 1e3,
            "kv_write_ms": kvw["ms"] / steps}


def branches_128k(n_layers=80, reps=1):
    """Segment-batch attention on the Llama-3.1-70B-shaped 128K cache (80 layers, 64 q / 8 kv heads,
    d 128): the 64 spans repositioned in place (shifts in +-64K), then 32 branches (forks sharing every
    page) each append 1,024 new tokens and attend as one segment hiding a seeded quarter of the spans;
    one launch per layer covers the 32 segments (32K query rows over ~100K visible keys each).  Every
    layer is timed once (one Q reused per layer)."""
    import torch
    from agentic_kv_cache_gb300 import akv, runner, synth
    w = synth.llama70b_128k(n_layers=n_layers)
    s = w.shape
    cfg = akv.config_from_shape(s, w.n_pages)
    pools = akv.make_pools(cfg)
    eng = akv.Engine(cfg, pools)
    st = torch.cuda.current_stream()
    names = runner.run_ops(eng, w, kv_source=runner.torch_device_kv_source(w), stream=st)
    nq = w.n_queries
    gen = torch.Generator(device="cuda")
    gen.manual_seed(12)
    q = torch.randn((nq, s.n_q_heads, s.d_rot), generator=gen, device="cuda").to(torch.bfloat16)
    o = torch.empty((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
    segs = runner.engine_segments(w, names)
    eng.attend(0, segs, q, nq, o, None, s.scale, stream=st)
    torch.cuda.synchronize()
    eng.profile_enable(True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        for layer in range(n_layers):
            eng.attend(layer, segs, q, nq, o, None, s.scale, stream=st)
    b.record(st)
    torch.cuda.synchronize()
    att = eng.profile_read()["segment_attn"]
    eng.profile_enable(False)
    assert eng.check_device_error(st) == 0
    del eng, pools, q, o
    torch.cuda.empty_cache()
    _, bf16_peak, bf16_sus, _ = load_peaks()
    tf = att["flops"] / max(att["ms"], 1e-9) / 1e9
    return {"workload": f"llama70b_128k: 32 branches x 1,024 queries over 131,072 keys (a quarter of the spans "
                        f"hidden per branch), 64 q / 8 kv heads, d 128, {n_layers} layers",
            "ms_all_layers": a.elapsed_time(b) / reps, "attn_ms_per_layer": att["ms"] / max(att["launches"], 1),
            "attn_flops_per_layer": att["flops"] / max(att["launches"], 1), "attn_TFLOP/s": tf,
            "attn_frac_of_bf16_dense": tf / bf16_peak,
            "attn_frac_of_bf16_sustained": tf / bf16_sus if bf16_sus else None}


def mass_pass(t, reps=5):
    """Per-token attention mass (the attn_mass kernel) of the 32K turn's 2,048 queries, after the
    attention pass that produced the lse.  `ms`: the kernel, CUDA events around its launch inside
    the library; `call_ms`: the whole call (host planning, upload, launch), events on the stream
    around it.  FLOPs: QK^T and the column-sum product ones(128 x 128) P over the visible pairs."""
    torch = t.torch
    names = dict(t.names)
    t.runner.run_ops(t.eng, t.w, kv_source=lambda *_: (t.new_k, t.new_v), ops=t.step_ops, names=names,
                     stream=t.stream)
    segs = t.runner.engine_segments(t.w, names)
    s = t.w.shape
    lse = torch.empty((t.nq, s.n_q_heads), dtype=torch.float32, device="cuda")
    t.eng.attend(0, segs, t.q, t.nq, t.o, lse, s.scale, stream=t.stream)
    total = sum(g["kv_end"] for g in t.w.segments)
    mass = torch.empty((total,), dtype=torch.float32, device="cuda")
    t.eng.attention_mass(0, segs, t.q, t.nq, lse, mass, s.scale, stream=t.stream)
    torch.cuda.synchronize()
    call_ms, kern_ms = [], []
    for _ in range(reps):
        t.flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t.eng.profile_enable(True)
        a.record(t.stream)
        t.eng.attention_mass(0, segs, t.q, t.nq, lse, mass, s.scale, stream=t.stream)
        b.record(t.stream)
        b.synchronize()
        st = t.eng.profile_read()["attn_mass"]
        t.eng.profile_enable(False)
        call_ms.append(a.elapsed_time(b))
        kern_ms.append(st["ms"] / max(st["launches"], 1))
        flops = st["flops"] / max(st["launches"], 1)
    assert t.eng.check_device_error(t.stream) == 0
    total_mass = float(mass.sum())
    t.eng.seq_free(names["F"])
    med = sorted(kern_ms)[len(kern_ms) // 2]
    _, bf16_peak, _, _ = load_peaks()
    tf = flops / (med * 1e-3) / 1e12
    tr = measured_traffic("attn_mass")
    return {"ms": med, "call_ms": sorted(call_ms)[len(call_ms) // 2], "mass_sum": total_mass,
            "expected_sum": t.nq * s.n_q_heads, "TFLOP/s": tf, "flops_per_launch": flops,
            "frac_of_bf16_dense": tf / bf16_peak, "traffic": tr["dram_bytes_per_launch"] if tr else None}


def mla_turns(concurrencies=(1, 4, 8, 16), steps=3, warmup=1):
    """DeepSeek-V2-Lite MLA turn per concurrency C (27 layers, latent 512 + K_pe 64, 16 heads, page 64,
    17K-token prompts): per session a branch of the prompt, the AMORTIZE splice of 2,016 tokens into a
    32-token stub, 256 new tokens; then one flush (K_pe of every downstream token, all layers) and
    segment attention of the 256 queries per session in each of the 27 layers."""
    import torch
    from agentic_kv_cache_gb300 import akv, runner, synth
    out = {}
    for C in concurrencies:
        w = synth.mla_dsv2lite(concurrency=C)
        s = w.shape
        cfg = akv.config_from_shape(s, w.n_pages + C * (17408 // 64 + 8))  # + copy-on-write K_pe pages of the branches
        pools = akv.make_pools(cfg)
        eng = akv.Engine(cfg, pools)
        st = torch.cuda.current_stream()
        src = runner.torch_device_kv_source(w)
        setup = [op for op in w.ops if op[0] == "alloc" or (op[0] == "append" and op[3].startswith("prompt"))]
        names = runner.run_ops(eng, w, kv_source=src, ops=setup, stream=st)
        turn = []
        for op in w.ops:
            if op[0] == "splice" or (op[0] == "append" and op[3].startswith("new")):
                turn.append(op)
        kv = {op[5] if op[0] == "splice" else op[3]: src(op[5] if op[0] == "splice" else op[3],
                                                          op[4] if op[0] == "splice" else op[2]) for op in turn}
        q32 = synth.q_array(w)
        q = torch.from_numpy(q32).cuda().to(torch.bfloat16)
        o = torch.empty((q.shape[0], s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
        prompt = next(op for op in w.ops if op[0] == "append")[2]

        def step():
            br = {}
            for c in range(C):
                br[f"C{c}"] = eng.seq_fork(names[f"C{c}"], prompt)
            runner.run_ops(eng, w, kv_source=lambda key, n: kv[key], ops=turn, names=br, stream=st)
            for c in range(C):
                eng.flush(br[f"C{c}"], stream=st)
            segs = runner.engine_segments(w, br)
            for layer in range(s.n_layers):
                eng.attend(layer, segs, q, q.shape[0], o, None, s.scale, stream=st)
            for c in range(C):
                eng.seq_free(br[f"C{c}"])

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        eng.profile_enable(True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(steps):
            step()
        b.record(st)
        torch.cuda.synchronize()
        stats = eng.profile_read()
        eng.profile_enable(False)
        assert eng.check_device_error(st) == 0
        att, rep = stats["segment_attn"], stats["repos_rotate"]
        out[f"C{C}"] = {
            "ms_per_turn": a.elapsed_time(b) / steps,
            "attn_ms_per_layer": att["ms"] / max(att["launches"], 1),
            "attn_TFLOP/s": att["flops"] / max(att["ms"], 1e-9) / 1e9,
            "flush_ms": rep["ms"] / max(rep["launches"], 1) * (rep["launches"] / steps),
            "repos_GB/s": rep["bytes"] / max(rep["ms"], 1e-9) / 1e6,
        }
        del eng, pools, q, o, kv
        torch.cuda.empty_cache()
    return out


def gpu_arm(args, rank, world):
    import torch
    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    t = Turn(seed=rank, host_inputs=True, attn_split=args.attn_split)
    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()

    clk = ClockSampler(dev).start()
    clk.mark()
    for _ in range(args.warmup):
        t.step()
        t.flush_l2()
    assert t.eng.check_device_error(t.stream) == 0

    # Timed steps: CUDA events around each turn on the turn's stream, the L2
    # flush between turns outside them.  Python's garbage collector is off
    # during timed loops (host noise of the harness, not of the library).
    # The library's per-launch events are off here: each acts as a barrier on
    # the stream (~13 us per turn); kernel durations come from a second pass.
    def timed_steps(profile):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier()
        if profile:
            t.eng.profile_enable(True)
        host_s = 0.0
        gc.disable()
        for i in range(args.steps):
            ev[i][0].record(t.stream)
            h0 = time.perf_counter()
            t.step()
            host_s += time.perf_counter() - h0
            ev[i][1].record(t.stream)
            t.flush_l2()
        gc.enable()
        barrier()
        st = None
        if profile:
            st = t.eng.profile_read()
            t.eng.profile_enable(False)
        assert t.eng.check_device_error(t.stream) == 0
        return [a.elapsed_time(b) for a, b in ev], host_s * 1e3 / args.steps, st

    ms, host_ms, _ = timed_steps(False)
    total_ms = sum(ms)
    ms_prof, _, stats = timed_steps(True)

    # End to end through the C ABI with pinned host buffers: turns run back to
    # back as a serving loop would run them (the host prepares turn i + 1 while
    # the GPU runs turn i); every turn copies its K, V and Q from pinned host
    # memory (on the library's copy stream) and its output back to pinned host
    # memory on an output stream (akv_set_output_stream), so turn i's output
    # copy overlaps turn i + 1's kernels; all of it is inside the timed region.
    # No L2 flush between these turns: a turn touches ~225 MB (the branch's
    # K/V, its copy-on-write pages, Q, O and the new K/V), more than the
    # 129 MB L2.  The same loop with the 512 MiB flush between turns (timed)
    # and the latency of one turn on its own are reported beside it.
    copy_back = torch.cuda.Stream()
    t.eng.set_output_stream(copy_back)

    def e2e_loop(flush):
        for _ in range(2):
            t.step(host=True)
            if flush:
                t.flush_l2()
        barrier()
        gc.disable()
        t0 = time.perf_counter()
        for i in range(args.steps):
            t.step(host=True)
            if flush:
                t.flush_l2()
        barrier()
        e = (time.perf_counter() - t0) * 1e3
        gc.enable()
        return e

    e2e_total = e2e_loop(False)
    e2e_flushed = e2e_loop(True)
    lat_ms = []
    for i in range(max(3, min(args.steps, 10))):
        t.flush_l2()
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        t.step(host=True)
        torch.cuda.synchronize()
        lat_ms.append((time.perf_counter() - t1) * 1e3)
    lat_ms.sort()
    clk.stop()

    if dist:
        total_ms, e2e_total, e2e_flushed = max_over_ranks([total_ms, e2e_total, e2e_flushed], "cuda")
    if rank != 0:
        return None

    hbm, bf16_peak, bf16_sus, peak_kind = load_peaks()
    rep, att, kvw = stats["repos_rotate"], stats["segment_attn"], stats["kv_write"]
    rep_ms = rep["ms"] / max(rep["launches"], 1)
    att_ms = att["ms"] / max(att["launches"], 1)
    rep_bytes = rep["bytes"] / max(rep["launches"], 1)
    att_flops = att["flops"] / max(att["launches"], 1)
    rot_tokens = rep_bytes / (2 * 8 * 128 * 2)  # token-layers per launch: read + write of 8 x 128 bf16
    rep_gbs = rep_bytes / (rep_ms * 1e-3) / 1e9
    att_tf = att_flops / (att_ms * 1e-3) / 1e12
    share = {k: v["ms"] for k, v in stats.items()}
    dominant = max(share, key=share.get)
    h2d, d2h = t.io_bytes()
    value = world * args.steps / (total_ms * 1e-3)
    e2e_value = world * args.steps / (e2e_total * 1e-3)
    if dominant == "segment_attn":
        tr = measured_traffic("segment_attn")
        roof = {"kernel": "segment_attn", "bound": "tensor", "achieved": att_tf, "peak": bf16_peak,
                "unit": "TFLOP/s", "frac": att_tf / bf16_peak,
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "peak_kind": f"{peak_kind} bf16 dense burst (sustained {bf16_sus})"}
    else:
        tr = measured_traffic("repos_rotate")
        roof = {"kernel": "repos_rotate", "bound": "hbm", "achieved": rep_gbs, "peak": hbm, "unit": "GB/s",
                "frac": rep_gbs / hbm, "traffic": None, "peak_kind": f"{peak_kind} HBM copy"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "flushed between steps (512 MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "attn_split": args.attn_split or "auto"},
        "repos_rotate": {"rotated_tokens_per_s": rot_tokens / (rep_ms * 1e-3), "rotated_tokens_per_launch": rot_tokens,
                         "GB/s": rep_gbs, "frac_of_hbm": rep_gbs / hbm, "frac_of_8TBs": rep_gbs / 8000.0,
                         "ms_per_launch": rep_ms},
        "segment_batch_attn": {"TFLOP/s": att_tf, "frac_of_bf16_dense": att_tf / bf16_peak,
                               "frac_of_bf16_sustained": att_tf / bf16_sus if bf16_sus else None,
                               "ms_per_launch": att_ms, "flops_per_launch": att_flops},
        "kv_write": {"ms_per_step": kvw["ms"] / args.steps, "GB/s": kvw["bytes"] / max(kvw["ms"], 1e-9) / 1e6},
        "ttft_equiv_ms": total_ms / args.steps,
        "ms_per_step_median": statistics.median(ms),
        "host_ms_per_step": host_ms,
        "kernel_timing": "kernel durations, shares and rooflines from a second pass of the same steps with CUDA "
                         f"events around every launch ({sum(ms_prof) / args.steps:.4f} ms per turn with them)",
        "kernel_share": {k: v / max(sum(share.values()), 1e-9) for k, v in share.items()},
        "roofline": roof,
        "gpu_launches": int(sum(v["launches"] for v in stats.values())),
        "clocks": clk.summary(),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_total / args.steps,
                "mode": "turns back to back through the C ABI, inputs from and outputs to pinned host memory; "
                        "no L2 flush (a turn touches ~225 MB > 129 MB L2); output copies on an output stream",
                "ms_per_step_l2_flushed": e2e_flushed / args.steps,
                "latency_ms_one_turn": lat_ms[len(lat_ms) // 2]},
    }
    if not args.no_extra:
        line["reprefill_equiv"] = reprefill_equiv(t)
        line["reprefill_equiv"]["turn_cache_path_ms"] = total_ms / args.steps
        line["attention_mass"] = mass_pass(t)
        fz = {"turn_2048_queries": fused_vs_materialised(t)}
        del t
        torch.cuda.empty_cache()
        t = Turn(seed=rank, attn_split=args.attn_split, n_new=16)
        fz["turn_16_queries"] = fused_vs_materialised(t)
        fz["mla_dsv2lite"] = mla_fused_rotation()
        line["fused_rotation"] = fz
    del t
    torch.cuda.empty_cache()
    if not args.no_sweep:
        line["repos_rotate_sweep"] = repos_sweep(steps=4, n_layers=args.sweep_layers)
    if not args.no_extra:
        line["turn_32_layers"] = turn_all_layers()
        line["sessions_64k_turn"] = sessions_turn()
        line["llama70b_128k_attention"] = branches_128k()
        line["mla_dsv2lite_turn"] = mla_turns()
        line["compact_copy"] = compaction()
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        if not args.no_extra:
            line["oracle_beside"] = oracle_beside(line)
    return line


def oracle_beside(line):
    """The float64 oracle timed on host cores beside the GPU numbers of the next rows (attention
    mass, compaction, one MLA layer), each on a bounded sample scaled to the GPU's workload."""
    from agentic_kv_cache_gb300 import synth
    from oracle import attention, bf16, kernels
    from oracle.cache import CacheModel
    out = {"cores": os.cpu_count(), "kind": "oracle"}
    ot = OracleTurn(extra_pages=2048)  # room for the compacted copy of the branch
    m, w, sh = ot.model, ot.w, ot.w.shape
    names = dict(ot.names)
    for op in ot.step_ops:
        if op[0] == "fork":
            names[op[1]] = m.seq_fork(names[op[2]], op[3])
        elif op[0] == "drop":
            m.drop(names[op[1]], op[2], op[3])
        elif op[0] == "repos":
            m.repos(names[op[1]], op[2], op[3], op[4])
        elif op[0] == "append":
            ot._write(m.append(names[op[1]], op[2]), op[3], op[2])
    g = w.segments[0]
    kernels.repos_runs(ot.kp, m.flush([names[g["seq"]]]), sh.rope_base, sh.rope_layout, out=ot.kp)
    seg_runs, _ = m.segment_runs(names[g["seq"]], g["kv_end"], g["q_len"], g["hide"])
    k = kernels.gather(ot.kp, 0, seg_runs, 0).astype(np.float64)
    # attention mass: the first `rows` queries against the entries they see (same cost per row)
    rows, q_len, q0 = 32, g["q_len"], g["q_row0"]
    t0 = time.perf_counter()
    attention.attention_mass(ot.qb[q0:q0 + rows], k[:k.shape[0] - q_len + rows], sh.scale)
    t_mass = (time.perf_counter() - t0) * q_len / rows
    gm = line.get("attention_mass", {}).get("call_ms")  # the whole call: planning, upload, kernel
    out["attention_mass"] = {"oracle_s": t_mass, "gpu_ms": gm, "gpu_speedup": t_mass / (gm * 1e-3) if gm else None,
                             "sample": f"{rows} of {q_len} query rows (all heads) over their visible entries, "
                                       "scaled to all rows"}
    # compaction: bookkeeping plus the copy of one layer (rotating the pending shifts), scaled to 32
    t0 = time.perf_counter()
    copies = m.compact(names["F"])
    t_book = time.perf_counter() - t0
    part = copies[:2048]
    t0 = time.perf_counter()
    kernels.compact_copy(ot.kp, ot.vp, [], sh.rope_base, sh.rope_layout)  # the pools' copy alone
    t_fixed = time.perf_counter() - t0
    t0 = time.perf_counter()
    kernels.compact_copy(ot.kp, ot.vp, part, sh.rope_base, sh.rope_layout)
    t_copy = t_fixed + max(time.perf_counter() - t0 - t_fixed, 0.0) * len(copies) / max(len(part), 1)
    gc = line.get("compact_copy", {}).get("ms_per_compaction")
    t_comp = t_book + 32 * t_copy
    out["compaction"] = {"oracle_s": t_comp, "gpu_ms": gc, "gpu_speedup": t_comp / (gc * 1e-3) if gc else None,
                         "sample": f"bookkeeping of the whole branch ({len(copies)} kept tokens) and the copy of "
                                   f"{len(part)} of them in one layer, the per-token part scaled to all tokens, "
                                   "the one-layer copy scaled linearly to 32 layers"}
    m.seq_free(names["F"])
    # one MLA layer of a one-session turn: the spliced 17K session, attention on sampled rows
    wm = synth.mla_dsv2lite(n_layers=1, concurrency=1)
    ms_ = wm.shape
    cm = CacheModel(wm.n_pages, ms_.page_size)
    kp = np.zeros((1, wm.n_pages, 1, ms_.page_size, ms_.d_rot), np.float32)
    vp = np.zeros((1, wm.n_pages, 1, ms_.page_size, ms_.d_v), np.float32)
    mn = {}
    for op in wm.ops:
        if op[0] == "alloc":
            mn[op[1]] = cm.seq_alloc()
            continue
        n, key = (op[2], op[3]) if op[0] == "append" else (op[4], op[5])
        slots = cm.append(mn[op[1]], n) if op[0] == "append" else cm.splice(mn[op[1]], op[2], op[3], op[4])
        k32, v32 = synth.kv_arrays(wm, key, n)
        idx = np.array(slots)
        kp[:, idx[:, 0], :, idx[:, 2]] = bf16.round_bf16(k32.astype(np.float64)).astype(np.float32).transpose(1, 0, 2, 3)
        vp[:, idx[:, 1], :, idx[:, 2]] = bf16.round_bf16(v32.astype(np.float64)).astype(np.float32).transpose(1, 0, 2, 3)
    gs = wm.segments[0]
    kernels.repos_runs(kp, cm.flush([mn[gs["seq"]]]), ms_.rope_base, ms_.rope_layout, out=kp)
    runs_m, _ = cm.segment_runs(mn[gs["seq"]], gs["kv_end"], gs["q_len"], gs["hide"])
    qm = bf16.round_bf16(synth.q_array(wm).astype(np.float64))[gs["q_row0"]:gs["q_row0"] + gs["q_len"]]
    rows_m = 8
    t0 = time.perf_counter()
    kernels.attend_segment(qm, kp, vp, 0, runs_m, ms_.scale, mla=True,
                           rows=np.linspace(0, gs["q_len"] - 1, rows_m).astype(np.int64))
    t_mla = (time.perf_counter() - t0) * gs["q_len"] / rows_m
    c1 = line.get("mla_dsv2lite_turn", {}).get("C1", {}).get("attn_ms_per_layer")
    out["mla_attention_one_layer_c1"] = {
        "oracle_s": t_mla, "gpu_ms": c1, "gpu_speedup": t_mla / (c1 * 1e-3) if c1 else None,
        "sample": f"{rows_m} of {gs['q_len']} query rows (16 heads, d_qk 576) over the spliced session, scaled"}
    return out


# ------------------------------------------------------------------ oracle (CPU) arm
class OracleTurn:
    """The float64 oracle on the same turn: resident trajectory built once, then per step
    the turn's bookkeeping, the full repos and attention on a sample of query rows."""

    def __init__(self, seed=0, extra_pages=0):
        from agentic_kv_cache_gb300 import synth
        from oracle import attention, bf16, kernels
        from oracle.cache import CacheModel
        self.synth, self.bf16, self.kernels, self.attention = synth, bf16, kernels, attention
        self.w = w = synth.llama8b_32k(seed=seed, fork=True)
        s = w.shape
        fork_at = next(i for i, op in enumerate(w.ops) if op[0] == "fork")
        self.step_ops = w.ops[fork_at:]
        self.model = CacheModel(w.n_pages + extra_pages, s.page_size)
        self.kp = np.zeros((1, w.n_pages + extra_pages, s.n_kv_heads, s.page_size, s.d_rot), np.float32)
        self.vp = np.zeros_like(self.kp)
        self.names = {}
        self.values = {}
        for op in w.ops[:fork_at]:
            if op[0] == "alloc":
                self.names[op[1]] = self.model.seq_alloc()
            elif op[0] == "append":
                self._write(self.model.append(self.names[op[1]], op[2]), op[3], op[2])
        new = next(op for op in self.step_ops if op[0] == "append")
        self._values(new[3], new[2])
        self.qb = bf16.round_bf16(synth.q_array(w).astype(np.float64))

    def _values(self, key, n):
        if key not in self.values:
            k32, v32 = self.synth.kv_arrays(self.w, key, n)
            self.values[key] = (self.bf16.round_bf16(k32.astype(np.float64)).astype(np.float32),
                                self.bf16.round_bf16(v32.astype(np.float64)).astype(np.float32))
        return self.values[key]

    def _write(self, slots, key, n):
        kb, vb = self._values(key, n)
        idx = np.array(slots)
        self.kp[:, idx[:, 0], :, idx[:, 2]] = kb.transpose(1, 0, 2, 3)
        self.vp[:, idx[:, 1], :, idx[:, 2]] = vb.transpose(1, 0, 2, 3)

    def step(self, rows, offset=0):
        """Run one turn (attention on `rows` query rows, evenly spaced from `offset`); returns (seconds
        per full turn, parts)."""
        s, m = self.w.shape, self.model
        names = dict(self.names)
        t0 = time.perf_counter()
        for op in self.step_ops:
            if op[0] == "fork":
                names[op[1]] = m.seq_fork(names[op[2]], op[3])
            elif op[0] == "drop":
                m.drop(names[op[1]], op[2], op[3])
            elif op[0] == "repos":
                m.repos(names[op[1]], op[2], op[3], op[4])
            elif op[0] == "append":
                self._write(m.append(names[op[1]], op[2]), op[3], op[2])
        g = self.w.segments[0]
        runs = m.flush([names[g["seq"]]])
        seg_runs, _ = m.segment_runs(names[g["seq"]], g["kv_end"], g["q_len"], g["hide"])
        t_book = time.perf_counter() - t0
        t0 = time.perf_counter()
        self.kernels.repos_runs(self.kp, runs, s.rope_base, s.rope_layout, out=self.kp)
        t_rep = time.perf_counter() - t0
        stride = g["q_len"] // rows
        if stride >= 2:  # every stride-th row from a rotating offset
            sample = np.arange(rows, dtype=np.int64) * stride + offset % stride
        else:            # most rows: spread evenly over the segment (later rows see more keys)
            sample = np.linspace(0, g["q_len"] - 1, rows).astype(np.int64)
        # attention = gather of the segment's KV (once per turn) + per-row work (scaled to all rows)
        t0 = time.perf_counter()
        k = self.kernels.gather(self.kp, 0, seg_runs, 0).astype(np.float64)
        v = self.kernels.gather(self.vp, 0, seg_runs, 1).astype(np.float64)
        t_gather = time.perf_counter() - t0
        t0 = time.perf_counter()
        self.attention.segment_attention(self.qb, k, v, s.scale, rows=sample)
        t_att = t_gather + (time.perf_counter() - t0) * g["q_len"] / rows
        m.seq_free(names["F"])
        return t_book + t_rep + t_att, dict(bookkeeping_s=t_book, repos_s=t_rep, attention_s=t_att,
                                            gather_s=t_gather, rows=rows)


def cpu_baseline(seconds=15.0):
    ot = OracleTurn()
    est, parts = ot.step(rows=16)
    att_per_row = (parts["attention_s"] - parts["gather_s"]) / 2048
    fixed = parts["bookkeeping_s"] + parts["repos_s"] + parts["gather_s"]
    rows = int(np.clip((seconds - fixed) / max(att_per_row, 1e-6), 16, 2048))
    est, parts = ot.step(rows=rows)
    return {"value": 1.0 / est, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"float64 numpy oracle, one turn: full bookkeeping and repos, attention on {rows} of 2048 "
                       f"query rows (all heads, full visible KV) scaled to 2048; BLAS threads = all host cores"),
            "seconds_per_turn": est, "parts": parts}


REF_ROWS = 128  # query rows of the reference arm's attention sample per step


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    ot = OracleTurn()
    for i in range(args.warmup):
        ot.step(rows=REF_ROWS, offset=i)
    # each step takes a different slice of the query rows: after 2048 / REF_ROWS steps every row was timed
    times = [ot.step(rows=REF_ROWS, offset=args.warmup + i)[0] for i in range(args.steps)]
    total = sum(times)
    value = args.steps / total
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "n/a (host)", "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"per step: full bookkeeping and repos, attention on {REF_ROWS} of 2048 query "
                                       f"rows (every {2048 // REF_ROWS}th, offset by the step number, so successive "
                                       f"steps time different rows) scaled to the full turn"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the large repos_rotate sweep measurement")
    ap.add_argument("--only-sweep", action="store_true", help="run only the repos_rotate sweep (for profiling)")
    ap.add_argument("--sweep-layers", type=int, default=80)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--only-mla", type=int, default=0, metavar="C",
                    help="run only the MLA turn at concurrency C (for profiling)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the re-prefill equivalent and the MLA per-concurrency turns")
    ap.add_argument("--only-leg", default="", choices=["", "turn32", "sessions", "branches128k", "mlafused", "fused32"],
                    help="run only one measurement leg (for profiling): the 32-layer 32K turn, the 8 x 64K "
                         "sessions turn, the 128K branches' attention, fused vs materialised rotation on "
                         "the MLA turn or on the 32K turn (2,048 and 16 queries)")
    ap.add_argument("--leg-layers", type=int, default=0, help="layers of the --only-leg workload (0: full)")
    ap.add_argument("--attn-split", type=int, default=0,
                    help="KV chunks per attention work item: 0 chooses automatically, 1 never splits")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", args.gpus if "RANK" in os.environ else 1))
    if args.only_mla:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        from agentic_kv_cache_gb300 import build
        build.build()
        print(json.dumps(mla_turns((args.only_mla,), steps=args.steps, warmup=args.warmup)), flush=True)
        return
    if args.only_leg:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        from agentic_kv_cache_gb300 import build
        build.build()
        L = args.leg_layers
        if args.only_leg == "turn32":
            out = turn_all_layers(steps=args.steps, warmup=args.warmup, n_layers=L or 32)
        elif args.only_leg == "sessions":
            out = sessions_turn(steps=args.steps, warmup=args.warmup, n_layers=L or 32)
        elif args.only_leg == "mlafused":
            out = mla_fused_rotation(steps=args.steps, warmup=args.warmup)
        elif args.only_leg == "fused32":
            out = {"turn_2048_queries": fused_vs_materialised(Turn(seed=0), args.steps, args.warmup)}
            torch.cuda.empty_cache()
            out["turn_16_queries"] = fused_vs_materialised(Turn(seed=0, n_new=16), args.steps, args.warmup)
        else:
            out = branches_128k(n_layers=L or 80)
        print(json.dumps(out), flush=True)
        return
    if args.only_sweep:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        from agentic_kv_cache_gb300 import build
        build.build()
        print(json.dumps(repos_sweep(args.steps, args.warmup, args.sweep_layers)), flush=True)
        return
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as tdist
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            tdist.init_process_group("nccl")
        line = gpu_arm(args, rank, world)
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
