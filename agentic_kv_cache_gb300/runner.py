"""Drive a synth.Workload through the engine.

``run_ops`` replays the workload's operation list on an ``akv.Engine``;
``kv_source`` supplies the K/V data of each append / splice as device (or
host) tensors in the layouts of include/akv.h.  Returns the symbolic sequence
names mapped to engine ids.
"""
import numpy as np

from . import synth


def torch_kv_source(w, device="cuda"):
    """K/V tensors for each append/splice key: seeded N(0,1) rounded to bf16 by torch."""
    import torch

    def source(key, n):
        k, v = synth.kv_arrays(w, key, n)
        return (torch.from_numpy(k).to(device=device, dtype=torch.bfloat16),
                torch.from_numpy(v).to(device=device, dtype=torch.bfloat16))
    return source


def torch_device_kv_source(w, device="cuda"):
    """Same shapes, drawn on the device with a seeded torch generator (for the large workloads)."""
    import torch
    import zlib

    def source(key, n):
        g = torch.Generator(device=device)
        g.manual_seed((w.seed * 1000003 + zlib.crc32(key.encode())) % (2 ** 63))
        s = w.shape
        k = torch.randn((s.n_layers, n, s.n_kv_heads, s.d_rot), generator=g, device=device).to(torch.bfloat16)
        v = torch.randn((s.n_layers, n, s.n_kv_heads, s.d_v), generator=g, device=device).to(torch.bfloat16)
        return k, v
    return source


def run_ops(engine, w, kv_source=None, stream=None, ops=None, names=None):
    """Replay ops on the engine; kv_source(key, n) -> (k, v) or None for metadata-only engines.
    Consecutive drop / repos ops on one sequence go to the engine as one akv_edit call."""
    names = {} if names is None else names
    ops = list(w.ops if ops is None else ops)
    i = 0
    while i < len(ops):
        op = ops[i]
        kind = op[0]
        if kind in ("drop", "repos"):
            j = i
            while j < len(ops) and ops[j][0] in ("drop", "repos") and ops[j][1] == op[1]:
                j += 1
            engine.edit(names[op[1]], [(o[0],) + tuple(o[2:]) for o in ops[i:j]])
            i = j
            continue
        i += 1
        if kind == "alloc":
            names[op[1]] = engine.seq_alloc()
        elif kind == "fork":
            names[op[1]] = engine.seq_fork(names[op[2]], op[3])
        elif kind == "append":
            k, v = kv_source(op[3], op[2]) if kv_source else (None, None)
            engine.append(names[op[1]], op[2], k, v, stream=stream)
        elif kind == "splice":
            k, v = kv_source(op[5], op[4]) if kv_source else (None, None)
            engine.splice(names[op[1]], op[2], op[3], op[4], k, v, stream=stream)
        elif kind == "flush":
            engine.flush(names[op[1]], stream=stream)
        elif kind == "compact":
            engine.compact(names[op[1]], stream=stream)
        else:
            raise ValueError(f"unknown op {kind}")
    return names


def engine_segments(w, names):
    """The workload's segments with engine sequence ids."""
    return [dict(seq=names[s["seq"]], kv_end=s["kv_end"], q_len=s["q_len"], hide=np.asarray(s["hide"]).reshape(-1),
                 q_row0=s["q_row0"]) for s in w.segments]
