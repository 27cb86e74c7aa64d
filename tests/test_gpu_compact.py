"""akv_compact on the GPU (the compact_copy kernel) against the oracle.

[AKV-blog] "Dilemma 2: Memory Fragmentation in Paged Pools": visible tokens
are copied into fresh dense pages, a pending shift applied to the copied key.
Bars: values copied without a shift (every V / latent row and unshifted K
rows) bit-identical; rotated key rows under the rotated-key rule of the
repos tests (within one bf16 ulp of the rounded float64 rotation plus the
float32 allowance, >= 99.9 % bit-identical); every other pool row untouched;
attention over the compacted sequence equals the oracle's within the
attention bar."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


def remap_segments(w, states, names_o):
    """Segments in post-compaction indices: a logical index i becomes the number of visible tokens
    before it (dropped tokens left the sequence)."""
    out = []
    for g in w.segments:
        vis = np.asarray(states[names_o[g["seq"]]]["visible"], bool)
        before = np.concatenate([[0], np.cumsum(vis)])
        out.append(dict(g, kv_end=int(before[g["kv_end"]]),
                        hide=[(int(before[a]), int(before[b])) for a, b in g["hide"]]))
    return out


def compact_case(w, check_attention=True):
    from gpu_case import Case
    from oracle import kernels, rope
    from test_gpu_attention import ATOL
    from test_gpu_repos import compare_rotated, rotated_mask
    c = Case(w)
    c.run_ops()
    s = w.shape
    ids = sorted({c.names_o[g["seq"]] for g in w.segments})
    states = {i: c.model.state(i) for i in ids}
    rot = rotated_mask(c, c.flush_runs)
    a, b = rope.pair_indices(s.d_rot, s.rope_layout)
    n_rot = 0
    for i in ids:
        copies = c.model.compact(i)
        rot0, term0 = rot.copy(), c.kterm.copy()
        for sk, sv, ss, dk, dv, ds, d in copies:
            if d:
                x = np.abs(c.kp[:, sk, :, ss, :].astype(np.float64))
                t = 2.0 ** -20 * (x[..., a] + x[..., b])
                view = c.kterm[:, dk, :, ds, :]        # basic indexing: a view [L][H][d]
                view[..., a] = t
                view[..., b] = t
                rot[:, dk, :, ds] = True
                n_rot += 1
            else:  # a plain copy carries the source row's state (rotated earlier or not)
                c.kterm[:, dk, :, ds, :] = term0[:, sk, :, ss, :]
                rot[:, dk, :, ds] = rot0[:, sk, :, ss]
        ko, vo = kernels.compact_copy(c.kp, c.vp, copies, s.rope_base, s.rope_layout)
        c.kp[:], c.vp[:] = ko, vo
        c.eng.compact(i, stream=c.stream)
        assert c.eng.fragmentation(i) == c.model.fragmentation(i)
        assert c.model.fragmentation(i) < 1.0 / max(len(copies) // s.page_size, 1) + 1e-12
    kg, vg = c.gpu_pools()
    assert np.array_equal(vg, c.vp), "V pool after compaction"
    compare_rotated(kg, c.kp, rot, c.kterm)
    assert c.eng.check_device_error() == 0
    assert n_rot > 0, "workload had no pending shift to fuse into the copy"
    if check_attention:
        w.segments = remap_segments(w, states, c.names_o)
        q32, o, lse = c.attend_gpu()
        for k, g in enumerate(w.segments):
            rows = np.arange(g["q_len"])
            want_o, want_lse = c.attend_oracle(q32, k, rows)
            assert np.abs(o[g["q_row0"] + rows] - want_o).max() <= ATOL
            assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL
    return c


def test_compact_tiny_branch():
    compact_case(synth.tiny())


def test_compact_32k_trajectory_small():
    w = synth.llama8b_32k(total=4096, n_new=200, fork=True, n_layers=2)
    w.n_pages += 300
    compact_case(w)


def test_compact_half_layout():
    w = synth.llama8b_32k(total=4096, n_new=100, fork=True, n_layers=1)
    w.shape.rope_layout = "half"
    w.n_pages += 300
    compact_case(w)


def test_compact_mla_spliced():
    w = synth.mla_dsv2lite(n_layers=2, concurrency=2, prompt=3000, span=700, stub=20, n_new=100)
    w.n_pages += 120
    compact_case(w)
