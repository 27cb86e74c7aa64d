"""akv_attend_fused on the GPU: the rotation applied to K tiles inside the
attention kernel, pending shifts left pending ([AKV-blog] section 4, keys
rotated on their way to the tensor core instead of materialised in HBM; under
MLA only K_pe is rotated, [Leyline] "Method").

Bars: the same as segment_batch_attn (bf16 output vs the float64 oracle on the
oracle's materialised keys within max-abs 2e-2, LSE within 2e-2); the pools are
bit-for-bit untouched and the shifts stay pending; against flush-then-attend on
the same inputs the output differs only by float summation order (the rotated
key bits are the same; fused runs also break where the shift changes)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import akv, synth

pytestmark = pytest.mark.gpu

ATOL = 2e-2


def fused_case(w, k_rows=None, seed=0, also_materialised=True):
    from gpu_case import Case
    from test_gpu_attention import sample_rows
    c = Case(w)
    c.run_ops()
    c.flush_segments(engine=False)           # oracle keys at the composed positions
    k0, v0 = c.pools[0].clone(), c.pools[1].clone()
    seqs = sorted({c.names_e[g["seq"]] for g in w.segments})
    pending = {i: c.eng.export_state(i)["delta"].copy() for i in seqs}
    q32, o, lse = c.attend_gpu(fused=True)
    torch.cuda.synchronize()
    assert torch.equal(c.pools[0], k0) and torch.equal(c.pools[1], v0), "the fused path wrote to the pools"
    for i in seqs:
        assert np.array_equal(c.eng.export_state(i)["delta"], pending[i]), "pending shifts changed"
    assert any(np.any(d != 0) for d in pending.values()), "workload has no pending shift to fuse"
    rng = np.random.default_rng(seed)
    G = w.shape.n_q_heads // w.shape.n_kv_heads
    worst = 0.0
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"]) if k_rows is None else sample_rows(g["q_len"], k_rows, rng, 128 // G)
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        err = np.abs(o[g["q_row0"] + rows] - want_o).max()
        worst = max(worst, err)
        assert err <= ATOL, f"segment {i}: max abs error {err}"
        assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL
    if also_materialised:
        _, o2, lse2 = c.attend_gpu(fused=False)  # now flushes the engine, then attends
        written = np.zeros(o.shape[0], bool)
        for g in w.segments:
            written[g["q_row0"]:g["q_row0"] + g["q_len"]] = True
        assert np.abs(o[written] - o2[written]).max() <= 1e-2
        assert np.abs(lse[written] - lse2[written]).max() <= 1e-3
    return worst


def test_fused_tiny_branch():
    fused_case(synth.tiny())


def test_fused_32k_trajectory_small():
    fused_case(synth.llama8b_32k(total=4096, n_new=300, fork=True))


def test_fused_half_layout_and_head_dim_64():
    w = synth.llama8b_32k(total=4096, n_new=200, n_layers=1, fork=True)
    w.shape.rope_layout = "half"
    fused_case(w)
    w = synth.tiny()
    w.shape.rope_layout = "half"
    fused_case(w)


def test_fused_shifts_inside_pages_and_hidden_spans():
    # repos spans that start and end mid-page (runs break inside a page) and shifts of both signs
    w = synth.tiny()
    w.ops = [("alloc", "A"), ("append", "A", 600, "ctx"), ("fork", "B", "A", 600),
             ("drop", "B", 37, 91), ("repos", "B", 91, 600, -54), ("repos", "B", 200, 333, 1000),
             ("repos", "B", 250, 257, -70000), ("append", "B", 150, "new")]
    w.n_pages = 128
    w.segments = [dict(seq="B", kv_end=750, q_len=150, hide=[(400, 417)], q_row0=0)]
    fused_case(w)


def test_fused_sessions_many_segments():
    w = synth.sessions_64k(n_layers=1, n_sessions=3, prefix=1024, per_session=8192, q_per_seg=128,
                           span_len=(64, 512))
    fused_case(w, k_rows=40)


def test_fused_without_pending_shift_equals_attend():
    from gpu_case import Case
    w = synth.tiny()
    c = Case(w)
    c.run_ops()
    c.flush_segments()                      # nothing left pending
    _, o1, l1 = c.attend_gpu(fused=True)
    _, o2, l2 = c.attend_gpu(fused=False)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("page", [16, 64, 128])
def test_fused_mla_spliced_session(page):
    # MLA: K_pe of the tokens after the spliced span rotated inside the pair kernel, the latent as stored
    import dataclasses
    w = synth.mla_dsv2lite(n_layers=1, concurrency=1, prompt=3000, span=700, stub=20, n_new=100)
    w.shape = dataclasses.replace(w.shape, page_size=page)
    w.n_pages = w.n_pages * 64 // page + 64  # the workload's pool is sized for 64-token pages
    fused_case(w)


def test_fused_mla_half_layout_and_sessions():
    import dataclasses
    w = synth.mla_dsv2lite(n_layers=1, concurrency=3, prompt=2500, span=600, stub=16, n_new=70)
    w.shape = dataclasses.replace(w.shape, rope_layout="half")
    fused_case(w)
