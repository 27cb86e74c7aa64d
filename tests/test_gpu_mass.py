"""akv_attention_mass on the GPU (the attn_mass kernel) against the float64 oracle.

Bar: per token, |gpu - oracle| <= 5e-3 * oracle + 1e-5 * q_len * Hq.  Each
probability enters as bf16 (relative rounding <= 2^-9) and comes from float32
scores and the attention pass's float32 lse; a sum of non-negative terms keeps
the relative bound, the small absolute floor covers tokens with almost no mass.
Tokens a segment does not see must be exactly 0; each segment's total is
q_len * Hq (every row's probabilities sum to one) within the same relative
bound."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import runner, synth

pytestmark = pytest.mark.gpu


def mass_case(w, split=0):
    from gpu_case import Case, bf16_of
    from oracle import attention, kernels
    c = Case(w)
    c.run_ops()
    c.flush_segments()
    s = w.shape
    q32, qd = c.queries()
    nq = q32.shape[0]
    o = torch.empty((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((nq, s.n_q_heads), dtype=torch.float32, device="cuda")
    segs = runner.engine_segments(w, c.names_e)
    c.eng.attend(0, segs, qd, nq, o, lse, s.scale, stream=c.stream)
    total = sum(g["kv_end"] for g in w.segments)
    mass = torch.full((total,), float("nan"), dtype=torch.float32, device="cuda")
    c.eng.set_attention_split(split)
    c.eng.attention_mass(0, segs, qd, nq, lse, mass, s.scale, stream=c.stream)
    torch.cuda.synchronize()
    assert c.eng.check_device_error(c.stream) == 0
    got = mass.cpu().numpy().astype(np.float64)
    off = 0
    for i, g in enumerate(w.segments):
        sid = c.names_o[g["seq"]]
        runs, kv_len = c.model.segment_runs(sid, g["kv_end"], g["q_len"], g["hide"])
        qb = bf16_of(q32[g["q_row0"]:g["q_row0"] + g["q_len"]])
        want_e = kernels.mass_segment(qb, c.kp, c.vp, 0, runs, s.scale)
        hidden = np.zeros(g["kv_end"], bool)
        for a, b in g["hide"]:
            hidden[a:b] = True
        st = c.model.state(sid)
        toks = [t for t in range(g["kv_end"]) if st["visible"][t] and not hidden[t]]
        assert len(toks) == kv_len
        want = np.zeros(g["kv_end"])
        want[toks] = want_e
        seg_got = got[off:off + g["kv_end"]]
        bound = 5e-3 * want + 1e-5 * g["q_len"] * s.n_q_heads
        assert np.all(np.abs(seg_got - want) <= bound), f"segment {i}: worst {np.max(np.abs(seg_got - want) / bound)}"
        unseen = np.ones(g["kv_end"], bool)
        unseen[toks] = False
        assert np.all(seg_got[unseen] == 0.0)
        n = g["q_len"] * s.n_q_heads
        assert abs(seg_got.sum() - n) <= 5e-3 * n
        off += g["kv_end"]


def test_mass_tiny_two_branches():
    mass_case(synth.tiny())


def test_mass_32k_trajectory_small():
    mass_case(synth.llama8b_32k(total=4096, n_new=300))


def test_mass_partial_pages_and_hidden_span():
    w = synth.tiny()
    ops = [("alloc", "A"), ("append", "A", 900, "ctx")]
    for a in range(5, 800, 41):
        ops.append(("drop", "A", a, a + 13))
    ops.append(("append", "A", 200, "new"))
    w.ops = ops
    w.n_pages = 128
    w.segments = [dict(seq="A", kv_end=1100, q_len=200, hide=[(300, 333)], q_row0=0)]
    mass_case(w)


def test_mass_sessions_many_segments_group_8():
    w = synth.llama70b_128k(n_layers=1, total=8192, n_branches=3, q_per_branch=130)
    mass_case(w)


@pytest.mark.parametrize("split", [1, 2, 3, 8])
def test_mass_forced_k_ranges(split):
    mass_case(synth.llama8b_32k(total=4096, n_new=300), split=split)
