"""Bounded waits of the attention kernel, on the GPU.

Every device-side wait of segment_batch_attn gives up after a time limit,
records AKV_ERR_DEVICE_TIMEOUT, drains its copies and tensor-core work, frees
its TMEM and exits.  Here the copy-issuing threads are capped (a test hook) so
that the waits for the K/V copies they never issue run out after 20 ms, at
three points of a launch: before any copy, with the first MMAs in flight, and
mid-stream -- for the GQA kernel on the tiny two-branch launch, and for the MLA
pair kernel (plain and fused rotation) on a small spliced session.  Each launch must report the time-out, leave
the pools as they were (attention only reads them), and leave the context
usable: with the hook removed the next launch matches the float64 oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import akv, synth

pytestmark = pytest.mark.gpu

TIMEOUT = 7  # AKV_ERR_DEVICE_TIMEOUT


def test_wait_runs_out_reports_timeout_and_context_recovers():
    from gpu_case import Case
    from test_gpu_attention import ATOL
    w = synth.tiny()
    c = Case(w)
    c.run_ops()
    c.flush_segments()                 # materialise now: the launches below only read the pools
    kg0, vg0 = c.gpu_pools()
    s = w.shape
    q32, qd = c.queries()
    nq = q32.shape[0]
    segs = None
    from agentic_kv_cache_gb300 import runner
    segs = runner.engine_segments(w, c.names_e)
    for cap in (0, 1, 3):
        c.eng.debug_wait_limit(20_000_000, cap)
        o = torch.zeros((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
        c.eng.attend(0, segs, qd, nq, o, None, s.scale, stream=c.stream)
        assert c.eng.check_device_error(c.stream) == TIMEOUT, cap
        assert c.eng.check_device_error(c.stream) == 0       # the word is cleared by reading it
        kg, vg = c.gpu_pools()
        assert np.array_equal(kg, kg0) and np.array_equal(vg, vg0)
    c.eng.debug_wait_limit(0, -1)
    q32, o, lse = c.attend_gpu()
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"])
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        assert np.abs(o[g["q_row0"] + rows] - want_o).max() <= ATOL
        assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL


def test_wait_limit_hook_rejects_bad_cap():
    from gpu_case import Case
    c = Case(synth.tiny())
    with pytest.raises(akv.AKVError):
        c.eng.debug_wait_limit(0, -2)


@pytest.mark.parametrize("fused", [False, True])
def test_mla_wait_runs_out_reports_timeout_and_context_recovers(fused):
    # the MLA pair kernel: copy threads capped at 0, 1 and 3 ring rounds, so the MMA threads' and the
    # rotation warps' waits run out; the launch reports the time-out, drains, and the next launch
    # (hook removed) matches the oracle
    from gpu_case import Case
    from test_gpu_attention import ATOL
    w = synth.mla_dsv2lite(n_layers=1, concurrency=1, prompt=2000, span=500, stub=16, n_new=60)
    c = Case(w)
    c.run_ops()
    if not fused:
        c.flush_segments()
    kg0, vg0 = c.gpu_pools()
    s = w.shape
    q32, qd = c.queries()
    nq = q32.shape[0]
    from agentic_kv_cache_gb300 import runner
    segs = runner.engine_segments(w, c.names_e)
    for cap in (0, 1, 3):
        c.eng.debug_wait_limit(20_000_000, cap)
        o = torch.zeros((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
        c.eng.attend(0, segs, qd, nq, o, None, s.scale, stream=c.stream, fused=fused)
        assert c.eng.check_device_error(c.stream) == TIMEOUT, cap
        assert c.eng.check_device_error(c.stream) == 0
        kg, vg = c.gpu_pools()
        assert np.array_equal(kg, kg0) and np.array_equal(vg, vg0)
    c.eng.debug_wait_limit(0, -1)
    if fused:
        c.flush_segments(engine=False)   # oracle keys at the composed positions; the engine keeps them pending
    q32, o, lse = c.attend_gpu(fused=fused)
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"])
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        assert np.abs(o[g["q_row0"] + rows] - want_o).max() <= ATOL
        assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL
