"""Host buffers through the C ABI: inputs staged into library memory on the
library's copy stream (ahead of the caller's stream, which waits for each
copy), outputs copied back on the caller's stream -- or, with an output stream
set (akv_set_output_stream), on that stream, overlapping the next turn.

Post-drop turns run back to back on one stream with no synchronisation
between them, as a serving loop runs them: every turn forks the trajectory,
edits the branch, appends its own new K/V and attends with its own queries,
all from host buffers (pinned, and pageable for one turn's queries), writing
its output and lse to its own pinned host buffers.  After one synchronisation
each turn's output and lse must be bit-identical to the same turn run with
device buffers (same kernels, same plans), so no turn read another turn's
staged inputs.  The attention-mass pass from host buffers must match the
device-buffer pass up to the order of its float atomics."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import akv, runner, synth

pytestmark = pytest.mark.gpu

N_TURNS = 4


class Side:
    """One engine with its own pools, the trajectory's shared history already appended."""

    def __init__(self, w, src, setup_ops):
        self.cfg = akv.config_from_shape(w.shape, w.n_pages)
        self.pools = akv.make_pools(self.cfg)
        self.eng = akv.Engine(self.cfg, self.pools)
        self.stream = torch.cuda.current_stream()
        self.names = runner.run_ops(self.eng, w, kv_source=src, ops=setup_ops, stream=self.stream)


@pytest.mark.parametrize("out_stream", [False, True])
def test_back_to_back_host_turns_match_device_turns(out_stream):
    w = synth.llama8b_32k(total=4096, n_new=300, fork=True)
    s = w.shape
    fork_at = next(i for i, op in enumerate(w.ops) if op[0] == "fork")
    setup_ops, step_ops = w.ops[:fork_at], w.ops[fork_at:]
    new_op = next(op for op in step_ops if op[0] == "append")
    src = runner.torch_kv_source(w)
    k0, v0 = src(new_op[3], new_op[2])
    q0 = torch.from_numpy(synth.q_array(w)).cuda().to(torch.bfloat16)
    nq = q0.shape[0]
    # each turn its own inputs (scaled copies, so a stale staging buffer would show in the output)
    ks = [(k0.float() * (1 + t / 8)).to(torch.bfloat16) for t in range(N_TURNS)]
    vs = [(v0.float() * (1 - t / 16)).to(torch.bfloat16) for t in range(N_TURNS)]
    qs = [(q0.float() * (1 + t / 4)).to(torch.bfloat16) for t in range(N_TURNS)]
    h_k = [x.cpu().pin_memory() for x in ks]
    h_v = [x.cpu().pin_memory() for x in vs]
    h_q = [x.cpu().pin_memory() for x in qs]
    h_q[2] = qs[2].view(torch.int16).cpu().numpy()  # pageable host memory for one turn's queries
    h_o = [torch.empty((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16).pin_memory() for _ in range(N_TURNS)]
    h_lse = [torch.empty((nq, s.n_q_heads), dtype=torch.float32).pin_memory() for _ in range(N_TURNS)]

    dev = Side(w, src, setup_ops)
    host = Side(w, src, setup_ops)
    if out_stream:
        copy_back = torch.cuda.Stream()
        host.eng.set_output_stream(copy_back)
    torch.cuda.synchronize()

    def turn(side, t, k, v, q, o, lse):
        names = runner.run_ops(side.eng, w, kv_source=lambda *_: (k, v), ops=step_ops, names=dict(side.names),
                               stream=side.stream)
        segs = runner.engine_segments(w, names)
        side.eng.attend(0, segs, q, nq, o, lse, s.scale, stream=side.stream)
        return names, segs

    want_o, want_lse = [], []
    for t in range(N_TURNS):
        o = torch.empty((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((nq, s.n_q_heads), dtype=torch.float32, device="cuda")
        names, _ = turn(dev, t, ks[t], vs[t], qs[t], o, lse)
        dev.eng.seq_free(names["F"])
        want_o.append(o)
        want_lse.append(lse)
    for t in range(N_TURNS):  # no synchronisation between the turns
        names, _ = turn(host, t, h_k[t], h_v[t], h_q[t], h_o[t], h_lse[t])
        host.eng.seq_free(names["F"])
    torch.cuda.synchronize()
    assert dev.eng.check_device_error(dev.stream) == 0
    assert host.eng.check_device_error(host.stream) == 0
    for t in range(N_TURNS):
        assert torch.equal(h_o[t], want_o[t].cpu()), f"turn {t}: output differs"
        assert torch.equal(h_lse[t], want_lse[t].cpu()), f"turn {t}: lse differs"
    # distinct inputs gave distinct outputs (the comparison above is not vacuous)
    assert not torch.equal(h_o[0], h_o[1])

    # the attention-mass pass of one more turn, from host Q / lse into a host output
    names_d, segs_d = turn(dev, 0, ks[3], vs[3], qs[3], want_o[0], want_lse[0])
    names_h, segs_h = turn(host, 0, h_k[3], h_v[3], h_q[3], h_o[0], h_lse[0])
    total = sum(g["kv_end"] for g in w.segments)
    m_dev = torch.empty((total,), dtype=torch.float32, device="cuda")
    dev.eng.attention_mass(0, segs_d, qs[3], nq, want_lse[0], m_dev, s.scale, stream=dev.stream)
    # the host lse is an output of the attend above: a host input must be final when the call is
    # made (it is read on the copy stream, not in the caller's stream order), so synchronise first
    torch.cuda.synchronize()
    m_host = np.full((total,), np.nan, np.float32)
    host.eng.attention_mass(0, segs_h, h_q[3], nq, h_lse[0], m_host, s.scale, stream=host.stream)
    torch.cuda.synchronize()
    assert host.eng.check_device_error(host.stream) == 0
    np.testing.assert_allclose(m_host, m_dev.cpu().numpy(), rtol=1e-5, atol=1e-6)
    assert abs(float(m_host.sum()) - nq * s.n_q_heads) <= 5e-3 * nq * s.n_q_heads
