"""Randomised segment_batch_attn workloads against the float64 oracle (and,
for GQA, the fused-rotation path on histories with pending shifts and the
attention-mass pass).

Each case draws a small cache history (prompt, drops, repositions, a splice, a
fork with its own edits, new tokens on both branches, hidden spans) for GQA
(group 4 or 8, head dim 64 or 128, page 16 or 32) or MLA (page 16, 64 or
128), and a split-KV factor (automatic or forced), then compares every query
row with the oracle (bf16 output within 2e-2, lse within 2e-2)."""
import dataclasses

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 2e-2


def random_workload(seed, mla, force_repos=False):
    rng = np.random.default_rng(9100 + seed)
    if mla:
        w = synth.mla_dsv2lite(n_layers=1, concurrency=1)
        w.shape = dataclasses.replace(w.shape, page_size=int(rng.choice([16, 64, 128])))
    else:
        w = synth.tiny()
        d = int(rng.choice([64, 128]))
        g = int(rng.choice([4, 8]))
        w.shape = dataclasses.replace(w.shape, n_q_heads=2 * g, n_kv_heads=2, d_rot=d, d_v=d,
                                      page_size=int(rng.choice([16, 32])))
    n_a = int(rng.integers(40, 1500))
    ops = [("alloc", "A"), ("append", "A", n_a, "pA")]
    length = {"A": n_a}
    key = [0]

    def span(n, lo=0):
        a = int(rng.integers(lo, max(lo + 1, n)))
        return a, int(rng.integers(a, n + 1))

    def edits(seq, n_edits):
        for _ in range(n_edits):
            n = length[seq]
            kind = rng.choice(["drop", "repos", "splice"], p=[0.45, 0.4, 0.15])
            s, e = span(n)
            if kind == "drop":
                ops.append(("drop", seq, s, e))
            elif kind == "repos":
                ops.append(("repos", seq, s, e, int(rng.integers(-3000, 3000))))
            else:
                stub = int(rng.integers(0, 40))
                key[0] += 1
                ops.append(("splice", seq, s, e, stub, f"st{key[0]}"))
                length[seq] = n - (e - s) + stub

    edits("A", int(rng.integers(0, 6)))
    if force_repos:  # at least one pending shift on A
        a = int(rng.integers(0, length["A"]))
        ops.append(("repos", "A", a, int(rng.integers(a + 1, length["A"] + 1)), int(rng.choice([-1, 1])) *
                    int(rng.integers(1, 3000))))
    fork_at = int(rng.integers(1, length["A"] + 1))
    ops.append(("fork", "B", "A", fork_at))
    length["B"] = fork_at
    edits("B", int(rng.integers(0, 6)))
    segs, row = [], 0
    for seq in ("A", "B"):
        q = int(rng.integers(1, 160))
        key[0] += 1
        ops.append(("append", seq, q, f"n{key[0]}"))
        n_hist = length[seq]
        length[seq] += q
        hide = []
        if n_hist > 2 and rng.random() < 0.5:
            hide = [span(n_hist)]
        segs.append(dict(seq=seq, kv_end=length[seq], q_len=q, hide=hide, q_row0=row))
        row += q
    w.ops, w.segments = ops, segs
    page = w.shape.page_size
    w.n_pages = 4 * (sum(length.values()) // page + 8) + 64
    return w


def check_all_rows(w, split):
    from gpu_case import Case
    c = Case(w)
    c.run_ops()
    c.flush_segments()
    c.eng.set_attention_split(split)
    q32, o, lse = c.attend_gpu()
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"])
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        got_o = o[g["q_row0"] + rows]
        got_lse = lse[g["q_row0"] + rows]
        err = np.abs(got_o - want_o).max()
        assert err <= ATOL, f"segment {i}: max abs error {err}"
        assert np.abs(got_lse - want_lse).max() <= ATOL


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("mla", [False, True])
def test_random_workloads_match_oracle(seed, mla):
    w = random_workload(seed, mla)
    split = 0 if seed % 2 == 0 else int(np.random.default_rng(seed).integers(2, 6))
    check_all_rows(w, split)


@pytest.mark.parametrize("seed", range(8))
def test_random_fused_histories_match_oracle(seed):
    from test_gpu_fused import fused_case
    fused_case(random_workload(100 + seed, False, force_repos=True))


@pytest.mark.parametrize("seed", range(4))
def test_random_fused_mla_histories_match_oracle(seed):
    from test_gpu_fused import fused_case
    fused_case(random_workload(300 + seed, True, force_repos=True))


@pytest.mark.parametrize("seed", range(8))
def test_random_histories_attention_mass(seed):
    from test_gpu_mass import mass_case
    mass_case(random_workload(200 + seed, False))
