"""repos_rotate and kv_write on the GPU against the oracle.

Bar (see the tolerance reading for rotated keys): every rotated bf16 value is
within one bf16 ulp of RNE_bf16(float64 rotation) and at least 99.9% are
bit-identical (only near-ties may differ, because the kernel rotates in
float32); every row a flush does not rotate, and every V / latent row, is
bit-identical.  kv_write is a pure copy: bit-exact."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth
from oracle import bf16

pytestmark = pytest.mark.gpu


def compare_rotated(gpu, want, rows_mask):
    """gpu/want float32 pools holding bf16 values; rows_mask marks rotated rows (broadcast over d)."""
    g, w_ = gpu[rows_mask], want[rows_mask]
    ulp = bf16.ulp_bf16(w_)
    diff = np.abs(g.astype(np.float64) - w_.astype(np.float64))
    assert np.all(diff <= ulp), f"max diff {diff.max()} vs ulp"
    eq = np.mean(g == w_)
    assert eq >= 0.999, f"bit-equal fraction {eq}"
    rest_g, rest_w = gpu[~rows_mask], want[~rows_mask]
    assert np.array_equal(rest_g, rest_w)
    return eq


def rotated_mask(case, runs):
    s = case.w.shape
    m = np.zeros(case.kp.shape[:4], bool)
    for src, dst, lo, hi, d in runs:
        m[:, dst, :, lo:hi] = True
    return m


def run_case(w):
    from gpu_case import Case
    c = Case(w)
    c.run_ops()
    kg, vg = c.gpu_pools()
    assert np.array_equal(kg, c.kp), "K pool after appends / explicit flushes"
    assert np.array_equal(vg, c.vp), "V pool after appends"
    runs = c.flush_segments()
    kg, vg = c.gpu_pools()
    assert np.array_equal(vg, c.vp)
    eq = compare_rotated(kg, c.kp, rotated_mask(c, runs))
    assert c.eng.check_device_error() == 0
    return c, runs, eq


def test_tiny_branch_copy_on_write():
    c, runs, eq = run_case(synth.tiny())
    assert len(runs) == 8 and all(r[0] != r[1] and r[4] == -64 for r in runs)


def test_llama8b_32k_single_layer_full_size():
    c, runs, eq = run_case(synth.llama8b_32k())
    assert sum(r[3] - r[2] for r in runs) > 15000


def test_llama8b_32k_fork_branch_copy_on_write():
    c, runs, eq = run_case(synth.llama8b_32k(total=8192, n_new=256, n_layers=2, fork=True))
    assert all(r[0] != r[1] for r in runs)


def test_mla_splice_rotates_k_pe_only():
    c, runs, eq = run_case(synth.mla_dsv2lite(n_layers=3, concurrency=4))
    assert {r[4] for r in runs} == {-1984}


def test_sessions_shifts_of_both_signs():
    w = synth.sessions_64k(n_layers=2, n_sessions=3, prefix=1024, per_session=8192, q_per_seg=128,
                           span_len=(64, 512))
    c, runs, eq = run_case(w)
    ds = {r[4] for r in runs}
    assert min(ds) < 0 < max(ds)


def test_llama70b_sweep_large_shifts():
    # explicit in-place sweep with |delta| up to 64K (the fp64 angle table matters here)
    c, runs, eq = run_case(synth.llama70b_128k(n_layers=2, total=16384, n_branches=4, q_per_branch=128))


def test_half_layout_and_head_dim_64():
    w = synth.llama8b_32k(total=4096, n_new=64, n_layers=2)
    w.shape.rope_layout = "half"
    run_case(w)
    w = synth.tiny()
    w.shape.rope_layout = "half"
    run_case(w)


def test_zero_shift_is_identity_bitwise():
    from gpu_case import Case
    w = synth.tiny()
    w.ops = [("alloc", "A"), ("append", "A", 100, "x"), ("fork", "B", "A", 100), ("repos", "B", 10, 90, 7),
             ("repos", "B", 10, 90, -7), ("repos", "B", 20, 30, 1)]
    w.segments = [dict(seq="B", kv_end=100, q_len=1, hide=[], q_row0=0)]
    c = Case(w)
    c.run_ops()
    runs = c.flush_segments()
    kg, _ = c.gpu_pools()
    assert np.array_equal(kg, c.kp)   # delta 0 copies (cos 1, sin 0) are exact
    assert any(r[4] == 0 for r in runs)
