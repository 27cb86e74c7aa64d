"""repos_rotate and kv_write on the GPU against the oracle.

Bars (the tolerance reading for rotated keys):
* bf16 in the pool: every rotated value is within one bf16 ulp of
  RNE_bf16(float64 rotation) plus the float32 rounding allowance of the
  rotation, 2^-20 (|x_a| + |x_b|) of its input pair (which only matters where
  the result cancels towards zero), and at least 99.9% are bit-identical;
* the float32 debug mode of the same kernel meets the stated rotated-key
  tolerance against float64: |err| <= 2e-3 + 1e-3 |ref|;
* every row a flush does not rotate, and every V / latent row, is
  bit-identical; kv_write is a pure copy: bit-exact."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth
from oracle import bf16

pytestmark = pytest.mark.gpu


def compare_rotated(gpu, want, rows_mask, term):
    """gpu/want float32 pools holding bf16 values; rows_mask marks rotated rows (broadcast over d);
    term: the float32 rounding allowance per element."""
    rest_g, rest_w = gpu[~rows_mask], want[~rows_mask]
    assert np.array_equal(rest_g, rest_w)
    if not rows_mask.any():
        return 1.0
    g, w_ = gpu[rows_mask], want[rows_mask]
    bound = bf16.ulp_bf16(w_) + term[rows_mask]
    diff = np.abs(g.astype(np.float64) - w_.astype(np.float64))
    assert np.all(diff <= bound), f"worst diff / bound {np.max(diff / bound)}"
    eq = np.mean(g == w_)
    assert eq >= 0.999, f"bit-equal fraction {eq}"
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
    compare_rotated(kg, c.kp, rotated_mask(c, c.flush_runs), c.kterm)   # appends + explicit flushes
    assert np.array_equal(vg, c.vp), "V pool after appends"
    runs = c.flush_segments()
    kg, vg = c.gpu_pools()
    assert np.array_equal(vg, c.vp)
    eq = compare_rotated(kg, c.kp, rotated_mask(c, c.flush_runs), c.kterm)
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


@pytest.mark.parametrize("layout", ["interleaved", "half"])
def test_f32_debug_mode_meets_rotated_key_tolerance(layout):
    # The pre-flush pool of the 32K trajectory, every flush run of the turn plus
    # shifts up to +-64K, rotated without rounding and compared with float64.
    from gpu_case import Case
    from oracle import rope
    w = synth.llama8b_32k(total=8192, n_new=128, n_layers=2)
    w.shape.rope_layout = layout
    c = Case(w)
    c.run_ops()
    ids = sorted({c.names_o[g["seq"]] for g in w.segments})
    import copy
    runs = copy.deepcopy(c.model).flush(ids)
    rng = np.random.default_rng(5)
    req = [(src, lo, hi, d) for src, dst, lo, hi, d in runs]
    req += [(int(rng.integers(0, 40)), 0, 16, int(rng.integers(-65536, 65537))) for _ in range(32)]
    req = np.array(req, np.int32)
    n_rows = int((req[:, 2] - req[:, 1]).sum())
    s = w.shape
    out = torch.empty((s.n_layers, n_rows, s.n_kv_heads, s.d_rot), dtype=torch.float32, device="cuda")
    c.eng.debug_rotate_f32(req, out, stream=c.stream)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = np.concatenate([rope.repos(c.kp[:, pg, :, lo:hi, :].transpose(0, 2, 1, 3),
                                      np.full((s.n_layers, hi - lo, s.n_kv_heads), d, np.float64),
                                      s.rope_base, layout) for pg, lo, hi, d in req], axis=1)
    err = np.abs(got - want)
    assert np.all(err <= 2e-3 + 1e-3 * np.abs(want)), err.max()
    assert err.max() < 1e-5          # float32 rotation: far inside the tolerance
    kg, _ = c.gpu_pools()
    assert np.array_equal(kg, c.kp)  # the debug mode only reads the pool


def test_one_flush_of_two_sharers_copies_before_rotating_in_place():
    # attend flushes both branches in one call: each shared page is copied out (copy-on-write,
    # rotated for A) and then rotated in place for B, its last holder; the copies must read the
    # page before the in-place rotation writes it
    from gpu_case import Case
    from test_bookkeeping_parity import shared_prefix_both_shifted
    from test_gpu_attention import ATOL
    w = shared_prefix_both_shifted()
    c = Case(w)
    c.run_ops()
    runs = c.flush_segments(engine=False)  # the oracle's flush; the engine's runs inside attend
    assert {r[0] for r in runs if r[0] != r[1]} & {r[1] for r in runs if r[0] == r[1]}
    q32, o, lse = c.attend_gpu()
    kg, vg = c.gpu_pools()
    compare_rotated(kg, c.kp, rotated_mask(c, c.flush_runs), c.kterm)
    assert np.array_equal(vg, c.vp)
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"])
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        assert np.abs(o[g["q_row0"] + rows] - want_o).max() <= ATOL
        assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL
