"""The checked build (libakv_checked.so, -DAKV_CHECKED) on the GPU.

Every kernel of that build checks the descriptors it reads before touching
memory: pages inside the pool, row ranges inside a page, segments and runs
inside their tables, query rows inside Q.  A failed check records
AKV_ERR_DEVICE in the device error word and skips the named work (attention:
the CTA returns before any barrier or TMEM use); nothing traps.

The outer test runs, in a child process with AKV_CHECKED=1 (so the binding
loads the checked library), a parity subset of the other GPU tests -- the
checks must not fire on valid descriptors -- and the inner tests below, which
corrupt one descriptor after host validation through akv_debug_corrupt.  The
corruptions are chosen so that even an unchecked kernel would stay inside its
buffers (a row range ending one row past a low page; a K page id equal to the
pool size, which a TMA load reads as zero fill), so no case can fault."""
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEVICE = 8  # AKV_ERR_DEVICE
inner = pytest.mark.skipif(os.environ.get("AKV_CHECKED", "") != "1", reason="runs in the checked child process")


@pytest.mark.skipif(os.environ.get("AKV_CHECKED", "") == "1", reason="the parent of the checked child process")
def test_checked_build_parity_subset_and_corrupt_descriptors():
    env = dict(os.environ, AKV_CHECKED="1")
    cases = ["tests/test_gpu_checked.py::test_inner_corrupt_flush_run_is_skipped_and_reported",
             "tests/test_gpu_checked.py::test_inner_corrupt_attention_run_is_refused_then_context_recovers",
             "tests/test_gpu_repos.py::test_tiny_branch_copy_on_write",
             "tests/test_gpu_repos.py::test_mla_splice_rotates_k_pe_only",
             "tests/test_gpu_repos.py::test_one_flush_of_two_sharers_copies_before_rotating_in_place",
             "tests/test_gpu_attention.py::test_tiny_two_branches_one_launch",
             "tests/test_gpu_attention.py::test_partial_pages_everywhere",
             "tests/test_gpu_attention.py::test_mla_small_full_compare",
             "tests/test_gpu_attention.py::test_split_kv_many_segments_group_8",
             "tests/test_gpu_compact.py::test_compact_tiny_branch",
             "tests/test_gpu_mass.py::test_mass_tiny_two_branches"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu"] + cases,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    import re
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= len(cases) and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-500:]


def in_place_case():
    """One sequence, a repos of [64, 256) by -64 flushed in place (no copy-on-write): the flush's
    first run is the first run the oracle lists."""
    w = synth.tiny()
    w.ops = [("alloc", "A"), ("append", "A", 256, "ctx"), ("repos", "A", 64, 256, -64), ("append", "A", 16, "new")]
    w.segments = [dict(seq="A", kv_end=272, q_len=16, hide=[], q_row0=0)]
    return w


@inner
def test_inner_corrupt_flush_run_is_skipped_and_reported():
    from agentic_kv_cache_gb300 import akv
    from gpu_case import Case
    assert akv.LIB_PATH.endswith("libakv_checked.so")
    w = in_place_case()
    c = Case(w)
    c.run_ops()
    before, _ = c.gpu_pools()
    sid = c.names_o["A"]
    runs = c.model.flush([sid])
    assert all(r[0] == r[1] for r in runs) and len(runs) > 2
    c.eng.debug_corrupt(1)
    c.eng.flush(sid, stream=c.stream)
    assert c.eng.check_device_error(c.stream) == DEVICE
    kg, _ = c.gpu_pools()
    src, dst, lo, hi, d = runs[0]
    assert np.array_equal(kg[:, dst, :, lo:hi], before[:, dst, :, lo:hi])   # the corrupt run wrote nothing
    # every other run rotated as the oracle rotates it (rows of the first run stay as appended)
    from test_gpu_repos import compare_rotated, rotated_mask
    c._apply_runs(runs[1:])
    compare_rotated(kg, c.kp, rotated_mask(c, runs[1:]), c.kterm)


@inner
def test_inner_corrupt_attention_run_is_refused_then_context_recovers():
    from agentic_kv_cache_gb300 import runner
    from gpu_case import Case
    from test_gpu_attention import ATOL
    w = synth.tiny()
    c = Case(w)
    c.run_ops()
    c.flush_segments()
    s = w.shape
    q32, qd = c.queries()
    nq = q32.shape[0]
    o = torch.zeros((nq, s.n_q_heads, s.d_v), dtype=torch.bfloat16, device="cuda")
    c.eng.debug_corrupt(2)
    c.eng.attend(0, runner.engine_segments(w, c.names_e), qd, nq, o, None, s.scale, stream=c.stream)
    assert c.eng.check_device_error(c.stream) == DEVICE
    q32, o, lse = c.attend_gpu()
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"])
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        assert np.abs(o[g["q_row0"] + rows] - want_o).max() <= ATOL
        assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL
