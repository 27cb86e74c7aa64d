"""akv_tree_reuse on the GPU: a retrigger match rotates the holder's keys into
copy-on-write pages (the repos_rotate kernel), an exact match shares them.
Bars as in the repos tests (rotated-key rule, everything else bit-identical);
the oracle replays the same fork / reposition / flush on its own pools."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


def test_retrigger_reuse_rotates_into_copy_on_write_pages():
    from gpu_case import Case
    from test_gpu_repos import compare_rotated, rotated_mask
    w = synth.tiny()
    w.ops = [("alloc", "A"), ("append", "A", 300, "ctx")]
    w.n_pages = 128
    w.segments = []
    c = Case(w)
    c.run_ops()
    a = c.names_e["A"]
    path = [("tok", 1000 + i, i) for i in range(300)]
    holder = c.eng.tree_insert(path, a)
    assert holder == c.model.seq_fork(a, 300)
    # the request: the same 300 tokens two thousand positions further on, and 20 more
    req = [("tok", 1000 + i, 2000 + i) for i in range(320)]
    m, new = c.eng.tree_reuse(req, stream=c.stream)
    assert m == dict(kind="retrigger", seq=holder, n_items=300, n_tokens=300)
    b = c.model.seq_fork(holder, 300)
    assert new == b
    c.model.repos(b, 0, 300, 2000)
    c._apply_runs(c.model.flush([b]))
    kg, vg = c.gpu_pools()
    assert np.array_equal(vg, c.vp)                         # values stay shared
    compare_rotated(kg, c.kp, rotated_mask(c, c.flush_runs), c.kterm)
    st = c.eng.export_state(new)
    assert np.array_equal(st["pos"], np.arange(2000, 2300))
    # the holder still has its own pages and positions
    assert np.array_equal(c.eng.export_state(holder)["pos"], np.arange(300))
    # an exact request shares the holder's pages without a kernel
    m2, new2 = c.eng.tree_reuse(path[:100], stream=c.stream)
    assert m2["kind"] == "exact"
    assert np.array_equal(c.eng.export_state(new2)["k_page"], c.eng.export_state(holder)["k_page"][:100])
    assert c.eng.check_device_error(c.stream) == 0
