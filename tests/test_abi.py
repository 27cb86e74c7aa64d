"""The C ABI library loads, exports every symbol include/akv.h declares, and
rejects bad arguments with a status (no GPU needed: metadata-only contexts)."""
import ctypes
import os
import re

import pytest

from agentic_kv_cache_gb300 import akv, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    build.build()
    return akv.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "akv.h")).read()
    return sorted(set(re.findall(r"^AKV_API\s+[\w\s\*]+?\b(akv_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    raw = ctypes.CDLL(akv.LIB_PATH)
    for n in names:
        getattr(raw, n)


def cfg(**kw):
    c = dict(layout=0, n_layers=2, n_q_heads=8, n_kv_heads=2, d_rot=64, d_v=64, page_size=16, n_pages=32,
             rope_layout=0, rope_base=1e4)
    c.update(kw)
    return c


@pytest.mark.parametrize("bad", [dict(page_size=24), dict(n_q_heads=6, n_kv_heads=4), dict(d_rot=63, d_v=63),
                                 dict(layout=1), dict(rope_base=-1.0), dict(n_pages=0), dict(d_v=128),
                                 dict(n_q_heads=384, n_kv_heads=1)])
def test_bad_configs_are_rejected(lib, bad):
    with pytest.raises(akv.AKVError) as e:
        akv.Engine(cfg(**bad))
    assert e.value.code == "ARG"


def test_errors_leave_state_unchanged(lib):
    e = akv.Engine(cfg(n_pages=4))
    s = e.seq_alloc()
    e.append(s, 60)
    before = (e.export_state(s), e.refcounts())
    for call, code in [(lambda: e.append(s, 10), "NO_PAGES"), (lambda: e.drop(s, 5, 61), "RANGE"),
                       (lambda: e.repos(s, 0, 10, 2 ** 31 - 5), "OVERFLOW"), (lambda: e.seq_free(7), "ARG"),
                       (lambda: e.repos(s, 9, 3, 1), "RANGE"), (lambda: e.splice(s, 0, 1, 100), "NO_PAGES")]:
        with pytest.raises(akv.AKVError) as x:
            call()
        assert x.value.code == code
    after = (e.export_state(s), e.refcounts())
    for k in before[0]:
        assert (before[0][k] == after[0][k]).all()
    assert (before[1][0] == after[1][0]).all() and (before[1][1] == after[1][1]).all()


def test_edit_list_is_all_or_nothing_and_equals_single_calls(lib):
    # akv_edit: a turn's drop / repos list in one call; a failing entry anywhere leaves every
    # earlier entry unapplied (overflow needs the saved-state path: the bound is near int32)
    e = akv.Engine(cfg(n_pages=16))
    s = e.seq_alloc()
    e.append(s, 100)
    e.repos(s, 0, 100, 2 ** 31 - 200)          # positions near the int32 limit
    before = e.export_state(s)
    bad = [[("drop", 10, 20), ("repos", 20, 50, 3), ("drop", 5, 101)],               # span outside
           [("repos", 0, 10, -4), ("drop", 30, 40), ("repos", 50, 60, 150)],         # overflow
           [("drop", 1, 2), ("bogus", 1, 2)]]                                        # unknown kind
    for ops, code in zip(bad, ["RANGE", "OVERFLOW", "ARG"]):
        with pytest.raises(akv.AKVError) as x:
            e.edit(s, ops)
        assert x.value.code == code
        after = e.export_state(s)
        for k in before:
            assert (before[k] == after[k]).all(), (code, k)
    # the same list through akv_edit and through single calls gives the same state
    ops = [("drop", 10, 20), ("repos", 20, 100, -10), ("drop", 40, 45), ("repos", 50, 100, 7), ("repos", 0, 5, -3)]
    a, b = akv.Engine(cfg(n_pages=16)), akv.Engine(cfg(n_pages=16))
    for eng in (a, b):
        eng.append(eng.seq_alloc(), 100)
    a.edit(0, ops)
    for op in ops:
        (b.drop(0, *op[1:]) if op[0] == "drop" else b.repos(0, *op[1:]))
    sa, sb = a.export_state(0), b.export_state(0)
    for k in sa:
        assert (sa[k] == sb[k]).all(), k


def test_segment_validation(lib):
    e = akv.Engine(cfg())
    s = e.seq_alloc()
    e.append(s, 100)
    e.drop(s, 95, 97)
    with pytest.raises(akv.AKVError) as x:
        e.segment_runs(dict(seq=s, kv_end=100, q_len=8))     # a dropped query token
    assert x.value.code == "ARG"
    with pytest.raises(akv.AKVError) as x:
        e.segment_runs(dict(seq=s, kv_end=101, q_len=1))
    assert x.value.code == "RANGE"
    with pytest.raises(akv.AKVError) as x:
        e.segment_runs(dict(seq=s, kv_end=90, q_len=4, hide=[10, 95]))
    assert x.value.code == "RANGE"
    runs, n = e.segment_runs(dict(seq=s, kv_end=94, q_len=4, hide=[10, 20]))
    assert n == 84


def test_metadata_only_attend_plans_without_device(lib):
    e = akv.Engine(cfg())
    s = e.seq_alloc()
    e.append(s, 64)
    e.repos(s, 10, 64, -3)
    e.attend(0, [dict(seq=s, kv_end=64, q_len=4)], None, 4, None)   # flushes; no data touched
    assert (e.export_state(s)["delta"] == 0).all()
    assert len(e.last_flush_runs()) == 4


def test_checked_build_exports_every_symbol_and_plain_build_refuses_the_hook(lib):
    # the -DAKV_CHECKED variant (device-side descriptor checks) builds and exports the same ABI;
    # its corruption hook is refused by the plain library
    path = build.build(checked=True)
    raw = ctypes.CDLL(path)
    for n in declared_symbols():
        getattr(raw, n)
    eng = akv.Engine(cfg(), None)
    with pytest.raises(akv.AKVError) as e:
        eng.debug_corrupt(1)
    assert e.value.code == "ARG"
