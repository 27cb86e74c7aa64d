"""The engine's bookkeeping (metadata-only context, no GPU) must equal the
oracle's independent model bit for bit: per-token page map, slots, positions,
pending shifts, visibility, page reference counts, flush run lists and segment
run lists, and the status of every rejected operation."""
import numpy as np
import pytest

from agentic_kv_cache_gb300 import akv, build, runner, synth
from oracle.cache import CacheError, CacheModel
from drive import oracle_model, oracle_run_ops


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def engine_for(w):
    return akv.Engine(akv.config_from_shape(w.shape, w.n_pages))


def assert_same_state(eng, model, names_e, names_o):
    for name in names_e:
        if names_o[name] not in model.seqs:
            continue
        a = eng.export_state(names_e[name])
        b = model.state(names_o[name])
        for k in ("k_page", "v_page", "slot", "pos", "delta", "visible"):
            assert np.array_equal(a[k], np.asarray(b[k], np.int32)), (name, k)
    ke, ve = eng.refcounts()
    ko, vo = model.refcounts()
    assert np.array_equal(ke, ko) and np.array_equal(ve, vo)


WORKLOADS = [
    ("tiny", lambda: synth.tiny()),
    ("llama8b_32k", lambda: synth.llama8b_32k()),
    ("llama8b_32k_fork", lambda: synth.llama8b_32k(fork=True)),
    ("sessions_64k_small", lambda: synth.sessions_64k(n_layers=2, n_sessions=3, prefix=1024, per_session=8192,
                                                      q_per_seg=128, span_len=(64, 512))),
    ("mla_c4", lambda: synth.mla_dsv2lite(n_layers=2, concurrency=4)),
    ("llama70b_small", lambda: synth.llama70b_128k(n_layers=2, total=16384, n_branches=6, q_per_branch=256)),
]


@pytest.mark.parametrize("name,make", WORKLOADS, ids=[n for n, _ in WORKLOADS])
def test_workload_bookkeeping_matches_oracle(name, make):
    w = make()
    eng, model = engine_for(w), oracle_model(w)
    ne = runner.run_ops(eng, w)
    no = oracle_run_ops(model, w)
    assert ne == no
    assert_same_state(eng, model, ne, no)
    # the flush that attention triggers: sequences of the segments, in id order
    ids = sorted({no[s["seq"]] for s in w.segments})
    runs_o = model.flush(ids)
    for i in ids:
        eng.flush(i)
    assert_same_state(eng, model, ne, no)
    for s in w.segments:
        seg = dict(seq=ne[s["seq"]], kv_end=s["kv_end"], q_len=s["q_len"], hide=np.asarray(s["hide"]).reshape(-1))
        runs_e, kv_e = eng.segment_runs(seg)
        runs_m, kv_m = model.segment_runs(no[s["seq"]], s["kv_end"], s["q_len"], s["hide"])
        assert kv_e == kv_m
        assert np.array_equal(runs_e, np.asarray(runs_m, np.int32).reshape(-1, 4))


@pytest.mark.parametrize("name,make", WORKLOADS[:3] + WORKLOADS[4:5], ids=[n for n, _ in WORKLOADS[:3] + WORKLOADS[4:5]])
def test_flush_run_lists_match_oracle(name, make):
    w = make()
    eng, model = engine_for(w), oracle_model(w)
    ne = runner.run_ops(eng, w)
    no = oracle_run_ops(model, w)
    runs_o = model.flush()          # every live sequence, increasing id
    eng.flush(-1)
    assert np.array_equal(eng.last_flush_runs(), np.asarray(runs_o, np.int32).reshape(-1, 5))
    assert_same_state(eng, model, ne, no)


def apply_both(eng, model, op, args):
    """Run one operation on both sides; both must succeed or fail with the same status."""
    err_e = err_o = None
    out_e = out_o = None
    try:
        out_e = getattr(eng, op)(*args)
    except akv.AKVError as x:
        err_e = x.code
    try:
        out_o = getattr(model, op)(*args)
    except CacheError as x:
        err_o = x.code
    assert err_e == err_o, (op, args, err_e, err_o)
    return out_e, out_o, err_e


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    P = int(rng.choice([16, 32]))
    n_pages = int(rng.integers(12, 80))
    cfg = dict(layout=0, n_layers=1, n_q_heads=4, n_kv_heads=1, d_rot=64, d_v=64, page_size=P, n_pages=n_pages,
               rope_layout=0, rope_base=1e4)
    eng, model = akv.Engine(cfg), CacheModel(n_pages, P)
    ids = [eng.seq_alloc()]
    assert model.seq_alloc() == ids[0]
    for step in range(150):
        live = sorted(model.seqs)
        s = live[int(rng.integers(len(live)))]
        n = len(model.seqs[s])
        op = rng.choice(["append", "fork", "drop", "repos", "splice", "flush", "flush_all", "free", "seg", "bad",
                         "compact"])
        if op == "append":
            apply_both(eng, model, "append", (s, int(rng.integers(0, 3 * P))))
        elif op == "fork" and len(live) < 8:
            e_id, o_id, err = apply_both(eng, model, "seq_fork", (s, int(rng.integers(0, n + 1))))
            assert e_id == o_id
        elif op == "drop":
            a = int(rng.integers(0, n + 1))
            apply_both(eng, model, "drop", (s, a, int(rng.integers(a, n + 1))))
        elif op == "repos":
            a = int(rng.integers(0, n + 1))
            d = int(rng.integers(-3000, 3000)) if rng.random() < 0.9 else int(rng.choice([2 ** 31 - 1, -2 ** 31]))
            apply_both(eng, model, "repos", (s, a, int(rng.integers(a, n + 1)), d))
        elif op == "splice":
            a = int(rng.integers(0, n + 1))
            apply_both(eng, model, "splice", (s, a, int(rng.integers(a, n + 1)), int(rng.integers(0, 2 * P))))
        elif op == "flush":
            try:
                runs_o = model.flush([s])
                err_o = None
            except CacheError as x:
                err_o, runs_o = x.code, []
            try:
                eng.flush(s)
                err_e = None
            except akv.AKVError as x:
                err_e = x.code
            assert err_e == err_o
            if runs_o:
                assert np.array_equal(eng.last_flush_runs(), np.asarray(runs_o, np.int32).reshape(-1, 5))
        elif op == "flush_all":
            try:
                runs_o = model.flush()
                err_o = None
            except CacheError as x:
                err_o, runs_o = x.code, []
            try:
                eng.flush(-1)
                err_e = None
            except akv.AKVError as x:
                err_e = x.code
            assert err_e == err_o
            if runs_o:
                assert np.array_equal(eng.last_flush_runs(), np.asarray(runs_o, np.int32).reshape(-1, 5))
        elif op == "free" and len(live) > 1:
            apply_both(eng, model, "seq_free", (s,))
        elif op == "seg" and n:
            q = int(rng.integers(1, min(n, 8) + 1))
            a = int(rng.integers(0, n - q + 1))
            hide = [(a, int(rng.integers(a, n - q + 1)))] if rng.random() < 0.5 else []
            try:
                ro, ko = model.segment_runs(s, n, q, hide)
                err_o = None
            except CacheError as x:
                err_o = x.code
            try:
                re_, ke = eng.segment_runs(dict(seq=s, kv_end=n, q_len=q, hide=np.asarray(hide).reshape(-1)))
                err_e = None
            except akv.AKVError as x:
                err_e = x.code
            assert err_e == err_o
            if err_o is None:
                assert ke == ko and np.array_equal(re_, np.asarray(ro, np.int32).reshape(-1, 4))
        elif op == "bad":
            apply_both(eng, model, "drop", (s, -1, 2))
            apply_both(eng, model, "repos", (s, 0, n + 1, 1))
        elif op == "compact":
            assert eng.fragmentation(s) == model.fragmentation(s)
            apply_both(eng, model, "compact", (s,))
            assert eng.fragmentation(s) == model.fragmentation(s)
        # full comparison after every step
        for sid in model.seqs:
            a, b = eng.export_state(sid), model.state(sid)
            for k in b:
                assert np.array_equal(a[k], np.asarray(b[k], np.int32)), (step, op, k)
        ke, ve = eng.refcounts()
        ko, vo = model.refcounts()
        assert np.array_equal(ke, ko) and np.array_equal(ve, vo), (step, op)


@pytest.mark.parametrize("seed", range(6))
def test_batched_repositions_fold_like_the_oracle(seed):
    """Several repositions recorded before any read fold into the tokens at once
    (the engine sweeps the spans' sorted end points).  Batches of 2-10 spans
    that overlap, cancel to a zero sum over part of the sequence, share end
    points or are empty, with drops between them, then a flush: the state
    after the fold and the flush run list equal the oracle's, which applies
    each reposition to its tokens one by one."""
    rng = np.random.default_rng(700 + seed)
    P = 16
    cfg = dict(layout=0, n_layers=1, n_q_heads=4, n_kv_heads=1, d_rot=64, d_v=64, page_size=P, n_pages=96,
               rope_layout=0, rope_base=1e4)
    eng, model = akv.Engine(cfg), CacheModel(96, P)
    s = eng.seq_alloc()
    assert model.seq_alloc() == s
    apply_both(eng, model, "append", (s, 600))
    for batch in range(8):
        n = len(model.seqs[s])
        ends = np.sort(rng.integers(0, n + 1, size=4))  # shared end points across the batch's spans
        for _ in range(int(rng.integers(2, 11))):
            kind = rng.random()
            if kind < 0.15:
                a = int(rng.integers(0, n + 1))
                apply_both(eng, model, "drop", (s, a, int(rng.integers(a, n + 1))))
                continue
            if kind < 0.5:
                a, b = sorted(int(x) for x in rng.choice(ends, size=2))
            else:
                a = int(rng.integers(0, n + 1))
                b = int(rng.integers(a, n + 1))
            d = int(rng.integers(-700, 700))
            apply_both(eng, model, "repos", (s, a, b, d))
            if rng.random() < 0.3:  # the same span undone: a zero sum where nothing else covers it
                apply_both(eng, model, "repos", (s, a, b, -d))
        a, b = eng.export_state(s), model.state(s)
        for k in b:
            assert np.array_equal(a[k], np.asarray(b[k], np.int32)), (batch, k)
        if batch % 2:
            runs_o = model.flush([s])
            eng.flush(s)
            if runs_o:
                assert np.array_equal(eng.last_flush_runs(), np.asarray(runs_o, np.int32).reshape(-1, 5))
            a, b = eng.export_state(s), model.state(s)
            for k in b:
                assert np.array_equal(a[k], np.asarray(b[k], np.int32)), (batch, "flushed", k)


@pytest.mark.parametrize("name,make", WORKLOADS, ids=[n for n, _ in WORKLOADS])
def test_compaction_matches_oracle(name, make):
    # every live sequence compacted in turn after the workload's operations (pending shifts
    # included); each step must agree, NO_PAGES included
    w = make()
    w.n_pages = int(w.n_pages * 1.6) + 64
    eng, model = engine_for(w), oracle_model(w)
    ne = runner.run_ops(eng, w)
    no = oracle_run_ops(model, w)
    for name_ in sorted(no):
        sid = no[name_]
        if sid not in model.seqs:
            continue
        assert eng.fragmentation(sid) == model.fragmentation(sid)
        apply_both(eng, model, "compact", (sid,))
        assert_same_state(eng, model, ne, no)
        assert eng.fragmentation(sid) == model.fragmentation(sid)


def shared_prefix_both_shifted(n=4096, q=16):
    """Two branches sharing an n-token prefix, every prefix token shifted on both (by different
    amounts), one segment each: attend flushes both in one call."""
    import dataclasses
    w = synth.tiny()
    w.shape = dataclasses.replace(w.shape, n_q_heads=8, n_kv_heads=2)
    w.ops = [("alloc", "A"), ("append", "A", n, "ctx"), ("fork", "B", "A", n),
             ("repos", "A", 0, n, 1000), ("repos", "B", 0, n, -2000),
             ("append", "A", q, "newA"), ("append", "B", q, "newB")]
    w.segments = [dict(seq="A", kv_end=n + q, q_len=q, hide=[], q_row0=0),
                  dict(seq="B", kv_end=n + q, q_len=q, hide=[], q_row0=q)]
    w.n_pages = 3 * (n // w.shape.page_size) + 16
    return w


def test_one_flush_copies_a_page_out_and_rotates_it_in_place():
    # The first sharer copies each shared page out (copy-on-write); the second, then its only
    # holder, rotates it in place.  The two kinds of run must not share a launch (the GPU runs a
    # launch's runs concurrently), which the engine orders; here: the run list holds both kinds.
    w = shared_prefix_both_shifted()
    eng = engine_for(w)
    names = runner.run_ops(eng, w)
    nq = sum(g["q_len"] for g in w.segments)
    eng.attend(0, runner.engine_segments(w, names), None, nq, None)
    runs = eng.last_flush_runs()
    model, names_o = oracle_model(w), {}
    oracle_run_ops(model, w, names=names_o)
    want = model.flush(sorted({names_o[g["seq"]] for g in w.segments}))
    assert np.array_equal(np.asarray(runs), np.asarray(want, np.int32).reshape(-1, 5))
    copied = {int(r[0]) for r in runs if r[0] != r[1]}
    in_place = {int(r[1]) for r in runs if r[0] == r[1]}
    assert len(copied & in_place) == w.ops[1][2] // w.shape.page_size
