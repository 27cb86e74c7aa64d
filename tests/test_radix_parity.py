"""The engine's extended radix tree (metadata-only context, no GPU) against the
oracle's brute-force matcher: kind, matched length and holder of every match,
on random token sets with operation markers and shifted positions; and the
bookkeeping of a reuse (fork, repositioning to the request's positions)."""
import numpy as np
import pytest

from agentic_kv_cache_gb300 import akv, build
from oracle.cache import CacheModel
from oracle.radix import RadixOracle


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def make_engine(n_pages=4000):
    cfg = dict(layout=0, n_layers=1, n_q_heads=4, n_kv_heads=1, d_rot=64, d_v=64, page_size=16, n_pages=n_pages,
               rope_layout=0, rope_base=1e4)
    return akv.Engine(cfg)


def random_path(rng, base=None):
    """A path of tokens from a small alphabet (so that many paths share prefixes), with
    occasional operation markers and position jumps."""
    if base is not None and rng.random() < 0.7:
        cut = int(rng.integers(0, len(base) + 1))
        path = list(base[:cut])
    else:
        path = []
    pos = max([it[2] for it in path if it[0] == "tok"], default=-1) + 1
    for _ in range(int(rng.integers(1, 25))):
        r = rng.random()
        if r < 0.1:
            path.append(("op", int(rng.integers(1, 3)), int(rng.integers(0, 4)), 0, 0))
        else:
            if r < 0.15:
                pos += int(rng.integers(-50, 50))
            path.append(("tok", int(rng.integers(0, 3)), pos))
            pos += 1
    return path


def mutate(rng, path):
    req = list(path[: int(rng.integers(0, len(path) + 1))])
    if req and rng.random() < 0.5:  # shift every position of a suffix
        k = int(rng.integers(0, len(req)))
        d = int(rng.integers(-100, 100))
        req = req[:k] + [(it[0], it[1], it[2] + d) if it[0] == "tok" else it for it in req[k:]]
    if req and rng.random() < 0.3:  # change one item
        k = int(rng.integers(0, len(req)))
        req[k] = ("tok", 9, 0) if req[k][0] == "op" else ("op", 1, 9, 0, 0)
    for _ in range(int(rng.integers(0, 5))):
        req.append(("tok", int(rng.integers(0, 3)), int(rng.integers(0, 1000))))
    return req


@pytest.mark.parametrize("seed", range(10))
def test_tree_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    eng, orc = make_engine(), RadixOracle()
    holders = {}  # engine holder seq -> oracle label
    paths = []
    for i in range(int(rng.integers(1, 12))):
        path = random_path(rng, paths[int(rng.integers(len(paths)))] if paths else None)
        n_tok = sum(1 for it in path if it[0] == "tok")
        sid = eng.seq_alloc()
        eng.append(sid, n_tok)
        h = eng.tree_insert(path, sid)
        eng.seq_free(sid)
        orc.insert(i, path)
        paths.append(path)
        if h >= 0:
            holders[h] = i
    for _ in range(60):
        req = mutate(rng, paths[int(rng.integers(len(paths)))]) if rng.random() < 0.9 else random_path(rng)
        m = eng.tree_match(req)
        kind, n, owner = orc.match(req)
        assert (m["kind"], m["n_items"]) == (kind, n), (req, m, kind, n)
        if kind != "none":
            # the holder the engine names is the earliest path with that match (the oracle's owner)
            assert holders[m["seq"]] == owner
            assert m["n_tokens"] == sum(1 for it in req[:n] if it[0] == "tok")


def test_reuse_repositions_to_the_request_and_leaves_the_holder_alone():
    eng = make_engine()
    model = CacheModel(4000, 16)
    path = [("tok", t, 100 + i) for i, t in enumerate(range(40))] + [("op", 1, 5, 9, 0)] + \
           [("tok", t, 140 + i) for i, t in enumerate(range(40, 60))]
    sid = eng.seq_alloc()
    eng.append(sid, 60, pos=np.arange(100, 160, dtype=np.int32))
    holder = eng.tree_insert(path, sid)
    before = eng.export_state(holder)
    req = [("tok", t, 7 + i) for i, t in enumerate(range(40))] + [("op", 1, 5, 9, 0)] + \
          [("tok", t, 47 + i) for i, t in enumerate(range(40, 55))]
    m, new = eng.tree_reuse(req)
    assert m == dict(kind="retrigger", seq=holder, n_items=56, n_tokens=55)
    st = eng.export_state(new)
    assert np.array_equal(st["pos"], np.arange(7, 62)) and not np.any(st["delta"])
    # the oracle's bookkeeping of the same fork + reposition + flush gives the same page map
    a = model.seq_alloc()
    model.append(a, 60, pos=list(range(100, 160)))
    b = model.seq_fork(a, 60)            # the tree's holder
    model.seq_free(a)
    c = model.seq_fork(b, 55)
    model.repos(c, 0, 55, -93)
    model.flush([c])
    want = model.state(c)
    for k in ("k_page", "v_page", "slot", "pos", "delta"):
        assert np.array_equal(st[k], np.asarray(want[k], np.int32)), k
    for k in before:
        assert np.array_equal(eng.export_state(holder)[k], before[k])
    # an exact request is a plain fork
    m2, new2 = eng.tree_reuse(path[:30])
    assert m2["kind"] == "exact" and np.array_equal(eng.export_state(new2)["pos"], np.arange(100, 130))
    eng.tree_clear()
    assert eng.tree_match(path)["kind"] == "none"
