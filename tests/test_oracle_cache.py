"""Pins for oracle.cache, the paged bookkeeping model."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle.cache import CacheError, CacheModel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_fresh_append_page_map_closed_form():
    c = CacheModel(64, 16)
    s = c.seq_alloc()
    c.append(s, 100)
    st = c.state(s)
    assert st["k_page"] == [i // 16 for i in range(100)]
    assert st["v_page"] == [i // 16 for i in range(100)]
    assert st["slot"] == [i % 16 for i in range(100)]
    assert st["pos"] == list(range(100))
    k_rc, v_rc = c.refcounts()
    assert k_rc[:7] == [1] * 7 and sum(k_rc) == 7


def test_blog_figure_drop_blocks_2_to_7_repos_8_9():
    g = load("akv_blog_s2_drop_repos_figure.json")
    P = g["page_size"]
    c = CacheModel(32, P)
    s = c.seq_alloc()
    c.append(s, g["n_blocks"] * P)
    d0, d1 = g["drop_blocks"]
    r0, r1 = g["repos_blocks"]
    c.drop(s, d0 * P, (d1 + 1) * P)
    c.repos(s, r0 * P, (r1 + 1) * P, g["delta_blog"])
    runs = c.flush()
    assert runs == [(b, b, 0, P, g["delta_blog"]) for b in range(r0, r1 + 1)]
    pos = c.state(s)["pos"]
    for b, (lo, hi) in zip(range(r0, r1 + 1), g["repos_block_positions_after"]):
        assert pos[b * P:(b + 1) * P] == list(range(lo, hi + 1))
    seg, n = c.segment_runs(s, g["n_blocks"] * P, 1)
    assert [r[0] for r in seg] == g["active_blocks"] and n == 4 * P


def test_blog_history_dependence_two_sessions():
    g = load("akv_blog_s3_history_dependence.json")
    c = CacheModel(600, 16)
    s2 = c.seq_alloc()
    c.append(s2, g["n_tokens"])
    s1 = c.seq_fork(s2, g["n_tokens"])              # both sessions share the prefix
    a, b = g["drop"]
    c.drop(s1, a, b)
    c.repos(s1, b, g["n_tokens"], g["delta"])
    runs = c.flush()
    st1, st2 = c.state(s1), c.state(s2)
    vis = [i for i, v in enumerate(st1["visible"]) if v]
    assert len(vis) == g["retained"]
    assert [st1["pos"][i] for i in vis] == list(range(g["retained"]))   # compacted coordinates
    assert st2["pos"] == list(range(g["n_tokens"]))                     # session 2 untouched
    # Session 1's rotated keys live in copies; V pages stay shared.  Page 218
    # holds tokens 3488..3503: its dropped tokens 3488..3499 stay behind.
    assert all(st1["k_page"][i] != st2["k_page"][i] for i in range(b, g["n_tokens"]))
    assert all(st1["k_page"][i] == st2["k_page"][i] for i in range(0, b))
    assert all(st1["v_page"][i] == st2["v_page"][i] for i in range(g["n_tokens"]))
    moved = sum(hi - lo for _, _, lo, hi, _ in runs)
    assert moved == g["n_tokens"] - b


def test_leyline_splice_delta():
    g = load("leyline_method_splice.json")
    c = CacheModel(400, 64)
    s = c.seq_alloc()
    n = 17408
    c.append(s, n)
    start = 5000
    c.splice(s, start, start + g["span"], g["stub"])
    st = c.state(s)
    assert len(st["pos"]) == n - g["span"] + g["stub"]
    stub = slice(start, start + g["stub"])
    assert st["pos"][stub] == list(range(start, start + g["stub"]))
    after = start + g["stub"]
    assert set(st["delta"][after:]) == {g["delta"]}
    assert set(st["delta"][:after]) == {0}
    assert st["pos"][after] + st["delta"][after] == start + g["stub"]   # contiguous after the stub


def test_splice_frees_pages_only_the_sequence_leaves():
    c = CacheModel(16, 16)
    s = c.seq_alloc()
    c.append(s, 80)                       # pages 0..4
    c.splice(s, 20, 70, 0)                # tokens 20..69 leave; page 2, 3 become unreferenced
    k_rc, _ = c.refcounts()
    assert k_rc[:5] == [1, 1, 0, 0, 1]
    c.splice(s, 20, 20, 20)               # stub of 20 into the lowest free pages: 2, 3
    st = c.state(s)
    assert st["k_page"][20:40] == [2] * 16 + [3] * 4


@pytest.mark.parametrize("n_dir", [2, 3])
def test_composition_commutes_brute_force(n_dir):
    # Non-overlapping drop+repos directives, applied in every order, give the
    # same final positions, and these equal the closed form: a retained token
    # moves back by the total length dropped before it.
    n, P = 64, 8
    rng = np.random.default_rng(n_dir)
    for trial in range(10):
        cuts = np.sort(rng.choice(np.arange(1, n), size=2 * n_dir, replace=False))
        spans = [(int(cuts[2 * i]), int(cuts[2 * i + 1])) for i in range(n_dir)]
        results = set()
        for order in itertools.permutations(spans):
            c = CacheModel(32, P)
            s = c.seq_alloc()
            c.append(s, n)
            for a, b in order:
                c.drop(s, a, b)
                c.repos(s, b, n, -(b - a))
            c.flush()
            st = c.state(s)
            results.add((tuple(st["pos"]), tuple(st["visible"]), tuple(st["delta"])))
        assert len(results) == 1
        pos, vis, _ = results.pop()
        for i in range(n):
            if vis[i]:
                assert pos[i] == i - sum(b - a for a, b in spans if b <= i)


def test_errors_leave_state_unchanged():
    c = CacheModel(4, 16)
    s = c.seq_alloc()
    c.append(s, 60)
    before = (c.state(s), c.refcounts())
    with pytest.raises(CacheError) as e:
        c.append(s, 10)                   # needs a 5th page
    assert e.value.code == "NO_PAGES"
    with pytest.raises(CacheError) as e:
        c.drop(s, 10, 61)
    assert e.value.code == "RANGE"
    with pytest.raises(CacheError) as e:
        c.repos(s, 0, 10, 2 ** 31 - 5)
    assert e.value.code == "OVERFLOW"
    f = c.seq_fork(s, 60)
    c.repos(f, 0, 60, 3)
    with pytest.raises(CacheError) as e:
        c.flush([f])                      # needs 4 copy-on-write pages, none free
    assert e.value.code == "NO_PAGES"
    c.seq_free(f)
    assert (c.state(s), c.refcounts()) == before


class ValueModel:
    """Brute force over the data: each pool slot holds (token id, position it is rotated to)."""

    def __init__(self, c):
        self.c = c
        self.k, self.v = {}, {}
        self.uid = 0
        self.tok_uid = {}  # (seq, logical index) is not stable; keep uids in a parallel list

    def write(self, seq, start_index, slots):
        st = self.c.state(seq)
        ids = []
        for j, (kp, vp, slot) in enumerate(slots):
            i = start_index + j
            self.uid += 1
            self.k[(kp, slot)] = (self.uid, st["pos"][i])
            self.v[(vp, slot)] = self.uid
            ids.append(self.uid)
        return ids

    def apply_runs(self, runs):
        new_k = dict(self.k)
        for src, dst, lo, hi, d in runs:
            for slot in range(lo, hi):
                uid, p = self.k[(src, slot)]
                new_k[(dst, slot)] = (uid, p + d)
        self.k = new_k


def test_random_operations_keep_every_sequence_intact():
    rng = np.random.default_rng(7)
    P = 8
    for trial in range(25):
        c = CacheModel(96, P)
        vm = ValueModel(c)
        uids = {}
        s = c.seq_alloc()
        uids[s] = vm.write(s, 0, c.append(s, int(rng.integers(1, 40))))
        for step in range(40):
            live = sorted(c.seqs)
            seq = live[int(rng.integers(len(live)))]
            n = len(c.seqs[seq])
            op = rng.choice(["append", "fork", "drop", "repos", "splice", "flush", "free"])
            try:
                if op == "append":
                    k = int(rng.integers(0, 20))
                    uids[seq] += vm.write(seq, n, c.append(seq, k))
                elif op == "fork" and len(live) < 6:
                    f = c.seq_fork(seq, int(rng.integers(0, n + 1)))
                    uids[f] = uids[seq][:len(c.seqs[f])]
                elif op == "drop" and n:
                    a = int(rng.integers(0, n))
                    c.drop(seq, a, int(rng.integers(a, n + 1)))
                elif op == "repos" and n:
                    a = int(rng.integers(0, n))
                    c.repos(seq, a, int(rng.integers(a, n + 1)), int(rng.integers(-50, 51)))
                elif op == "splice" and n:
                    a = int(rng.integers(0, n))
                    b = int(rng.integers(a, n + 1))
                    k = int(rng.integers(0, 12))
                    slots = c.splice(seq, a, b, k)
                    new = vm.write(seq, a, slots)
                    uids[seq] = uids[seq][:a] + new + uids[seq][b:]
                elif op == "flush":
                    vm.apply_runs(c.flush())
                elif op == "free" and len(live) > 1:
                    c.seq_free(seq)
                    del uids[seq]
            except CacheError as e:
                assert e.code in ("NO_PAGES", "OVERFLOW")
            # invariants: refcount = number of live sequences referencing the page
            k_rc, v_rc = c.refcounts()
            for p in range(c.n_pages):
                assert k_rc[p] == sum(any(t.kp == p for t in ts) for ts in c.seqs.values())
                assert v_rc[p] == sum(any(t.vp == p for t in ts) for ts in c.seqs.values())
        vm.apply_runs(c.flush())
        # every visible token of every sequence reads back its own key at its position
        for sid, ts in c.seqs.items():
            for t, uid in zip(ts, uids[sid]):
                assert vm.v[(t.vp, t.slot)] == uid
                if t.vis:
                    assert t.delta == 0
                    assert vm.k[(t.kp, t.slot)] == (uid, t.pos)


def test_segment_runs_hide_and_query_rules():
    c = CacheModel(32, 16)
    s = c.seq_alloc()
    c.append(s, 100)
    c.drop(s, 10, 20)
    runs, n = c.segment_runs(s, 100, 4, hide=[(40, 50)])
    assert n == 100 - 10 - 10
    assert runs[:4] == [(0, 0, 0, 10), (1, 1, 4, 16), (2, 2, 0, 8), (3, 3, 2, 16)]
    with pytest.raises(CacheError):
        c.segment_runs(s, 100, 4, hide=[(98, 99)])       # a query hidden
    c.repos(s, 20, 100, -10)
    with pytest.raises(CacheError):
        c.segment_runs(s, 100, 4)                          # pending delta must be flushed first


# ------------------------------------------------------------- compaction
def test_compaction_blog_example_64_blocks_every_second_dropped():
    # [AKV-blog] "Dilemma 2": 64 blocks with every second block dropped leave 32 live pages
    # among 32 dead ones; compaction copies the survivors into contiguous pages.
    P = 16
    c = CacheModel(200, P)
    s = c.seq_alloc()
    c.append(s, 64 * P)
    for b in range(1, 64, 2):
        c.drop(s, b * P, (b + 1) * P)
    assert c.fragmentation(s) == 0.5
    copies = c.compact(s)
    st = c.state(s)
    assert len(st["pos"]) == 32 * P and all(st["visible"])
    # fresh pages are the lowest free ids at the time of the copy: 64 .. 95, filled densely
    assert st["k_page"] == [64 + i // P for i in range(32 * P)]
    assert st["slot"] == [i % P for i in range(32 * P)]
    # survivors keep their positions and order: blocks 0, 2, 4, ...
    assert st["pos"] == [b * P + j for b in range(0, 64, 2) for j in range(P)]
    assert [cp[0] for cp in copies] == [b for b in range(0, 64, 2) for _ in range(P)]
    assert c.fragmentation(s) == 0.0
    k_rc, v_rc = c.refcounts()
    assert sum(k_rc[:64]) == 0 and k_rc[64:96] == [1] * 32 and sum(k_rc) == 32
    assert sum(v_rc) == 32


def test_compaction_fuses_pending_shift():
    P = 8
    c = CacheModel(32, P)
    s = c.seq_alloc()
    c.append(s, 20)
    c.drop(s, 3, 6)
    c.repos(s, 6, 20, -3)
    c.repos(s, 10, 12, 100)
    copies = c.compact(s)
    st = c.state(s)
    want_pos = [0, 1, 2] + [i - 3 for i in range(6, 20)]
    want_pos[10 - 3] += 100
    want_pos[11 - 3] += 100
    assert st["pos"] == want_pos and st["delta"] == [0] * 17
    assert [cp[6] for cp in copies] == [0, 0, 0] + [-3] * 4 + [97, 97] + [-3] * 8


def test_compaction_of_a_fork_leaves_the_parent_alone():
    P = 16
    c = CacheModel(64, P)
    a = c.seq_alloc()
    c.append(a, 100)
    b = c.seq_fork(a, 100)
    c.drop(b, 0, 40)
    before = c.state(a)
    c.compact(b)
    assert c.state(a) == before
    k_rc, _ = c.refcounts()
    assert k_rc[:7] == [1] * 7                     # only the parent references its pages now
    assert c.state(b)["k_page"] == [7 + i // P for i in range(60)]


def test_compaction_without_free_pages_changes_nothing():
    P = 16
    c = CacheModel(8, P)
    s = c.seq_alloc()
    c.append(s, 100)                                # 7 pages, 1 free
    c.drop(s, 0, 60)                                # 40 visible -> needs 3 fresh pages
    st, rc = c.state(s), c.refcounts()
    with pytest.raises(CacheError) as e:
        c.compact(s)
    assert e.value.code == "NO_PAGES"
    assert c.state(s) == st and c.refcounts() == rc


def test_compaction_keeps_the_visible_sequence_random():
    rng = np.random.default_rng(5)
    for trial in range(20):
        P = int(rng.choice([4, 8, 16]))
        c = CacheModel(400, P)
        s = c.seq_alloc()
        n = int(rng.integers(1, 300))
        c.append(s, n)
        for _ in range(int(rng.integers(0, 6))):
            a = int(rng.integers(0, n))
            b = int(rng.integers(a, n + 1))
            if rng.random() < 0.5:
                c.drop(s, a, b)
            else:
                c.repos(s, a, b, int(rng.integers(-500, 500)))
        old = c.state(s)
        vis = [i for i in range(n) if old["visible"][i]]
        copies = c.compact(s)
        new = c.state(s)
        assert len(new["pos"]) == len(vis) == len(copies)
        assert new["pos"] == [old["pos"][i] + old["delta"][i] for i in vis]
        assert [(cp[0], cp[2], cp[6]) for cp in copies] == [(old["k_page"][i], old["slot"][i], old["delta"][i])
                                                           for i in vis]
        k_rc, v_rc = c.refcounts()
        assert sum(k_rc) == sum(v_rc) == -(-len(vis) // P)
