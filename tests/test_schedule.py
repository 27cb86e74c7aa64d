"""Attention schedules planned on the host, checked without a GPU.

A metadata-only context runs the planners and keeps the last plan
(akv_last_attention_plan).  For the workloads' launches this checks what every
schedule must satisfy: each work item's KV tiles are covered exactly once by
its units; an item cut into several units has one partial slot per unit and
one merge item; no item is cut into more than 8 parts; the persistent lists
partition the units and give the CTAs equal work (MLA: no CTA pair far above
the mean); every MLA unit reads at least one tile and its two entries (a CTA
pair) agree.  The GPU tests check the results of the same plans against the
oracle."""
from collections import defaultdict

import numpy as np
import pytest

from agentic_kv_cache_gb300 import akv, build, runner, synth

N_SM = 152
UNIT_COST = 1        # GQA planner: start + epilogue of a unit, in query-tile steps
MLA_UNIT_COST = 6    # MLA planner: the same, in KV tiles


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return akv.load()


def plan(w, split=0):
    eng = akv.Engine(akv.config_from_shape(w.shape, w.n_pages), None)
    eng.last_attention_plan(n_sm=N_SM)
    eng.set_attention_split(split)
    names = runner.run_ops(eng, w)
    eng.attend(0, runner.engine_segments(w, names), None, w.n_queries, None, None, w.shape.scale)
    return eng.last_attention_plan()


def check_cover(units, key_cols, span_of):
    """Every item (identified by key_cols) covered exactly once by its units' [t0, t1); part slots
    distinct per item and present exactly when it has several units."""
    by_item = defaultdict(list)
    for u in units:
        by_item[tuple(u[key_cols])].append(u)
    for key, us in by_item.items():
        span = span_of(us[0])
        ranges = sorted((int(u[5]), int(u[6])) for u in us)
        assert ranges[0][0] == 0 and ranges[-1][1] == span, (key, ranges, span)
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:])), (key, ranges)
        assert all(t0 < t1 for t0, t1 in ranges), (key, ranges)
        parts = [int(u[7]) for u in us]
        if len(us) == 1:
            assert parts == [-1]
        else:
            assert len(us) <= 8 and len(set(parts)) == len(us) and min(parts) >= 0, (key, parts)
            assert len({int(u[8]) for u in us}) == 1
    return by_item


def gqa_cost(u):
    t0, t1 = int(u[5]), int(u[6])
    return UNIT_COST + max(0, min(u[3], t1) - t0) + max(0, min(u[4], t1) - t0)


@pytest.mark.parametrize("workload", ["llama8b_32k", "sessions_64k", "llama70b_128k"])
def test_gqa_persistent_schedule(workload):
    w = {"llama8b_32k": lambda: synth.llama8b_32k(fork=True),
         "sessions_64k": lambda: synth.sessions_64k(n_layers=1),
         "llama70b_128k": lambda: synth.llama70b_128k(n_layers=1)}[workload]()
    units, cta = plan(w)
    items = check_cover(units, [0, 1, 2], lambda u: max(int(u[3]), int(u[4])))
    assert cta.size == N_SM + 1 and cta[0] == 0 and cta[-1] == len(units) and np.all(np.diff(cta) >= 1)
    cost = np.array([sum(gqa_cost(u) for u in units[cta[b]:cta[b + 1]]) for b in range(N_SM)])
    # a cut moves by at most kMinSteps (4) steps of cost <= 2 at either end of a CTA's range, and
    # a piece that would be shorter stays with its item: a spread of a few such margins
    assert cost.max() - cost.min() <= 4 * (2 * 4 + UNIT_COST), (cost.min(), cost.max())
    if workload != "llama8b_32k":
        # many items per CTA: the K/V-grouped layout, so the CTAs running at one time share kv heads
        assert len(items) >= 4 * N_SM
        first = [units[cta[b]] for b in range(N_SM)]
        assert len({int(u[1]) for u in first}) <= 2   # all CTAs start in one or two kv heads


@pytest.mark.parametrize("concurrency", [1, 4, 16])
def test_mla_persistent_schedule(concurrency):
    w = synth.mla_dsv2lite(n_layers=1, concurrency=concurrency)
    units, cta = plan(w)
    assert len(units) % 2 == 0
    pairs = units.reshape(-1, 2, 9)
    for a, b in pairs:                       # the two CTAs of a pair share the KV range and the half
        assert a[0] == b[0] and tuple(a[3:7]) == tuple(b[3:7])
        assert a[5] < a[3], "a unit reads at least one KV tile"
    for m in (0, 1):                         # each CTA's entries cover their item exactly once
        check_cover(pairs[:, m, :], [0, 1, 2, 4], lambda u: max(1, int(u[3])))
    n_pairs = cta.size - 1
    assert 1 <= n_pairs <= N_SM // 2 and cta[-1] == len(pairs) and np.all(np.diff(cta) >= 1)
    cost = np.array([sum(MLA_UNIT_COST + int(p[0][6] - p[0][5]) for p in pairs[cta[b]:cta[b + 1]])
                     for b in range(n_pairs)])
    # the launch lasts as long as its busiest pair: within a start cost and two minimum pieces of
    # the mean (a pair closes early only when the next piece could not be cut at least 4 tiles long)
    assert cost.max() <= cost.sum() / n_pairs + MLA_UNIT_COST + 2 * 4, (cost.max(), cost.sum() / n_pairs)
    if concurrency == 1:
        assert n_pairs == N_SM // 2               # every resident pair has work


def test_forced_split_keeps_one_unit_per_cta():
    units, cta = plan(synth.mla_dsv2lite(n_layers=1, concurrency=2), split=3)
    assert cta.size == 0
    check_cover(units.reshape(-1, 2, 9)[:, 0, :], [0, 1, 2, 4], lambda u: max(1, int(u[3])))
    units, cta = plan(synth.llama8b_32k(total=4096, n_new=256, fork=True), split=2)
    assert cta.size == 0
    check_cover(units, [0, 1, 2], lambda u: max(int(u[3]), int(u[4])))
