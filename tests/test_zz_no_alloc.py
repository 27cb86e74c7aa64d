"""akv_repos_rotate_noalloc against the context path (akv_flush), on the GPU.

The no-allocation entry point serves callers that cannot call cudaMalloc (for
example a serving process whose KV pool has taken nearly all of HBM, or a
latency-critical path that must not trigger the device-wide synchronisation
cudaMalloc / cudaFree can cause).  It runs the same repos_rotate kernel with
its run list and (cos, sin) table in a fixed array of the library's own device
memory.  Here two flushes in a row of a 32K-style trajectory (copy-on-write
branch, then in place) go through akv_flush on one pool and through the
no-allocation entry point on a copy of it; the results must match within the
rotated-key bar of the other tests -- in fact bit for bit, since the kernel and
the table are the same.  A flush of two sequences sharing pages, whose run
list copies a page out before rotating it in place, is checked the same way
for both RoPE pair layouts; run lists whose runs would race are refused.  This file is collected last so that a stop at the
first failure has run every other test first; it also passes on its own.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import akv, build, runner, synth

pytestmark = pytest.mark.gpu


def test_noalloc_matches_flush_on_two_calls_in_a_row():
    build.build()
    w = synth.llama8b_32k(total=8192, n_new=128, n_layers=2, fork=True)
    cfg = akv.config_from_shape(w.shape, w.n_pages)
    pools = akv.make_pools(cfg)
    eng = akv.Engine(cfg, pools)
    stream = torch.cuda.current_stream()
    names = runner.run_ops(eng, w, kv_source=runner.torch_kv_source(w), stream=stream)
    seq = names["F"]
    k_copy = pools[0].clone()

    # call 1: the turn's flush (drops + composed shifts, copy-on-write of shared pages)
    eng.flush(seq, stream=stream)
    runs1 = eng.last_flush_runs()
    assert len(runs1) > 100 and any(r[0] != r[1] for r in runs1)
    akv.repos_rotate_noalloc(k_copy, cfg, runs1, stream=stream)
    torch.cuda.synchronize()
    assert torch.equal(k_copy, pools[0])

    # call 2 right after: more shifts of either sign (in place on the branch's private pages,
    # copy-on-write where the branch still shares prefix pages)
    n = eng.seq_len(seq)
    eng.repos(seq, 100, n // 2, 777)
    eng.repos(seq, n // 3, n, -65000)
    eng.flush(seq, stream=stream)
    runs2 = eng.last_flush_runs()
    assert any(r[0] == r[1] for r in runs2)
    akv.repos_rotate_noalloc(k_copy, cfg, runs2, stream=stream)
    torch.cuda.synchronize()
    assert torch.equal(k_copy, pools[0])
    assert eng.check_device_error(stream) == 0


def test_noalloc_rejects_what_does_not_fit():
    build.build()
    cfg = dict(layout=0, n_layers=1, n_q_heads=4, n_kv_heads=1, d_rot=64, d_v=64, page_size=16, n_pages=32,
               rope_layout=0, rope_base=1e4)
    pool = torch.zeros((1, 32, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    before = pool.clone()
    too_many = np.tile(np.array([[0, 0, 0, 16, 5]], np.int32), (20000, 1))   # 20000 x 16 B > 256 KiB
    with pytest.raises(akv.AKVError) as e:
        akv.repos_rotate_noalloc(pool, cfg, too_many)
    assert e.value.code == "RANGE"
    with pytest.raises(akv.AKVError) as e:
        akv.repos_rotate_noalloc(pool, cfg, [[0, 40, 0, 16, 5]])            # page outside the pool
    assert e.value.code == "RANGE"
    torch.cuda.synchronize()
    assert torch.equal(pool, before)


@pytest.mark.parametrize("layout", ["interleaved", "half"])
def test_noalloc_orders_copies_before_in_place_rotations(layout):
    # One flush of two branches that share every prefix page: each shared page is copied out for
    # the first sharer and rotated in place for the second; the copies must read it first.
    import dataclasses
    from test_bookkeeping_parity import shared_prefix_both_shifted
    build.build()
    w = shared_prefix_both_shifted()
    w.shape = dataclasses.replace(w.shape, rope_layout=layout)
    cfg = akv.config_from_shape(w.shape, w.n_pages)
    pools = akv.make_pools(cfg)
    eng = akv.Engine(cfg, pools)
    stream = torch.cuda.current_stream()
    runner.run_ops(eng, w, kv_source=runner.torch_kv_source(w), stream=stream)
    k_copy = pools[0].clone()
    eng.flush(-1, stream=stream)
    runs = eng.last_flush_runs()
    assert {r[0] for r in runs if r[0] != r[1]} & {r[1] for r in runs if r[0] == r[1]}
    akv.repos_rotate_noalloc(k_copy, cfg, runs, stream=stream)
    torch.cuda.synchronize()
    assert torch.equal(k_copy, pools[0])
    assert eng.check_device_error(stream) == 0


def test_noalloc_refuses_runs_that_would_race():
    build.build()
    cfg = dict(layout=0, n_layers=1, n_q_heads=4, n_kv_heads=1, d_rot=64, d_v=64, page_size=16, n_pages=32,
               rope_layout=0, rope_base=1e4)
    pool = torch.randn((1, 32, 1, 16, 64), device="cuda").to(torch.bfloat16)
    before = pool.clone()
    for runs in ([[3, 3, 0, 8, 5], [3, 3, 4, 12, 7]],          # two in-place runs write rows 4..7
                 [[1, 5, 0, 16, 5], [2, 5, 8, 9, 6]],          # two copies write row 8 of page 5
                 [[1, 5, 0, 16, 5], [5, 6, 0, 4, 6]],          # a copy reads rows another copy writes
                 [[1, 5, 0, 16, 5], [5, 5, 2, 3, 6]]):         # a copy and an in-place run write one row
        with pytest.raises(akv.AKVError) as e:
            akv.repos_rotate_noalloc(pool, cfg, runs)
        assert e.value.code == "ARG", runs
    # refused under stream capture (its host-side list would be read only at replay)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    x = torch.zeros(16, device="cuda")
    with torch.cuda.graph(g, stream=s):
        x.add_(1)
        with pytest.raises(akv.AKVError) as e:
            akv.repos_rotate_noalloc(pool, cfg, [[3, 3, 0, 8, 5]], stream=s)
        assert e.value.code == "ARG"
    del g
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
    # disjoint rows of one page, and a copy reading rows that an in-place run rotates, are fine
    akv.repos_rotate_noalloc(pool, cfg, [[3, 3, 0, 8, 5], [3, 3, 8, 16, 7], [4, 9, 0, 16, 1], [4, 4, 0, 16, 2]])
    torch.cuda.synchronize()
    assert not torch.equal(pool, before)
