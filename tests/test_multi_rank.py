"""The N > 1 path on CPU: two gloo ranks.

The cache path shards with no exchange (replicas: each rank serves its own
sessions), so the only cross-rank steps are the barrier around the timed
region and the maximum of the per-rank timings.  Each rank here runs the
turn's bookkeeping on its own seed through a metadata-only engine and checks
it against the oracle's bookkeeping, then the ranks reduce their timings."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from agentic_kv_cache_gb300 import akv, build, runner, synth
        from oracle.cache import CacheModel
        build.build()
        # this rank's own sessions: the 32K turn's history on a per-rank seed (replicas)
        w = synth.llama8b_32k(seed=rank, fork=True, total=4096, n_new=300)
        eng = akv.Engine(akv.config_from_shape(w.shape, w.n_pages), None)
        names = runner.run_ops(eng, w)
        model, mn = CacheModel(w.n_pages, w.shape.page_size), {}
        for op in w.ops:
            if op[0] == "alloc":
                mn[op[1]] = model.seq_alloc()
            elif op[0] == "fork":
                mn[op[1]] = model.seq_fork(mn[op[2]], op[3])
            elif op[0] == "append":
                model.append(mn[op[1]], op[2])
            elif op[0] == "drop":
                model.drop(mn[op[1]], op[2], op[3])
            elif op[0] == "repos":
                model.repos(mn[op[1]], op[2], op[3], op[4])
        same = True
        for name in names:
            got, want = eng.export_state(names[name]), model.state(mn[name])
            same = same and all(np.array_equal(np.asarray(got[k]), np.asarray(want[k])) for k in
                                ("k_page", "v_page", "slot", "pos", "delta", "visible"))
        tdist.barrier()
        # per-rank timings: rank r reports (r + 1, 10 (world - r)); the job's time is the maximum
        red = bench.max_over_ranks([float(rank + 1), 10.0 * (world - rank)], "cpu")
        out.put((rank, same, red, len(w.ops)))
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_timing_reduction():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    for rank, same, red, n_ops in results:
        assert same, f"rank {rank}: bookkeeping differs from the oracle"
        assert red == [float(world), 10.0 * world]
    # the ranks served different histories (their own seeds)
    assert results[0][3] > 0 and results[1][3] > 0
