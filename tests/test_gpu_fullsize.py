"""Parity at the workloads' full sizes, on sampled outputs (see tests/gpu_sampled.py).

* eight 64K-token sessions sharing a 4K prefix, 32 layers (~72 GB of pools):
  sampled rotated rows of every session and layer; attention on layers 0 and
  31 for three segment classes -- a session's first segment (shortest
  history, nothing hidden), a middle one, a session's last (longest history,
  most hidden spans);
* the Llama-3.1-70B-shaped 128K cache, 80 layers (~54 GB of pools): the
  in-place full-cache sweep with shifts up to +-64K, sampled rows; attention
  on layers 0 and 79 for the branches hiding the fewest and the most spans
  and the first and last branch;
* 16 DeepSeek-V2-Lite MLA sessions, 27 layers: the splice's K_pe rotation;
  attention of three sessions, every query row;
* the benchmark's compaction: the post-drop branch of the 32K trajectory over
  32 layers, shifts still pending (fused into the copy): sampled K rows
  against the oracle's rotation, sampled V rows bit-identical, attention over
  the compacted branch on layers 0 and 31;
* the post-drop 32K turn's attention-mass launch as the benchmark runs it
  (2,048 queries x 32 heads over 24,479 visible entries, automatic K-tile
  ranges): every token against the float64 oracle.
Attention samples (tests/gpu_sampled.py): in every checked segment, at least
256 random query rows (every row when there are fewer) plus the first and last
row of each query tile, so each work item of the launch, split or not, is
checked; each row against the segment's full visible KV, all query heads.
Bars as in the other GPU tests (rotated keys: one bf16 ulp plus the float32
rotation allowance, >= 99.9% bit-identical; attention: 2e-2 max-abs)."""
import gc

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


def release(c):
    del c
    gc.collect()
    torch.cuda.empty_cache()


def test_sampled_harness_on_small_cases():
    # the same sampled harness on scaled workloads (fast): fails early if the harness is wrong
    from gpu_sampled import SampledCase
    for w in (synth.sessions_64k(n_layers=2, n_sessions=3, prefix=1024, per_session=8192, q_per_seg=128,
                                 span_len=(64, 512)),
              synth.llama70b_128k(n_layers=2, total=16384, n_branches=4, q_per_branch=200)):
        c = SampledCase(w)
        c.run()
        rng = np.random.default_rng(3)
        n_rot, _ = c.check_repos(512, rng)
        assert n_rot > 50
        c.check_attention(1, 6, rng, segments=[0, len(w.segments) - 1])
        release(c)


def test_sessions_64k_full_size_sampled():
    from gpu_sampled import SampledCase
    w = synth.sessions_64k()
    c = SampledCase(w)
    c.run()
    rng = np.random.default_rng(11)
    n_rot, worst = c.check_repos(4096, rng)
    assert n_rot > 1000
    last = len(w.segments) - 1
    by_seq = {}
    for i, g in enumerate(w.segments):
        by_seq.setdefault(g["seq"], []).append(i)
    seqs = sorted(by_seq)
    first = next(by_seq[q][0] for q in seqs if not w.segments[by_seq[q][0]]["hide"])
    middle = by_seq[seqs[len(seqs) // 2]][len(by_seq[seqs[len(seqs) // 2]]) // 2]
    final = max((by_seq[q][-1] for q in seqs), key=lambda i: (len(w.segments[i]["hide"]), i))
    assert w.segments[final]["hide"]
    for layer in (0, w.shape.n_layers - 1):
        _, n = c.check_attention(layer, 256, rng, segments=[first, middle, final])
        assert n >= 3 * 256
    release(c)


def test_llama70b_128k_full_size_sampled():
    from gpu_sampled import SampledCase
    w = synth.llama70b_128k()
    c = SampledCase(w)
    c.run()
    rng = np.random.default_rng(12)
    n_rot, worst = c.check_repos(4096, rng)
    assert n_rot > 1000
    n_hidden = [sum(b - a for a, b in g["hide"]) for g in w.segments]
    segs = sorted({0, len(w.segments) - 1, int(np.argmin(n_hidden)), int(np.argmax(n_hidden))})
    for layer in (0, w.shape.n_layers - 1):
        _, n = c.check_attention(layer, 256, rng, segments=segs)
        assert n >= len(segs) * 256
    release(c)


def test_mla_16_sessions_full_size_sampled():
    from gpu_sampled import SampledCase
    w = synth.mla_dsv2lite(concurrency=16)
    c = SampledCase(w)
    c.run()
    rng = np.random.default_rng(13)
    n_rot, worst = c.check_repos(4096, rng)
    assert n_rot > 1000
    for layer in (0, w.shape.n_layers - 1):
        _, n = c.check_attention(layer, 256, rng, segments=[0, 7, 15])
        assert n == 3 * 256      # every query row of the three sessions
    release(c)


def test_mass_32k_turn_full_size():
    from test_gpu_mass import mass_case
    mass_case(synth.llama8b_32k(seed=0, fork=True))


def test_compaction_32k_branch_full_size_sampled():
    from gpu_sampled import SampledCase
    from test_gpu_compact import remap_segments
    w = synth.llama8b_32k(fork=True, n_layers=32)
    w.n_pages += 2 * (32768 // 16)
    c = SampledCase(w)
    c.run(flush=False)
    sid = c.names["F"]
    assert c.model.fragmentation(sid) > 0.2
    states = {sid: c.model.state(sid)}
    copies = c.compact("F")
    assert sum(1 for cp in copies if cp[6]) > 1000, "no pending shift fused into the copy"
    rng = np.random.default_rng(5)
    n_rot, _ = c.check_repos(4096, rng)
    assert n_rot > 500
    assert c.check_values(2048, rng) > 1000
    w.segments = remap_segments(w, states, c.names)
    for layer in (0, w.shape.n_layers - 1):
        _, n = c.check_attention(layer, 256, rng)
        assert n >= 256
    release(c)
