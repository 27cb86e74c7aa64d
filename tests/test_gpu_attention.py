"""segment_batch_attn on the GPU against the float64 oracle.

Bar: bf16 output vs the float64 oracle (on the same bf16 inputs) within
max-abs 2e-2; LSE within 2e-2 absolute.  Configs that the oracle finishes in
seconds are compared in full; large ones on sampled query rows (each against
its full visible KV list), always including the first and last rows and the
rows at 128-row tile boundaries."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from agentic_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 2e-2


def sample_rows(q_len, k, rng, tpt):
    rows = {0, q_len - 1}
    for t in range(tpt, q_len, tpt):
        rows.update({t - 1, t})
    extra = rng.choice(q_len, size=min(k, q_len), replace=False)
    rows.update(int(x) for x in extra)
    return np.array(sorted(r for r in rows if 0 <= r < q_len))


def check(w, k_rows=None, seed=0, split=0):
    from gpu_case import Case
    c = Case(w)
    c.run_ops()
    c.flush_segments()
    c.eng.set_attention_split(split)
    q32, o, lse = c.attend_gpu()
    rng = np.random.default_rng(seed)
    G = w.shape.n_q_heads // w.shape.n_kv_heads
    worst = 0.0
    written = np.zeros(o.shape[0], bool)
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"]) if k_rows is None else sample_rows(g["q_len"], k_rows, rng, 128 // G)
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        got_o = o[g["q_row0"] + rows]
        got_lse = lse[g["q_row0"] + rows]
        err = np.abs(got_o - want_o).max()
        worst = max(worst, err)
        assert err <= ATOL, f"segment {i}: max abs error {err}"
        assert np.abs(got_lse - want_lse).max() <= ATOL
        written[g["q_row0"]:g["q_row0"] + g["q_len"]] = True
    assert np.isfinite(o[written]).all()
    return c, worst


def test_tiny_two_branches_one_launch():
    check(synth.tiny())


def test_llama8b_32k_full_size_sampled():
    check(synth.llama8b_32k(), k_rows=96)


def test_llama8b_small_full_compare():
    check(synth.llama8b_32k(total=4096, n_new=300))   # ragged query tail (300 = 9 tiles + 12)


def test_sessions_many_segments_with_hidden_spans():
    w = synth.sessions_64k(n_layers=1, n_sessions=3, prefix=1024, per_session=8192, q_per_seg=128,
                           span_len=(64, 512))
    check(w, k_rows=40)


def test_llama70b_shape_group_8_branches():
    w = synth.llama70b_128k(n_layers=1, total=16384, n_branches=4, q_per_branch=200)
    check(w, k_rows=40)


def test_single_query_and_single_key():
    w = synth.tiny()
    w.ops = [("alloc", "A"), ("append", "A", 1, "one"), ("alloc", "B"), ("append", "B", 37, "b"),
             ("drop", "B", 3, 30)]
    w.segments = [dict(seq="A", kv_end=1, q_len=1, hide=[], q_row0=0),
                  dict(seq="B", kv_end=37, q_len=5, hide=[], q_row0=1),
                  dict(seq="B", kv_end=35, q_len=1, hide=[(0, 2)], q_row0=6)]
    c, _ = check(w)


def test_partial_pages_everywhere():
    # drops at odd offsets leave partial runs in most tiles
    w = synth.tiny()
    ops = [("alloc", "A"), ("append", "A", 700, "ctx")]
    for a in range(5, 600, 37):
        ops.append(("drop", "A", a, a + 11))
    ops.append(("append", "A", 70, "new"))
    w.ops = ops
    w.segments = [dict(seq="A", kv_end=770, q_len=70, hide=[(300, 333)], q_row0=0)]
    check(w)


def test_mla_spliced_sessions():
    # DeepSeek-V2-Lite MLA shape: 16 heads over one latent (d_qk 512 + 64, d_v 512), page 64,
    # two ~17K-token sessions each spliced (2,016 -> 32 tokens), 256 new queries per session
    check(synth.mla_dsv2lite(n_layers=2, concurrency=2), k_rows=48)


def test_mla_small_full_compare():
    check(synth.mla_dsv2lite(n_layers=1, concurrency=1, prompt=3000, span=700, stub=20, n_new=100))


@pytest.mark.parametrize("page,split", [(16, 0), (32, 0), (128, 0), (16, 4)])
def test_mla_page_sizes_forks_and_drops(page, split):
    # MLA at other page sizes: a 64-key unit spans several pages (16, 32) or
    # half a page (128).  Branch B is a fork whose repositioned K_pe pages are
    # copies, so key and latent page ids differ and a unit's pages are not
    # always consecutive; dropped and hidden spans leave partial pages; 100
    # and 36 queries give odd query-tile counts (the pair's second tile is a
    # stand-in that writes nothing).
    import dataclasses
    w = synth.mla_dsv2lite(n_layers=1, concurrency=1)
    w.shape = dataclasses.replace(w.shape, page_size=page)
    w.ops = [("alloc", "A"), ("append", "A", 1500, "ctx"),
             ("fork", "B", "A", 1500),
             ("drop", "B", 100, 333), ("repos", "B", 333, 1500, -233),
             ("drop", "A", 700, 717), ("drop", "A", 901, 950),
             ("append", "A", 100, "newA"), ("append", "B", 36, "newB")]
    w.segments = [dict(seq="A", kv_end=1600, q_len=100, hide=[(40, 77)], q_row0=0),
                  dict(seq="B", kv_end=1536, q_len=36, hide=[], q_row0=100)]
    w.n_pages = 3 * (1600 // page + 4) + 16
    check(w, split=split)


@pytest.mark.parametrize("split", [0, 2])
def test_mla_tiny_sessions(split):
    # Degenerate MLA launches: a single query (one 8-token tile, 16 rows of 128
    # valid, its pair partner a shadow), key lists shorter than one tile, a
    # tile boundary exactly at the last key, several sessions in one launch.
    w = synth.mla_dsv2lite(n_layers=1, concurrency=1)
    w.ops, w.segments, row = [], [], 0
    for i, (prompt, q) in enumerate([(10, 1), (70, 3), (119, 9), (247, 17), (600, 1)]):
        name = f"S{i}"
        w.ops += [("alloc", name), ("append", name, prompt, f"p{i}"), ("append", name, q, f"n{i}")]
        w.segments.append(dict(seq=name, kv_end=prompt + q, q_len=q, hide=[], q_row0=row))
        row += q
    w.n_pages = 64
    check(w, split=split)


# Split-KV: an item's KV tiles cut into S parts whose partial (O, m, l) the
# combine kernel merges.  Forced factors cover parts that see no key of the
# shorter query tile (GQA), ragged part boundaries, and both MLA halves.
@pytest.mark.parametrize("split", [1, 2, 3, 8])
def test_split_kv_gqa_full_compare(split):
    check(synth.llama8b_32k(total=4096, n_new=300), split=split)


@pytest.mark.parametrize("split", [2, 5])
def test_split_kv_partial_pages(split):
    w = synth.tiny()
    ops = [("alloc", "A"), ("append", "A", 900, "ctx")]
    for a in range(5, 800, 41):
        ops.append(("drop", "A", a, a + 13))
    ops.append(("append", "A", 200, "new"))
    w.ops = ops
    w.n_pages = 128
    w.segments = [dict(seq="A", kv_end=1100, q_len=200, hide=[(300, 333)], q_row0=0)]
    check(w, split=split)


@pytest.mark.parametrize("split", [3, 8])
def test_split_kv_mla_full_compare(split):
    check(synth.mla_dsv2lite(n_layers=1, concurrency=1, prompt=3000, span=700, stub=20, n_new=100), split=split)


def test_split_kv_many_segments_group_8():
    w = synth.llama70b_128k(n_layers=1, total=16384, n_branches=4, q_per_branch=200)
    check(w, k_rows=40, split=4)


def test_outlier_keys_exercise_lazy_rescale():
    # Keys scaled up by 12-30x give score jumps far beyond the 2^8 lazy-rescale threshold:
    # inside a tile (the second 64-key half raises the running max after the first half's P
    # was formed) and across tiles (O rescaled in TMEM).  Same values on both sides.
    from gpu_case import Case

    class Outliers(Case):
        def _values(self, key, n):
            k32, v32 = super()._values(key, n)
            k32 = k32.copy()
            k32[:, 37::97] *= 12.0
            k32[:, 101::251] *= 30.0
            return k32, v32

    w = synth.llama8b_32k(total=2048, n_new=200)
    c = Outliers(w)
    c.run_ops()
    c.flush_segments()
    q32, o, lse = c.attend_gpu()
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"])
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        assert np.abs(o[g["q_row0"] + rows] - want_o).max() <= ATOL
        assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL


def test_mla_outlier_keys_exercise_lazy_rescale():
    # MLA keys are [latent | K_pe]: scale both parts (and so the latent value) of some tokens
    from gpu_case import Case

    class Outliers(Case):
        def _values(self, key, n):
            k32, v32 = super()._values(key, n)
            k32, v32 = k32.copy(), v32.copy()
            for a, step, f in ((37, 97, 6.0), (101, 251, 12.0)):
                k32[:, a::step] *= f
                v32[:, a::step] *= f
            return k32, v32

    w = synth.mla_dsv2lite(n_layers=1, concurrency=1, prompt=3000, span=700, stub=20, n_new=100)
    c = Outliers(w)
    c.run_ops()
    c.flush_segments()
    q32, o, lse = c.attend_gpu()
    for i, g in enumerate(w.segments):
        rows = np.arange(g["q_len"])
        want_o, want_lse = c.attend_oracle(q32, i, rows)
        scale = max(1.0, float(np.abs(want_o).max()))
        assert np.abs(o[g["q_row0"] + rows] - want_o).max() <= ATOL * scale
        assert np.abs(lse[g["q_row0"] + rows] - want_lse).max() <= ATOL
