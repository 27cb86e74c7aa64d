"""Pins for oracle.attention and oracle.kernels (attention and repos over pools)."""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle import attention, bf16, kernels, rope
from oracle.cache import CacheModel

RNG = np.random.default_rng(3)


def sdpa(q, k, v, mask, scale):
    """torch's scaled_dot_product_attention in float64 (q [n,d], k [N,d], mask [n,N] bool)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=t(mask), scale=scale)
    return o[0, 0].numpy()


def test_masked_attention_matches_sdpa_and_logsumexp():
    n, N, d, dv = 9, 40, 32, 24
    q, k, v = RNG.standard_normal((n, d)), RNG.standard_normal((N, d)), RNG.standard_normal((N, dv))
    mask = RNG.random((n, N)) < 0.6
    mask[:, 0] = True
    o, lse = attention.masked_attention(q, k, v, mask, 0.17)
    assert np.allclose(o, sdpa(q, k, v, mask, 0.17), atol=1e-12)
    s = np.where(mask, 0.17 * q @ k.T, -np.inf)
    assert np.allclose(lse, logsumexp(s, axis=1), atol=1e-12)


def test_single_visible_key_and_identical_keys():
    d = 16
    q, k, v = RNG.standard_normal((3, d)), RNG.standard_normal((5, d)), RNG.standard_normal((5, 7))
    mask = np.zeros((3, 5), bool)
    mask[:, 2] = True
    o, _ = attention.masked_attention(q, k, v, mask, 1.0)
    assert np.allclose(o, v[2], atol=1e-14)
    same = np.repeat(k[:1], 5, axis=0)
    o, _ = attention.masked_attention(q, same, v, np.ones((3, 5), bool), 1.0)
    assert np.allclose(o, v.mean(axis=0), atol=1e-13)


def test_empty_row_gives_zero_and_minus_inf():
    o, lse = attention.masked_attention(np.ones((2, 4)), np.ones((3, 4)), np.ones((3, 4)),
                                        np.array([[False] * 3, [True] * 3]), 1.0)
    assert np.all(o[0] == 0) and lse[0] == -np.inf and np.allclose(o[1], 1.0)


def test_one_segment_over_whole_sequence_is_textbook_causal():
    n, d = 33, 64
    q, k, v = (RNG.standard_normal((n, 2, d)) for _ in range(3))
    o, _ = attention.segment_attention(q, k, v, 0.125)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1), torch.from_numpy(k).transpose(0, 1),
        torch.from_numpy(v).transpose(0, 1), is_causal=True, scale=0.125).transpose(0, 1).numpy()
    assert np.allclose(o, ref, atol=1e-12)


def test_grouped_query_heads_read_their_kv_head():
    q = RNG.standard_normal((4, 8, 16))
    k, v = RNG.standard_normal((10, 2, 16)), RNG.standard_normal((10, 2, 16))
    o, _ = attention.segment_attention(q, k, v, 0.25)
    for h in range(8):
        ref, _ = attention.segment_attention(q[:, h:h + 1], k[:, h // 4:h // 4 + 1], v[:, h // 4:h // 4 + 1], 0.25)
        assert np.allclose(o[:, h], ref[:, 0], atol=1e-14)


def build_pools(c, L, H, d, dv, seed):
    rng = np.random.default_rng(seed)
    kpool = bf16.round_bf16(rng.standard_normal((L, c.n_pages, H, c.page, d)))
    vpool = bf16.round_bf16(rng.standard_normal((L, c.n_pages, H, c.page, dv)))
    return kpool, vpool


def test_F3_drop_equals_dense_attention_with_minus_inf_columns():
    P, L, H, d = 16, 1, 2, 32
    c = CacheModel(32, P)
    s = c.seq_alloc()
    c.append(s, 150)
    c.drop(s, 20, 47)
    c.drop(s, 90, 91)
    kpool, vpool = build_pools(c, L, H, d, d, 0)
    q_len = 6
    runs, n = c.segment_runs(s, 150, q_len)
    q = RNG.standard_normal((q_len, 4, d))
    o, _ = kernels.attend_segment(q, kpool, vpool, 0, runs, 0.2)
    # dense side: every one of the 150 keys, dropped columns masked to -inf
    st = c.state(s)
    K = np.stack([kpool[0, st["k_page"][i], :, st["slot"][i]] for i in range(150)])
    V = np.stack([vpool[0, st["v_page"][i], :, st["slot"][i]] for i in range(150)])
    vis = np.array(st["visible"], bool)
    for r in range(q_len):
        tok = 150 - q_len + r
        mask = (vis & (np.arange(150) <= tok))[None]
        for h in range(4):
            ref = sdpa(q[r:r + 1, h], K[:, h // 2], V[:, h // 2], mask, 0.2)
            assert np.allclose(o[r, h], ref[0], atol=1e-12)


def test_F4_segment_batch_equals_one_dense_masked_attention():
    # Three sequential segments of one sequence with different visible sets,
    # against one dense [n_q x N] masked attention with per-row visibility.
    P, H, d = 16, 1, 16
    c = CacheModel(64, P)
    s = c.seq_alloc()
    c.append(s, 300)
    c.drop(s, 30, 60)
    segs = [(200, 10, [(100, 120)]), (250, 10, [(100, 120), (150, 170)]), (300, 10, [])]
    kpool, vpool = build_pools(c, 1, H, d, d, 1)
    st = c.state(s)
    K = np.stack([kpool[0, st["k_page"][i], 0, st["slot"][i]] for i in range(300)])
    V = np.stack([vpool[0, st["v_page"][i], 0, st["slot"][i]] for i in range(300)])
    q = RNG.standard_normal((30, 1, d))
    outs, rows_mask = [], []
    for j, (kv_end, q_len, hide) in enumerate(segs):
        runs, _ = c.segment_runs(s, kv_end, q_len, hide)
        o, _ = kernels.attend_segment(q[10 * j:10 * j + 10], kpool, vpool, 0, runs, 0.3)
        outs.append(o[:, 0])
        for r in range(q_len):
            m = np.array(st["visible"], bool) & (np.arange(300) <= kv_end - q_len + r)
            for a, b in hide:
                m[a:b] = False
            rows_mask.append(m)
    dense = sdpa(q[:, 0], K, V, np.stack(rows_mask), 0.3)
    assert np.allclose(np.concatenate(outs), dense, atol=1e-12)


def test_translation_invariance_of_attention_under_rope():
    d, base = 64, 1.0e4
    x_q, x_k, v = RNG.standard_normal((5, 1, d)), RNG.standard_normal((20, 1, d)), RNG.standard_normal((20, 1, d))
    pq, pk = np.arange(15, 20), np.arange(20)
    o1, _ = attention.segment_attention(rope.rope(x_q, pq[:, None], base), rope.rope(x_k, pk[:, None], base), v, 0.125)
    o2, _ = attention.segment_attention(rope.rope(x_q, pq[:, None] + 4321, base),
                                        rope.rope(x_k, pk[:, None] + 4321, base), v, 0.125)
    assert np.allclose(o1, o2, atol=1e-10)


def test_repos_runs_pool_level_F1_within_bf16_rounding():
    # Keys stored as bf16(rope(x, m)); after a flush by delta, each rotated
    # pair must lie within (input rounding error, which the rotation carries
    # over with its 2-norm) + (output rounding error) of rope(x, m + delta).
    P, L, H, d, base = 16, 2, 3, 64, 1.0e4
    c = CacheModel(16, P)
    s = c.seq_alloc()
    c.append(s, 64)
    x = RNG.standard_normal((L, 64, H, d))
    m = np.arange(64)
    kpool = np.zeros((L, 16, H, P, d))
    st = c.state(s)
    exact = rope.rope(x, m[None, :, None], base)
    for i in range(64):
        kpool[:, st["k_page"][i], :, st["slot"][i]] = bf16.round_bf16(exact[:, i])
    c.repos(s, 10, 50, -7)
    c.repos(s, 30, 64, 1000)
    runs = c.flush()
    out = kernels.repos_runs(kpool, runs, base)
    st = c.state(s)
    target = rope.rope(x, np.array(st["pos"])[None, :, None], base)
    stored = np.zeros_like(target)
    for i in range(64):
        stored[:, i] = bf16.round_bf16(exact[:, i])
    pair_norm = lambda a: np.sqrt(a[..., 0::2] ** 2 + a[..., 1::2] ** 2)
    for i in range(64):
        got = out[:, st["k_page"][i], :, st["slot"][i]]
        bound = 0.5 * pair_norm(bf16.ulp_bf16(stored[:, i])) + 0.5 * pair_norm(bf16.ulp_bf16(got)) + 1e-12
        assert np.all(pair_norm(got - target[:, i]) <= bound)
    # untouched rows stay bit-identical
    assert np.array_equal(out[:, 0, :, :10], kpool[:, 0, :, :10])


def test_repos_runs_copy_on_write_and_identity():
    P = 8
    c = CacheModel(16, P)
    s = c.seq_alloc()
    c.append(s, 16)
    f = c.seq_fork(s, 16)
    c.repos(f, 4, 12, 0)                 # delta 0: nothing to do
    assert c.flush() == []
    c.repos(f, 4, 12, 5)
    runs = c.flush()
    # both pages shared -> copied; visible tokens with delta 0 are copied unrotated
    assert runs == [(0, 2, 0, 4, 0), (0, 2, 4, 8, 5), (1, 3, 0, 4, 5), (1, 3, 4, 8, 0)]
    kpool = bf16.round_bf16(np.random.default_rng(0).standard_normal((1, 16, 1, P, 16)))
    out = kernels.repos_runs(kpool, runs, 1.0e4)
    assert np.array_equal(out[:, 2, :, 0:4], kpool[:, 0, :, 0:4])
    assert np.array_equal(out[:, :2], kpool[:, :2])   # the shared source pages are not written


# ------------------------------------------------------------ attention mass
def test_attention_mass_totals_rows_times_heads():
    # every query row's probabilities sum to one, for every head
    rng = np.random.default_rng(11)
    for q_len, kv_len, hq, hkv in ((1, 1, 4, 1), (5, 37, 8, 2), (16, 16, 4, 4)):
        q = rng.standard_normal((q_len, hq, 16))
        k = rng.standard_normal((kv_len, hkv, 16))
        m = attention.attention_mass(q, k, 0.25)
        assert abs(m.sum() - q_len * hq) < 1e-9 * q_len * hq
        assert np.all(m >= 0)


def test_attention_mass_identical_keys_closed_form():
    # identical keys: row i spreads its weight evenly over the kv_len - q_len + i + 1 entries it sees
    q_len, kv_len, hq = 6, 20, 3
    rng = np.random.default_rng(2)
    q = rng.standard_normal((q_len, hq, 8))
    k = np.tile(rng.standard_normal((1, 1, 8)), (kv_len, 1, 1))
    m = attention.attention_mass(q, k, 0.3)
    want = np.zeros(kv_len)
    for i in range(q_len):
        seen = kv_len - q_len + i + 1
        want[:seen] += hq / seen
    assert np.allclose(m, want, rtol=0, atol=1e-12)


def test_attention_mass_one_dominant_key():
    # a key far more aligned with every query than the others takes (almost) all the weight of
    # the rows that see it; rows that do not see it spread theirs over the rest
    q = np.ones((2, 2, 4))
    k = np.zeros((5, 1, 4))
    k[4] = 50.0                       # entry 4 is only visible to the last row (bottom-right)
    m = attention.attention_mass(q, k, 1.0)
    assert abs(m[4] - 2.0) < 1e-9     # last row, both heads
    assert np.allclose(m[:4], 2.0 / 4)  # first row (sees entries 0..3) spread evenly, both heads
