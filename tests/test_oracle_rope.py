"""Pins for oracle.rope: RoPE angles, the rotation, and the repos primitive."""
import itertools

import numpy as np
import pytest

from oracle import rope

RNG = np.random.default_rng(1)


def test_theta_closed_form():
    th = rope.theta(64, 1.0e4)
    assert th[0] == 1.0
    assert np.isclose(th[1], 1.0e4 ** (-1.0 / 32.0), rtol=1e-15)
    assert np.isclose(th[-1], 1.0e4 ** (-62.0 / 64.0), rtol=1e-15)
    assert np.all(np.diff(th) < 0)


@pytest.mark.parametrize("layout", ["interleaved", "half"])
def test_rope_equals_complex_multiplication(layout):
    # Independent formulation: each pair (a, b) is the complex number a + ib,
    # and RoPE at position m multiplies it by exp(i m theta_j).
    d, base = 128, 5.0e5
    x = RNG.standard_normal((7, d))
    m = RNG.integers(-70000, 70000, size=7)
    a, b = rope.pair_indices(d, layout)
    z = (x[:, a] + 1j * x[:, b]) * np.exp(1j * m[:, None] * rope.theta(d, base))
    got = rope.rope(x, m, base, layout)
    assert np.allclose(got[:, a], z.real, rtol=0, atol=1e-12)
    assert np.allclose(got[:, b], z.imag, rtol=0, atol=1e-12)


def test_rotation_sign_on_unit_vector():
    # R(phi) (1, 0) = (cos phi, sin phi): pair 0 has theta_0 = 1, so phi = delta.
    k = np.zeros(64)
    k[0] = 1.0
    out = rope.repos(k, 3, 1.0e4)
    assert np.isclose(out[0], np.cos(3.0)) and np.isclose(out[1], np.sin(3.0))


def test_matches_blog_delta_matrix_with_opposite_sign():
    # The AKV blog moves a key from m to m - D with [[cos, sin], [-sin, cos]] (D theta);
    # with delta = -D this is our R(delta).
    d, base, D = 64, 1.0e4, 37
    k = RNG.standard_normal(d)
    th = rope.theta(d, base)
    c, s = np.cos(D * th), np.sin(D * th)
    blog = np.empty(d)
    blog[0::2] = c * k[0::2] + s * k[1::2]
    blog[1::2] = -s * k[0::2] + c * k[1::2]
    assert np.allclose(rope.repos(k, -D, base), blog, atol=1e-13)


@pytest.mark.parametrize("layout", ["interleaved", "half"])
def test_F1_repos_of_rope_is_rope_at_new_position(layout):
    d, base = 128, 5.0e5
    x = RNG.standard_normal((50, d))
    m = RNG.integers(0, 131072, size=50)
    delta = RNG.integers(-65536, 65537, size=50)
    lhs = rope.repos(rope.rope(x, m, base, layout), delta, base, layout)
    rhs = rope.rope(x, m + delta, base, layout)
    assert np.max(np.abs(lhs - rhs)) < 1e-9


def test_F2_composed_directives_equal_one_rotation():
    d, base = 128, 5.0e5
    k = RNG.standard_normal((20, d))
    deltas = RNG.integers(-4000, 4000, size=(20, 4))
    step = k
    for j in range(4):
        step = rope.repos(step, deltas[:, j], base)
    once = rope.repos(k, deltas.sum(axis=1), base)
    assert np.max(np.abs(step - once)) < 1e-11


def test_identity_inverse_and_norms():
    d, base = 128, 5.0e5
    k = RNG.standard_normal((30, d))
    assert np.array_equal(rope.repos(k, np.zeros(30), base), k)         # delta 0 is exact
    back = rope.repos(rope.repos(k, np.full(30, 12345), base), np.full(30, -12345), base)
    assert np.max(np.abs(back - k)) < 1e-12
    r = rope.repos(k, np.full(30, -777), base)
    assert np.allclose(r[:, 0::2] ** 2 + r[:, 1::2] ** 2, k[:, 0::2] ** 2 + k[:, 1::2] ** 2, atol=1e-12)


def test_relative_position_property():
    # q_n . k_m depends only on m - n (blog section 2), so shifting both by c changes nothing.
    d, base = 128, 5.0e5
    q, k = RNG.standard_normal(d), RNG.standard_normal(d)
    for n, m, c in itertools.product([0, 17, 4000], [3, 999, 30000], [-5000, 1, 65536]):
        a = rope.rope(q, n, base) @ rope.rope(k, m, base)
        b = rope.rope(q, n + c, base) @ rope.rope(k, m + c, base)
        assert abs(a - b) < 1e-9


def test_compact_copy_rotates_by_the_pending_shift_and_copies_values():
    # a key stored unrotated (position 0) and moved by delta must equal RoPE at position delta
    # (closed form of [AKV-blog] section 2); values are copied bit for bit
    from oracle import bf16, kernels, rope
    rng = np.random.default_rng(3)
    for layout in ("interleaved", "half"):
        k = bf16.round_bf16(rng.standard_normal((1, 4, 2, 8, 64)))
        v = bf16.round_bf16(rng.standard_normal((1, 4, 2, 8, 32)))
        copies = [(0, 1, 3, 2, 3, 0, 777), (0, 1, 5, 2, 3, 1, 0)]
        ko, vo = kernels.compact_copy(k, v, copies, 1.0e4, layout)
        want = bf16.round_bf16(rope.rope(k[:, 0, :, 3, :], np.full((1, 2), 777.0), 1.0e4, layout))
        assert np.array_equal(ko[:, 2, :, 0, :], want)
        assert np.array_equal(ko[:, 2, :, 1, :], k[:, 0, :, 5, :])
        assert np.array_equal(vo[:, 3, :, 0, :], v[:, 1, :, 3, :])
        assert np.array_equal(vo[:, 3, :, 1, :], v[:, 1, :, 5, :])
