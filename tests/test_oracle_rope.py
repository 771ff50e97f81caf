"""Pins for the oracle's 3D RoPE (CPU only).

The pages fix only that RoPE is applied to q and k at the original token
positions before the rearrange ("Open-Sora Plan" docs, "Skiparse Attention",
implementation note); the formula itself is this library's reading (axis split
D/4, 3D/8, 3D/8; adjacent channel pairs; theta**(-2j/d)). The pins check the
oracle against an independent complex-multiplication form, the identity at
position 0, norm preservation, the relative-position property and the
inverse rotation.
"""
import numpy as np
import pytest

from oracle import skiparse_oracle as O


def _x(B, N, h, D, seed=0):
    return np.random.default_rng(seed).standard_normal((B, N, h, D))


@pytest.mark.parametrize("D", [16, 64, 128])
def test_rope_matches_complex_closed_form(D):
    T, H, W = 3, 4, 5
    x = _x(2, T * H * W, 2, D)
    a = O.apply_rope(x, T, H, W, 10000.0)
    b = O.rope_closed_form(x, T, H, W, 10000.0)
    assert np.max(np.abs(a - b)) < 1e-13


def test_rope_identity_at_origin():
    x = _x(1, 1, 3, 64)
    assert np.array_equal(O.apply_rope(x, 1, 1, 1, 10000.0), x)


@pytest.mark.parametrize("D", [64, 128])
def test_rope_preserves_pair_norms(D):
    T, H, W = 2, 8, 8
    x = _x(1, T * H * W, 2, D)
    y = O.apply_rope(x, T, H, W, 10000.0)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.max(np.abs(nx - ny)) < 1e-12


def test_rope_inverse_is_transpose():
    T, H, W = 4, 8, 8
    x = _x(1, T * H * W, 2, 64)
    y = O.apply_rope(O.apply_rope(x, T, H, W, 10000.0), T, H, W, 10000.0, inverse=True)
    assert np.max(np.abs(x - y)) < 1e-12
    # <R q, g> == <q, R^T g> for random q, g
    g = _x(1, T * H * W, 2, 64, seed=3)
    lhs = np.sum(O.apply_rope(x, T, H, W, 10000.0) * g)
    rhs = np.sum(x * O.apply_rope(g, T, H, W, 10000.0, inverse=True))
    assert abs(lhs - rhs) < 1e-9


def test_rope_relative_position_property():
    """<R(p) q, R(p') k> depends only on p' - p, axis by axis."""
    D = 64
    T, H, W = 6, 6, 6
    rng = np.random.default_rng(5)
    q = rng.standard_normal(D)
    k = rng.standard_normal(D)
    N = T * H * W
    Q = np.broadcast_to(q, (1, N, 1, D)).copy()
    K = np.broadcast_to(k, (1, N, 1, D)).copy()
    Qr = O.apply_rope(Q, T, H, W, 10000.0)[0, :, 0]
    Kr = O.apply_rope(K, T, H, W, 10000.0)[0, :, 0]

    def tok(t, h, w):
        return (t * H + h) * W + w

    pairs =[((0, 0, 0), (1, 2, 3)), ((2, 1, 1), (3, 3, 4)), ((4, 3, 2), (5, 5, 5))]
    for p, p2 in pairs:
        v1 = Qr[tok(*p)] @ Kr[tok(*p2)]
        # shift both positions by the same amount on every axis
        s = (1, 0, 0) if p2[0] < T - 1 else (0, 0, 0)
        v2 = Qr[tok(*[a + b for a, b in zip(p, s)])] @ Kr[tok(*[a + b for a, b in zip(p2, s)])]
        assert abs(v1 - v2) < 1e-12
        # and equals <q, R(p'-p) k> built with a zero origin for q
        if all(b >= a for a, b in zip(p, p2)):
            dq = tok(0, 0, 0)
            dk = tok(*[b - a for a, b in zip(p, p2)])
            assert abs(v1 - Qr[dq] @ Kr[dk]) < 1e-12


def test_rope_chunk_split_and_angle_by_hand():
    """One token at (t, h, w) = (2, 1, 3), D = 16, theta = 1e4, worked by hand:
    chunks t: channels 0-3 (d=4), h: 4-9 (d=6), w: 10-15 (d=6).
    Unit vector in channel 0 rotates by angle t*1 = 2 into (cos 2, sin 2);
    channel 2 (pair 1 of the t chunk, omega = 1e4**(-1/2) = 0.01) by 0.02;
    channel 4 (pair 0 of the h chunk) by h = 1;
    channel 12 (pair 1 of the w chunk, omega = 1e4**(-1/3)) by 3 * 0.0464158883361278."""
    T, H, W, D = 3, 2, 4, 16
    i = (2 * H + 1) * W + 3
    for ch, ang in [(0, 2.0), (2, 0.02), (4, 1.0), (12, 3 * 0.0464158883361278)]:
        x = np.zeros((1, T * H * W, 1, D))
        x[0, i, 0, ch] = 1.0
        y = O.apply_rope(x, T, H, W, 10000.0)[0, i, 0]
        assert abs(y[ch] - np.cos(ang)) < 1e-14 and abs(y[ch + 1] - np.sin(ang)) < 1e-14
        others = np.delete(y, [ch, ch + 1])
        assert np.all(others == 0)
