"""Pins for the Q/K/V projection + RoPE oracle (oracle/skiparse_proj_oracle.py), on CPU.

Each check rests on something other than the oracle's own arithmetic: a
pure-Python triple loop for the linear maps, the independent complex-number
RoPE (rope_closed_form), and properties of rotations.
"""
import numpy as np

from oracle import skiparse_oracle as O
from oracle import skiparse_proj_oracle as P


def _case(seed=0, B=2, T=2, H=2, W=3, C=10, heads=2, D=16):
    rs = np.random.RandomState(seed)
    N = T * H * W
    x = rs.randn(B, N, C)
    w = rs.randn(3 * heads * D, C)
    b = rs.randn(3 * heads * D)
    return x, w, b, dict(heads=heads, D=D, T=T, H=H, W=W)


def _brute_projection(x, w, b):
    B, N, C = x.shape
    out = np.zeros((B, N, w.shape[0]))
    for bi in range(B):
        for n in range(N):
            for o in range(w.shape[0]):
                acc = 0.0 if b is None else float(b[o])
                for c in range(C):
                    acc += float(x[bi, n, c]) * float(w[o, c])
                out[bi, n, o] = acc
    return out


def test_against_triple_loop_and_complex_rope():
    x, w, b, g = _case()
    q, k, v = P.qkv_rope(x, w, b, **g)
    y = _brute_projection(x, w, b)
    B, N = x.shape[:2]
    hd = g["heads"] * g["D"]
    shape = (B, N, g["heads"], g["D"])
    qr = O.rope_closed_form(y[..., :hd].reshape(shape), g["T"], g["H"], g["W"], 10000.0)
    kr = O.rope_closed_form(y[..., hd:2 * hd].reshape(shape), g["T"], g["H"], g["W"], 10000.0)
    assert np.allclose(q, qr, atol=1e-12)
    assert np.allclose(k, kr, atol=1e-12)
    assert np.allclose(v, y[..., 2 * hd:].reshape(shape), atol=1e-12)     # v is not rotated


def test_block_order_q_k_v():
    x, w, b, g = _case(1)
    hd = g["heads"] * g["D"]
    wk = np.zeros_like(w)
    wk[hd:2 * hd] = w[hd:2 * hd]                   # only K's rows
    q, k, v = P.qkv_rope(x, wk, None, **g)
    assert np.all(q == 0) and np.all(v == 0) and np.abs(k).max() > 0.1


def test_bias_enters_before_rope():
    """x = 0: q is the rotated bias, so it equals b_q only at position (0,0,0)."""
    x, w, b, g = _case(2)
    q, _, v = P.qkv_rope(np.zeros_like(x), w, b, **g)
    hd, D = g["heads"] * g["D"], g["D"]
    bq = b[:hd].reshape(g["heads"], D)
    assert np.allclose(q[:, 0], bq[None], atol=1e-12)                   # token 0: identity rotation
    assert not np.allclose(q[:, -1], bq[None], atol=1e-3)
    assert np.allclose(v, b[2 * hd:].reshape(g["heads"], D)[None, None], atol=1e-12)


def test_rotation_keeps_pair_norms():
    x, w, b, g = _case(3)
    q, _, _ = P.qkv_rope(x, w, b, **g)
    hd = g["heads"] * g["D"]
    plain = (x @ w.T + b)[..., :hd].reshape(q.shape)
    n_rot = q[..., 0::2] ** 2 + q[..., 1::2] ** 2
    n_plain = plain[..., 0::2] ** 2 + plain[..., 1::2] ** 2
    assert np.allclose(n_rot, n_plain, rtol=1e-12, atol=1e-12)


def test_row_sampler_matches_full():
    x, w, b, g = _case(4, B=3, T=3, H=2, W=4, C=12, heads=3, D=32)
    q, k, v = P.qkv_rope(x, w, b, **g)
    rows = [(0, 0), (2, 5), (1, 23), (2, 17)]
    qs, ks, vs = P.qkv_rope_rows(x, w, b, rows=rows, **g)
    for i, (bi, n) in enumerate(rows):
        assert np.allclose(qs[i], q[bi, n], atol=1e-12)
        assert np.allclose(ks[i], k[bi, n], atol=1e-12)
        assert np.allclose(vs[i], v[bi, n], atol=1e-12)


def test_prerotated_attention_equals_attention_with_rope():
    """theta = 0 takes q and k as already rotated: attention on RoPE'd inputs
    without rotation equals attention with rotation on the raw inputs, and the
    gradients relate by R^T (dq = R^T dq_rot), as the chain rule demands."""
    rs = np.random.RandomState(8)
    B, heads, D, T, H, W, k = 1, 2, 16, 2, 4, 4, 2
    N = T * H * W
    q, kk, v, do = (rs.randn(B, N, heads, D) for _ in range(4))
    assert np.array_equal(O.apply_rope(q, T, H, W, 0.0), q)
    qr, kr = O.apply_rope(q, T, H, W, 10000.0), O.apply_rope(kk, T, H, W, 10000.0)
    for mode in (O.SINGLE, O.GROUP):
        o1, l1 = O.skiparse_fwd(q, kk, v, T, H, W, k, mode)
        o0, l0 = O.skiparse_fwd(qr, kr, v, T, H, W, k, mode, theta=0.0)
        assert np.allclose(o0, o1, atol=1e-12) and np.allclose(l0, l1, atol=1e-12)
        dq1, dk1, dv1 = O.skiparse_bwd(q, kk, v, do, T, H, W, k, mode)[:3]
        dq0, dk0, dv0 = O.skiparse_bwd(qr, kr, v, do, T, H, W, k, mode, theta=0.0)[:3]
        assert np.allclose(O.apply_rope(dq0, T, H, W, 10000.0, inverse=True), dq1, atol=1e-12)
        assert np.allclose(O.apply_rope(dk0, T, H, W, 10000.0, inverse=True), dk1, atol=1e-12)
        assert np.allclose(dv0, dv1, atol=1e-12)
