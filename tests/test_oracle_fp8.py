"""Pins for the 8-bit forward oracle (oracle/skiparse_fp8_oracle.py), on CPU.

Each check rests on something other than the oracle's own arithmetic: the
E4M3 format's definition, brute-force rounding, the exact softmax attention of
the main oracle (itself pinned against library routines), and closed forms.
"""
import math

import numpy as np
import pytest

from oracle import skiparse_fp8_oracle as F
from oracle import skiparse_oracle as O


def test_e4m3_grid_from_the_format():
    g = F.e4m3_values()
    assert len(g) == 127                              # 128 codes per sign, minus NaN
    assert g[0] == 0.0 and g[1] == 2.0 ** -9          # smallest subnormal: 1/8 * 2^-6
    assert g[8] == 2.0 ** -6                          # smallest normal
    assert g[-1] == 448.0 and g[-2] == 416.0
    assert np.all(np.diff(g) > 0)
    # within a binade [2^e, 2^(e+1)) the step is 2^(e-3)
    for e in range(-6, 8):
        sel = g[(g >= 2.0 ** e) & (g < 2.0 ** (e + 1))]
        assert np.allclose(np.diff(sel), 2.0 ** (e - 3))


def _brute_round(x):
    g = F.e4m3_values()
    a = min(abs(x), 448.0)
    d = np.abs(g - a)
    best = np.flatnonzero(d == d.min())
    idx = best[0] if len(best) == 1 else [i for i in best if i % 2 == 0][0]   # tie: even code
    return math.copysign(g[idx], x)


def test_round_e4m3_matches_brute_force_including_ties():
    g = F.e4m3_values()
    mids = (g[:-1] + g[1:]) / 2                       # exact ties
    rs = np.random.RandomState(3)
    xs = np.concatenate([mids, -mids, g, rs.randn(400) * 50, rs.rand(50) * 2.0 ** -8, [500.0, -1e6, 0.0]])
    got = F.round_e4m3(xs)
    want = np.array([_brute_round(x) for x in xs])
    assert np.array_equal(got, want)
    assert F.round_e4m3(np.array([1e9]))[0] == 448.0  # saturating


def test_row_quantizer_reconstructs_within_half_ulp():
    rs = np.random.RandomState(5)
    x = rs.randn(7, 3, 128) * np.array([1e-3, 1.0, 50.0])[None, :, None]
    codes, scale = F.quantize_rows(x)
    assert np.all(np.abs(codes) <= 448.0)
    assert np.allclose(np.abs(codes).max(axis=-1), 448.0)      # each row's max maps to 448
    err = np.abs(codes * scale[..., None] - x)
    # half an ulp: relative 2^-4 in normal range, absolute 2^-10 * scale below it
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale[..., None])
    assert np.all(err <= bound * (1 + 1e-12))
    zc, zs = F.quantize_rows(np.zeros((2, 128)))
    assert np.all(zc == 0) and np.all(zs == 1.0)


def test_block_quantizer_one_scale_per_128_rows():
    rs = np.random.RandomState(4)
    x = rs.randn(300, 64)
    x[130] *= 10.0                                     # an outlier row sets block 1's scale
    codes, scale = F.quantize_blocks(x)
    assert np.all(scale[:128] == scale[0]) and np.all(scale[128:256] == scale[128]) and np.all(scale[256:] == scale[256])
    assert np.isclose(scale[128], np.abs(x[128:256]).max() / 448.0)
    assert np.isclose(np.abs(codes[128:256]).max(), 448.0)
    assert np.all(np.abs(codes * scale[:, None] - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) * (1 + 1e-12))


def test_channel_quantizer_scales_over_tokens():
    rs = np.random.RandomState(6)
    v = rs.randn(2, 300, 3, 64)
    codes, scale = F.quantize_channels(v)
    assert scale.shape == (2, 3, 64)
    assert np.allclose(np.abs(codes).max(axis=1), 448.0)
    assert np.allclose(scale, np.abs(v).max(axis=1) / 448.0)


@pytest.mark.parametrize("mode", [O.SINGLE, O.GROUP])
@pytest.mark.parametrize("peaky", [False, True])
def test_blocked_online_softmax_is_exact_without_quantization(mode, peaky):
    """With every rounding replaced by the identity the blocked, lazily rescaled
    online softmax must equal plain softmax attention (scopes of 3 blocks)."""
    B, heads, D, T, H, W, k = 1, 2, 64, 3, 10, 20, 2     # L = 300: blocks of 128, 128, 44
    rs = np.random.RandomState(11)
    q = rs.randn(B, T * H * W, heads, D) * (6.0 if peaky else 1.0)
    kk = rs.randn(B, T * H * W, heads, D)
    v = rs.randn(B, T * H * W, heads, D)
    if peaky:
        # make later blocks win the max by a wide margin so the lazy rule rescales
        kk[:, ::7] *= 3.0
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, mode, quantize=False)
    rout, rlse = O.skiparse_fwd(q, kk, v, T, H, W, k, mode)
    assert np.max(np.abs(out - rout)) < 1e-12
    assert np.max(np.abs(lse - rlse)) < 1e-10


def test_quantized_p_never_saturates():
    """P is below 2^LAZY_LOG2 by the lazy rule, so its scaled codes stay below
    E4M3's largest finite value."""
    assert 2.0 ** F.LAZY_LOG2 * F.P_SCALE <= F.E4M3_MAX


def test_uniform_attention_closed_form():
    """q = 0: every score is 0, P = 1 is exact in E4M3 (P * 2^6 = 64), so each
    output row is the mean over its scope of the dequantized v."""
    B, heads, D, T, H, W, k = 1, 1, 64, 2, 8, 16, 2
    N = T * H * W
    rs = np.random.RandomState(2)
    q = np.zeros((B, N, heads, D))
    kk = rs.randn(B, N, heads, D)
    v = rs.randn(B, N, heads, D)
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, O.GROUP)
    v8, sv = F.quantize_channels(v)
    vd = v8 * sv[:, None]
    L = N // k
    for s in range(k):
        toks = O.scope_tokens(N, k, O.GROUP, s)
        want = vd[0, toks, 0].mean(axis=0)
        assert np.allclose(out[0, toks, 0], want[None, :], atol=1e-12)
        assert np.allclose(lse[0, 0, toks], math.log(L))


def test_quantized_forward_error_is_of_the_expected_size():
    """8-bit operands change the result by about the E4M3 rounding error: its
    relative step is 2^-3, so q, k, P and v each carry ~3 % RMS rounding error,
    which add roughly in quadrature to ~5-6 % at the output. Bound: 8 %, far
    from exact (quantization is on) and far from garbage (~100 %)."""
    B, heads, D, T, H, W, k = 1, 2, 128, 2, 8, 16, 2
    rs = np.random.RandomState(9)
    q, kk, v = (rs.randn(B, T * H * W, heads, D) for _ in range(3))
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, O.SINGLE)
    rout, rlse = O.skiparse_fwd(q, kk, v, T, H, W, k, O.SINGLE)
    rel = np.sqrt(np.sum((out - rout) ** 2) / np.sum(rout ** 2))
    assert 1e-3 < rel < 8e-2
    assert np.max(np.abs(lse - rlse)) < 5e-2


@pytest.mark.parametrize("mode", [O.SINGLE, O.GROUP], ids=["single", "group"])
def test_scope_rows_match_the_whole_forward(mode):
    """The row-sampled scope routine (used on full-size inputs) gives the whole
    8-bit forward's numbers for the rows it is asked for: several key blocks
    with a ragged last one, two batches and heads (v's channel scales span all
    tokens of a (batch, head))."""
    B, heads, D, T, H, W, k = 2, 2, 64, 3, 10, 12, 2
    N = T * H * W
    rs = np.random.RandomState(21)
    q, kk, v = (rs.randn(B, N, heads, D) for _ in range(3))
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, mode)
    L = N // k
    rows = np.array([0, 1, 127, 128, 129, L - 1])
    for b, h, s in [(0, 0, 0), (1, 1, 1), (1, 0, 0)]:
        tok, o, l = F.skiparse_fwd_fp8_scope(q, kk, v, T, H, W, k, mode, b, h, s, rows)
        assert np.array_equal(tok, O.scope_tokens(N, k, mode, s)[rows])
        assert np.allclose(o, out[b, tok, h], rtol=0, atol=1e-12)
        assert np.allclose(l, lse[b, h, tok], rtol=0, atol=1e-12)
