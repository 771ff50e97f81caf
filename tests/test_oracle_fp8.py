"""Pins for the 8-bit forward oracle (oracle/skiparse_fp8_oracle.py), on CPU.

Each check rests on something other than the oracle's own arithmetic: the
E4M3 and INT8 formats' definitions, brute-force rounding, a pure-Python
restatement of the method on a tiny scope, the exact softmax attention of the
main oracle (itself pinned against library routines), and closed forms.
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


def _brute_round_e4m3(x):
    g = F.e4m3_values()
    a = min(abs(x), 448.0)
    d = np.abs(g - a)
    best = np.flatnonzero(d == d.min())
    idx = best[0] if len(best) == 1 else [i for i in best if i % 2 == 0][0]   # tie: even code
    return math.copysign(g[idx], x)


def _brute_round_int8(x):
    lo = math.floor(x)
    c = lo if x - lo < 0.5 else (lo + 1 if x - lo > 0.5 else (lo if lo % 2 == 0 else lo + 1))
    return float(min(127, max(-127, c)))


def test_round_e4m3_matches_brute_force_including_ties():
    g = F.e4m3_values()
    mids = (g[:-1] + g[1:]) / 2                       # exact ties
    rs = np.random.RandomState(3)
    xs = np.concatenate([mids, -mids, g, rs.randn(400) * 50, rs.rand(50) * 2.0 ** -8, [500.0, -1e6, 0.0]])
    got = F.round_e4m3(xs)
    want = np.array([_brute_round_e4m3(x) for x in xs])
    assert np.array_equal(got, want)
    assert F.round_e4m3(np.array([1e9]))[0] == 448.0  # saturating


def test_round_int8_matches_brute_force_including_ties():
    rs = np.random.RandomState(4)
    xs = np.concatenate([np.arange(-130, 131) + 0.5, np.arange(-130, 131), rs.randn(500) * 60, [1e9, -1e9]])
    got = F.round_int8(xs)
    want = np.array([_brute_round_int8(x) for x in xs])
    assert np.array_equal(got, want)
    assert F.round_int8(np.array([126.5, 127.4, 128.0, -127.6]))[0] == 126.0   # tie to even
    assert np.all(np.abs(F.round_int8(xs)) <= 127)


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_row_quantizer_reconstructs_within_half_a_step(fmt):
    rs = np.random.RandomState(5)
    x = rs.randn(7, 3, 128) * np.array([1e-3, 1.0, 50.0])[None, :, None]
    codes, scale = F.quantize_rows(x, fmt)
    qmax = 127.0 if fmt == "int8" else 448.0
    assert np.all(np.abs(codes) <= qmax)
    assert np.allclose(np.abs(codes).max(axis=-1), qmax)        # each row's max maps to the top code
    assert np.allclose(scale, np.abs(x).max(axis=-1) / qmax)
    err = np.abs(codes * scale[..., None] - x)
    if fmt == "int8":
        bound = 0.5 * scale[..., None] * np.ones_like(x)          # integer codes: half a unit
        assert np.all(codes == np.rint(codes))
    else:
        # half an ulp: relative 2^-4 in the normal range, absolute 2^-10 * scale below it
        bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale[..., None])
    assert np.all(err <= bound * (1 + 1e-6))
    zc, zs = F.quantize_rows(np.zeros((2, 128)), fmt)
    assert np.all(zc == 0) and np.all(zs == 1.0)


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_block_quantizer_one_scale_per_128_rows(fmt):
    rs = np.random.RandomState(4)
    x = rs.randn(300, 64)
    x[130] *= 10.0                                     # an outlier row sets block 1's scale
    codes, scale = F.quantize_blocks(x, fmt)
    qmax = 127.0 if fmt == "int8" else 448.0
    assert np.all(scale[:128] == scale[0]) and np.all(scale[128:256] == scale[128]) and np.all(scale[256:] == scale[256])
    assert np.isclose(scale[128], np.abs(x[128:256]).max() / qmax)
    assert np.isclose(np.abs(codes[128:256]).max(), qmax)


def test_channel_quantizer_scales_over_tokens():
    rs = np.random.RandomState(6)
    v = rs.randn(2, 300, 3, 64)
    codes, scale = F.quantize_channels(v)
    assert scale.shape == (2, 3, 64)
    assert np.allclose(np.abs(codes).max(axis=1), 448.0)
    assert np.allclose(scale, np.abs(v).max(axis=1) / 448.0)


@pytest.mark.parametrize("recipe", F.RECIPES)
@pytest.mark.parametrize("mode", [O.SINGLE, O.GROUP])
@pytest.mark.parametrize("peaky", [False, True])
def test_blocked_online_softmax_is_exact_without_quantization(recipe, mode, peaky):
    """With every rounding replaced by the identity the blocked online softmax
    with its integer reference must equal plain softmax attention (scopes of
    three key blocks; the peaky case raises the reference in later blocks)."""
    B, heads, D, T, H, W, k = 1, 2, 64, 3, 10, 20, 2     # L = 300: blocks of 128, 128, 44
    rs = np.random.RandomState(11)
    q = rs.randn(B, T * H * W, heads, D) * (6.0 if peaky else 1.0)
    kk = rs.randn(B, T * H * W, heads, D)
    v = rs.randn(B, T * H * W, heads, D)
    if peaky:
        kk[:, ::7] *= 3.0
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, mode, quantize=False, recipe=recipe)
    rout, rlse = O.skiparse_fwd(q, kk, v, T, H, W, k, mode)
    assert np.max(np.abs(out - rout)) < 1e-12
    assert np.max(np.abs(lse - rlse)) < 1e-10


def _method_by_hand(qs, ks, vs, sv_all, D, recipe):
    """The 8-bit method for one tiny scope, restated with plain loops from the
    definitions (no oracle routine): q rows and k blocks quantized by the
    symmetric rule, exact integer / E4M3 products, an integer base-2 reference
    per block, E4M3(2^8 P) by brute-force nearest-value search, float64
    accumulation. qs, ks, vs: lists of rows (scope order); sv_all: the
    channel max |v| over the whole (batch, head)."""
    Q = 127.0 if recipe == "int8" else 448.0
    rnd = _brute_round_int8 if recipe == "int8" else _brute_round_e4m3

    def quant_row(row, amax):
        if amax == 0:
            return [0.0] * len(row), 1.0
        return [rnd(float(np.float32(x) * np.float32(np.float32(Q) / np.float32(amax)))) for x in row], amax / Q

    qc = [quant_row(r, max(abs(float(np.float32(x))) for x in r)) for r in qs]
    kc = [None] * len(ks)
    for j0 in range(0, len(ks), 128):
        blk = ks[j0:j0 + 128]
        amax = max(abs(float(np.float32(x))) for r in blk for x in r)
        for j in range(j0, min(j0 + 128, len(ks))):
            kc[j] = quant_row(ks[j], amax)
    vc = []
    for r in vs:
        vc.append([_brute_round_e4m3(float(np.float32(x) * np.float32(np.float32(448.0) / np.float32(sv_all[d]))))
                   for d, x in enumerate(r)])
    outs, lses = [], []
    for (qq, sq) in qc:
        t = [sum(a * b for a, b in zip(qq, kk)) * sq * sk / math.sqrt(D) / math.log(2.0) for (kk, sk) in kc]
        M, l, acc = None, 0.0, [0.0] * D
        for j0 in range(0, len(t), 128):
            mb = math.ceil(max(t[j0:j0 + 128]))
            Mn = mb if M is None else max(M, mb)
            if M is not None:
                l *= 2.0 ** (M - Mn)
                acc = [a * 2.0 ** (M - Mn) for a in acc]
            M = Mn
            for j in range(j0, min(j0 + 128, len(t))):
                p = 2.0 ** (t[j] - M)
                l += p
                pq = _brute_round_e4m3(float(np.float32(p * 256.0)))
                acc = [a + pq * vc[j][d] for d, a in enumerate(acc)]
        outs.append([a * (sv_all[d] / 448.0) / (256.0 * l) for d, a in enumerate(acc)])
        lses.append((M + math.log2(l)) * math.log(2.0))
    return np.array(outs), np.array(lses)


@pytest.mark.parametrize("recipe", F.RECIPES)
def test_tiny_scope_by_hand(recipe):
    """The oracle's 8-bit forward on a scope of 160 keys (two blocks, the
    second partial) equals the method written out with loops, for every query
    row of the scope; the second block's keys are scaled up so the reference
    rises. (A reference taken as the floor instead of the ceiling lets 2^8 P
    reach 448 and saturate in about a fifth of the rows.)"""
    B, heads, D, T, H, W, k = 1, 1, 16, 2, 8, 20, 2    # N = 320, single skip: L = 160
    N = T * H * W
    rs = np.random.RandomState(17)
    q, kk, v = (rs.randn(B, N, heads, D) for _ in range(3))
    kk[:, 2 * 128:] *= 2.5                              # scope positions >= 128 (tokens >= 256)
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, O.SINGLE, recipe=recipe)
    s = 1
    tok = O.scope_tokens(N, k, O.SINGLE, s)
    qr = O.apply_rope(q, T, H, W, 10000.0)[0, :, 0]
    kr = O.apply_rope(kk, T, H, W, 10000.0)[0, :, 0]
    vv = v[0, :, 0]
    sv_all = [float(np.abs(vv[:, d].astype(np.float32)).max()) for d in range(D)]
    rows = list(range(len(tok)))
    want_o, want_l = _method_by_hand([list(qr[tok[r]]) for r in rows], [list(kr[t]) for t in tok],
                                     [list(vv[t]) for t in tok], sv_all, D, recipe)
    assert np.max(np.abs(out[0, tok[rows], 0] - want_o)) < 1e-9
    assert np.max(np.abs(lse[0, 0, tok[rows]] - want_l)) < 1e-9


def test_quantized_p_never_saturates():
    """P <= 1 by the integer reference (M >= every score of the blocks seen), so
    2^8 P <= 256 stays below E4M3's largest finite value, and P = 1 is exact."""
    assert 2.0 ** F.P_SHIFT <= F.E4M3_MAX
    assert F.round_e4m3(np.array([2.0 ** F.P_SHIFT]))[0] == 2.0 ** F.P_SHIFT


@pytest.mark.parametrize("recipe", F.RECIPES)
def test_uniform_attention_closed_form(recipe):
    """q = 0: every score is 0, so P = 1 exactly (2^8 P = 256 is an E4M3 value):
    each output row is the mean over its scope of the dequantized v, LSE = ln L."""
    B, heads, D, T, H, W, k = 1, 1, 64, 2, 8, 16, 2
    N = T * H * W
    rs = np.random.RandomState(2)
    q = np.zeros((B, N, heads, D))
    kk = rs.randn(B, N, heads, D)
    v = rs.randn(B, N, heads, D)
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, O.GROUP, recipe=recipe)
    v8, sv = F.quantize_channels(v)
    vd = v8 * sv[:, None]
    L = N // k
    for s in range(k):
        toks = O.scope_tokens(N, k, O.GROUP, s)
        want = vd[0, toks, 0].mean(axis=0)
        assert np.allclose(out[0, toks, 0], want[None, :], atol=1e-12)
        assert np.allclose(lse[0, 0, toks], math.log(L))


def test_error_sizes_of_both_recipes():
    """8-bit operands change the result by about their rounding error. E4M3 has
    a relative step of 2^-3, so q, k, P and v each carry ~3 % RMS rounding
    error, ~5 % at the output; INT8 q and k (steps of max|x| / 127) remove most
    of the S error, which is the page's reason for the mixed recipe: its output
    error must be clearly smaller, its LSE error several times smaller. Bounds:
    both far from exact (quantization is on) and far from garbage."""
    B, heads, D, T, H, W, k = 1, 2, 128, 2, 8, 16, 2
    rs = np.random.RandomState(9)
    q, kk, v = (rs.randn(B, T * H * W, heads, D) for _ in range(3))
    rout, rlse = O.skiparse_fwd(q, kk, v, T, H, W, k, O.SINGLE)
    rel, lerr = {}, {}
    for recipe in F.RECIPES:
        out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, O.SINGLE, recipe=recipe)
        rel[recipe] = np.sqrt(np.sum((out - rout) ** 2) / np.sum(rout ** 2))
        lerr[recipe] = np.max(np.abs(lse - rlse))
        assert 1e-3 < rel[recipe] < 8e-2
        assert lerr[recipe] < 5e-2
    assert rel["int8"] < 0.85 * rel["e4m3"]
    assert lerr["int8"] < 0.5 * lerr["e4m3"]


@pytest.mark.parametrize("recipe", F.RECIPES)
@pytest.mark.parametrize("mode", [O.SINGLE, O.GROUP], ids=["single", "group"])
def test_scope_rows_match_the_whole_forward(mode, recipe):
    """The row-sampled scope routine (used on full-size inputs) gives the whole
    8-bit forward's numbers for the rows it is asked for: several key blocks
    with a ragged last one, two batches and heads (v's channel scales span all
    tokens of a (batch, head))."""
    B, heads, D, T, H, W, k = 2, 2, 64, 3, 10, 12, 2
    N = T * H * W
    rs = np.random.RandomState(21)
    q, kk, v = (rs.randn(B, N, heads, D) for _ in range(3))
    out, lse, l = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, mode, recipe=recipe, with_l=True)
    L = N // k
    rows = np.array([0, 1, 127, 128, 129, L - 1])
    for b, h, s in [(0, 0, 0), (1, 1, 1), (1, 0, 0)]:
        tok, o, ls, ll = F.skiparse_fwd_fp8_scope(q, kk, v, T, H, W, k, mode, b, h, s, rows, recipe=recipe)
        assert np.array_equal(tok, O.scope_tokens(N, k, mode, s)[rows])
        assert np.allclose(o, out[b, tok, h], rtol=0, atol=1e-12)
        assert np.allclose(ls, lse[b, h, tok], rtol=0, atol=1e-12)
        assert np.allclose(ll, l[b, h, tok], rtol=0, atol=1e-12)
        assert np.all(ll > 0.5)


@pytest.mark.parametrize("recipe", F.RECIPES)
@pytest.mark.parametrize("mode", [O.SINGLE, O.GROUP], ids=["single", "group"])
def test_unequal_scopes_exact_without_quantization(mode, recipe):
    """N that k (single) or k^2 (group) does not divide: the prose scopes, of
    unequal length. With every rounding replaced by the identity the 8-bit
    method must equal exact Skiparse attention on those scopes (the main
    oracle, itself pinned to dense attention under the prose masks)."""
    B, heads, D, T, H, W, k = 2, 2, 64, 3, 10, 11, 4     # N = 330: scopes of 83, 83, 82, 82 (single)
    N = T * H * W
    assert not O.divisible(N, k, mode)
    rs = np.random.RandomState(41)
    q, kk, v = (rs.randn(B, N, heads, D) for _ in range(3))
    out, lse = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, mode, quantize=False, recipe=recipe)
    rout, rlse = O.skiparse_fwd(q, kk, v, T, H, W, k, mode)
    assert np.max(np.abs(out - rout)) < 1e-12
    assert np.max(np.abs(lse - rlse)) < 1e-10


@pytest.mark.parametrize("recipe", F.RECIPES)
@pytest.mark.parametrize("mode", [O.SINGLE, O.GROUP], ids=["single", "group"])
def test_scope_gathered_path_equals_the_rearrange(mode, recipe):
    """Where the listings' rearrange applies, gathering each scope by its token
    ids (the path unequal scopes take) gives the rearrange path's numbers."""
    B, heads, D, T, H, W, k = 2, 2, 64, 4, 8, 16, 2       # N = 512, L = 256: two key blocks
    N = T * H * W
    assert O.divisible(N, k, mode)
    rs = np.random.RandomState(43)
    q, kk, v = (rs.randn(B, N, heads, D) for _ in range(3))
    out, lse, l = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, mode, recipe=recipe, with_l=True)
    fmt = "int8" if recipe == "int8" else "e4m3"
    qr = O.apply_rope(q, T, H, W, 10000.0)
    kr = O.apply_rope(kk, T, H, W, 10000.0)
    q8, sq = F.quantize_rows(qr, fmt)
    v8, sv = F.quantize_channels(v)
    gout, glse, gl = F._by_scopes(q8, sq, kr, v8, sv, k, mode, 1.0 / math.sqrt(D), fmt, True)
    assert np.allclose(gout, out, rtol=0, atol=1e-12)
    assert np.allclose(glse, lse, rtol=0, atol=1e-12)
    assert np.allclose(gl, l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("recipe", F.RECIPES)
def test_scope_rows_match_the_whole_forward_unequal_scopes(recipe):
    """The row-sampled scope routine on unequal scopes (group skip, N = 330,
    k = 4: scopes of 84, 84, 82, 80 tokens) gives the whole forward's numbers."""
    B, heads, D, T, H, W, k, mode = 1, 2, 64, 3, 10, 11, 4, O.GROUP
    N = T * H * W
    rs = np.random.RandomState(45)
    q, kk, v = (rs.randn(B, N, heads, D) for _ in range(3))
    out, lse, l = F.skiparse_fwd_fp8(q, kk, v, T, H, W, k, mode, recipe=recipe, with_l=True)
    for s in range(k):
        Ls = len(O.scope_tokens(N, k, mode, s))
        rows = np.array([0, 1, Ls // 2, Ls - 1])
        for h in range(heads):
            tok, o, ls, ll = F.skiparse_fwd_fp8_scope(q, kk, v, T, H, W, k, mode, 0, h, s, rows, recipe=recipe)
            assert np.allclose(o, out[0, tok, h], rtol=0, atol=1e-12)
            assert np.allclose(ls, lse[0, h, tok], rtol=0, atol=1e-12)
            assert np.allclose(ll, l[0, h, tok], rtol=0, atol=1e-12)
