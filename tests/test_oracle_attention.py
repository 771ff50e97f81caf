"""Pins for the oracle's forward and backward (CPU only).

The path is "Open-Sora Plan" docs, section "Skiparse Attention": RoPE, sparse
rearrange, scaled_dot_product_attention per rearranged batch row, reverse
rearrange. Pins:
  * the listings' own library recipe re-run with the libraries they call
    (einops.rearrange with the listed patterns + torch's
    scaled_dot_product_attention, float64 on CPU), and torch autograd through
    it for the gradients;
  * the independent masked-dense routine under the prose masks;
  * k = 1 equals dense attention;
  * an unstabilised brute-force formula on tiny grids (pure Python loops);
  * central finite differences of <dO, out>;
  * invariants: constant V gives O = V; per scope sum_j dV_j = sum_i dO_i and
    the rotated-domain dK rows sum to zero;
  * mutation checks: mistakes planted in the oracle make a pin fail.
"""
import math

import einops
import numpy as np
import pytest
import torch

from oracle import skiparse_oracle as O

THETA = 10000.0
MODES = [O.SINGLE, O.GROUP]


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def small_case(mode, k=2, T=2, H=4, W=4, B=2, nh=2, D=16, seed=0):
    N = T * H * W
    q, kk, v, do = (rnd((B, N, nh, D), seed + i) for i in range(4))
    return dict(q=q, k=kk, v=v, do=do, T=T, H=H, W=W, sparse_k=k, mode=mode)


# ---- library recipe (einops + torch SDPA), the page's listing run with its own libraries

def _library_recipe(q, k, v, T, H, W, sparse_k, mode, rope=None):
    rope = rope or (lambda x: O.rope_closed_form(x, T, H, W, THETA))
    qt = torch.from_numpy(rope(q))
    kt = torch.from_numpy(rope(k))
    vt = torch.from_numpy(np.asarray(v, dtype=np.float64))
    if mode == O.SINGLE:
        fwd = "b (g k) h d -> (k b) h g d"
        bwd = "(k b) h g d -> b (g k) h d"
        kw = dict(k=sparse_k)
    else:
        fwd = "b (n m k) h d -> (m b) h (n k) d"
        bwd = "(m b) h (n k) d -> b (n m k) h d"
        kw = dict(m=sparse_k, k=sparse_k)
    qr, kr, vr = (einops.rearrange(x, fwd, **kw) for x in (qt, kt, vt))
    o = torch.nn.functional.scaled_dot_product_attention(qr, kr, vr)
    lse = torch.logsumexp((qr @ kr.transpose(-1, -2)) / math.sqrt(q.shape[-1]), dim=-1)
    out = einops.rearrange(o, bwd, **kw).numpy()
    lse = einops.rearrange(lse[..., None], bwd, **kw)[..., 0].permute(0, 2, 1).numpy()
    return out, lse


def pin_fwd_library(c, tol=1e-12):
    out, lse = O.skiparse_fwd(c["q"], c["k"], c["v"], c["T"], c["H"], c["W"], c["sparse_k"], c["mode"], THETA)
    ro, rl = _library_recipe(c["q"], c["k"], c["v"], c["T"], c["H"], c["W"], c["sparse_k"], c["mode"])
    return max(np.max(np.abs(out - ro)), np.max(np.abs(lse - rl))) < tol


def _rot_mats(N, T, H, W, D):
    """Per-token rotation matrices R_i (N, D, D) built column by column from the
    complex closed form applied to basis vectors (no reuse of apply_rope)."""
    eye = np.broadcast_to(np.eye(D)[None, None, :, :], (1, N, D, D)).copy()     # (1, N, basis, D)
    cols = O.rope_closed_form(eye, T, H, W, THETA)[0]                            # (N, basis, D)
    return np.transpose(cols, (0, 2, 1))                                         # R[i] @ x


def pin_bwd_autograd(c, tol=1e-10):
    q, k, v, do = c["q"], c["k"], c["v"], c["do"]
    B, N, nh, D = q.shape
    R = torch.from_numpy(_rot_mats(N, c["T"], c["H"], c["W"], D))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    rq = torch.einsum("nij,bnhj->bnhi", R, tq)
    rk = torch.einsum("nij,bnhj->bnhi", R, tk)
    sk, mode = c["sparse_k"], c["mode"]
    if mode == O.SINGLE:
        fwd, bwd, kw = "b (g k) h d -> (k b) h g d", "(k b) h g d -> b (g k) h d", dict(k=sk)
    else:
        fwd, bwd, kw = "b (n m k) h d -> (m b) h (n k) d", "(m b) h (n k) d -> b (n m k) h d", dict(m=sk, k=sk)
    o = torch.nn.functional.scaled_dot_product_attention(*(einops.rearrange(x, fwd, **kw) for x in (rq, rk, tv)))
    out = einops.rearrange(o, bwd, **kw)
    (out * torch.from_numpy(do)).sum().backward()
    dq, dk, dv, _, _ = O.skiparse_bwd(q, k, v, do, c["T"], c["H"], c["W"], sk, mode, THETA)
    err = max(np.max(np.abs(dq - tq.grad.numpy())), np.max(np.abs(dk - tk.grad.numpy())),
              np.max(np.abs(dv - tv.grad.numpy())))
    return err < tol


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("k,T,H,W,B", [(2, 2, 4, 4, 2), (4, 1, 4, 8, 1), (1, 2, 2, 4, 1), (3, 1, 6, 3, 2)])
def test_fwd_equals_library_recipe(mode, k, T, H, W, B):
    c = small_case(mode, k=k, T=T, H=H, W=W, B=B)
    assert pin_fwd_library(c)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("k,T,H,W", [(2, 2, 2, 4), (3, 1, 3, 6), (1, 1, 2, 4)])
def test_bwd_equals_autograd_of_library_recipe(mode, k, T, H, W):
    c = small_case(mode, k=k, T=T, H=H, W=W, B=2)
    assert pin_bwd_autograd(c)


@pytest.mark.parametrize("mode", MODES)
def test_k1_equals_dense_sdpa(mode):
    c = small_case(mode, k=1, B=1)
    out, lse = O.skiparse_fwd(c["q"], c["k"], c["v"], c["T"], c["H"], c["W"], 1, mode, THETA)
    qt = torch.from_numpy(O.rope_closed_form(c["q"], c["T"], c["H"], c["W"], THETA)).permute(0, 2, 1, 3)
    kt = torch.from_numpy(O.rope_closed_form(c["k"], c["T"], c["H"], c["W"], THETA)).permute(0, 2, 1, 3)
    vt = torch.from_numpy(c["v"]).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).permute(0, 2, 1, 3).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("k", [1, 2, 4])
def test_equals_masked_dense(mode, k):
    T, H, W = (1, 4, 8) if k == 4 else (2, 2, 4)
    c = small_case(mode, k=k, T=T, H=H, W=W, B=1, nh=1)
    q, kk, v, do = c["q"], c["k"], c["v"], c["do"]
    N, D = q.shape[1], q.shape[3]
    dq, dk, dv, out, lse = O.skiparse_bwd(q, kk, v, do, T, H, W, k, mode, THETA)
    qt = O.rope_closed_form(q, T, H, W, THETA)[0, :, 0]
    kt = O.rope_closed_form(kk, T, H, W, THETA)[0, :, 0]
    mask = O.skiparse_mask(N, k, mode)
    mo, ml = O.masked_dense_fwd(qt, kt, v[0, :, 0], mask, 1 / math.sqrt(D))
    gq, gk, gv = O.masked_dense_bwd(qt, kt, v[0, :, 0], do[0, :, 0], mask, 1 / math.sqrt(D))
    # back to pre-RoPE gradients with the transpose rotation built from the closed form
    R = _rot_mats(N, T, H, W, D)
    gq = np.einsum("nji,nj->ni", R, gq)
    gk = np.einsum("nji,nj->ni", R, gk)
    assert np.max(np.abs(out[0, :, 0] - mo)) < 1e-12
    assert np.max(np.abs(lse[0, 0] - ml)) < 1e-12
    assert np.max(np.abs(dq[0, :, 0] - gq)) < 1e-12
    assert np.max(np.abs(dk[0, :, 0] - gk)) < 1e-12
    assert np.max(np.abs(dv[0, :, 0] - gv)) < 1e-12


def _brute_force(qt, kt, v, same_scope, scale):
    """Unstabilised direct formula with pure Python loops."""
    N, D = len(qt), len(qt[0])
    out = [[0.0] * D for _ in range(N)]
    lse = [0.0] * N
    for i in range(N):
        den = 0.0
        num = [0.0] * D
        for j in range(N):
            if not same_scope(i, j):
                continue
            s = scale * sum(qt[i][d] * kt[j][d] for d in range(D))
            e = math.exp(s)
            den += e
            for d in range(D):
                num[d] += e * v[j][d]
        out[i] = [x / den for x in num]
        lse[i] = math.log(den)
    return np.array(out), np.array(lse)


@pytest.mark.parametrize("grid,k", [((1, 2, 4), 2), ((2, 2, 2), 2), ((1, 4, 4), 4)])
@pytest.mark.parametrize("mode", MODES)
def test_brute_force_tiny(grid, k, mode):
    T, H, W = grid
    c = small_case(mode, k=k, T=T, H=H, W=W, B=1, nh=1, D=16)
    out, lse = O.skiparse_fwd(c["q"], c["k"], c["v"], T, H, W, k, mode, THETA)
    qt = O.rope_closed_form(c["q"], T, H, W, THETA)[0, :, 0].tolist()
    kt = O.rope_closed_form(c["k"], T, H, W, THETA)[0, :, 0].tolist()
    if mode == O.SINGLE:
        same = lambda i, j: (i - j) % k == 0          # every k-th token
    else:
        same = lambda i, j: (i // k - j // k) % k == 0
    bo, bl = _brute_force(qt, kt, c["v"][0, :, 0].tolist(), same, 1 / 4.0)
    assert np.max(np.abs(out[0, :, 0] - bo)) < 1e-12
    assert np.max(np.abs(lse[0, 0] - bl)) < 1e-12


def pin_finite_differences(c, n_probe=12, h=1e-6, tol=1e-7):
    q, k, v, do = c["q"], c["k"], c["v"], c["do"]
    args = (c["T"], c["H"], c["W"], c["sparse_k"], c["mode"], THETA)
    dq, dk, dv, _, _ = O.skiparse_bwd(q, k, v, do, *args)
    rng = np.random.default_rng(11)
    worst = 0.0
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(n_probe):
            idx = tuple(rng.integers(0, s) for s in x.shape)
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            ins = {"q": q, "k": k, "v": v}
            ins[name] = xp
            lp = np.sum(O.skiparse_fwd(ins["q"], ins["k"], ins["v"], *args)[0] * do)
            ins[name] = xm
            lm = np.sum(O.skiparse_fwd(ins["q"], ins["k"], ins["v"], *args)[0] * do)
            fd = (lp - lm) / (2 * h)
            worst = max(worst, abs(fd - g[idx]) / max(1.0, abs(fd)))
    return worst < tol


@pytest.mark.parametrize("mode", MODES)
def test_backward_finite_differences(mode):
    assert pin_finite_differences(small_case(mode, k=2, T=1, H=2, W=4, B=1, nh=2))


@pytest.mark.parametrize("mode", MODES)
def test_invariants(mode):
    c = small_case(mode, k=2, T=2, H=2, W=8, B=1, nh=1, D=16)
    T, H, W = c["T"], c["H"], c["W"]
    N = T * H * W
    # constant V along tokens -> O = V
    v = np.broadcast_to(rnd((1, 1, 1, 16), 9), c["v"].shape).copy()
    out, _ = O.skiparse_fwd(c["q"], c["k"], v, T, H, W, 2, mode, THETA)
    assert np.max(np.abs(out - v)) < 1e-12
    # per scope: sum_j dV_j = sum_i dO_i, rotated-domain dK rows sum to zero
    qr = O.rearrange(O.apply_rope(c["q"], T, H, W, THETA), 2, mode)
    kr = O.rearrange(O.apply_rope(c["k"], T, H, W, THETA), 2, mode)
    vr = O.rearrange(c["v"], 2, mode)
    dor = O.rearrange(c["do"], 2, mode)
    for r in range(qr.shape[0]):
        o, lse = O.softmax_attention_fwd(qr[r, :, 0], kr[r, :, 0], vr[r, :, 0], 0.25)
        dq, dk, dv = O.softmax_attention_bwd(qr[r, :, 0], kr[r, :, 0], vr[r, :, 0], o, lse, dor[r, :, 0], 0.25)
        assert np.max(np.abs(dv.sum(0) - dor[r, :, 0].sum(0))) < 1e-12
        assert np.max(np.abs(dk.sum(0))) < 1e-12
    assert qr.shape[0] * qr.shape[1] == N


@pytest.mark.parametrize("mode", MODES)
def test_rope_order_matters(mode):
    """RoPE after the rearrange (positions by rearranged index) gives a different
    answer, so applying it at the original positions is actually exercised."""
    c = small_case(mode, k=2, T=2, H=4, W=4, B=1)
    T, H, W = c["T"], c["H"], c["W"]
    good, _ = O.skiparse_fwd(c["q"], c["k"], c["v"], T, H, W, 2, mode, THETA)
    qr = O.rearrange(c["q"], 2, mode)
    kr = O.rearrange(c["k"], 2, mode)
    L = qr.shape[1]
    # wrong order: rotate each scope as if its tokens sat at positions 0..L-1
    qw = O.apply_rope(qr, 1, 1, L, THETA)
    kw = O.apply_rope(kr, 1, 1, L, THETA)
    vr = O.rearrange(c["v"], 2, mode)
    o = np.stack([np.stack([O.softmax_attention_fwd(qw[r, :, h], kw[r, :, h], vr[r, :, h], 0.25)[0]
                            for h in range(qw.shape[2])], axis=1) for r in range(qw.shape[0])])
    bad = O.reverse(o, 2, mode)
    assert np.max(np.abs(good - bad)) > 1e-3


@pytest.mark.parametrize("mode", MODES)
def test_scope_sampler_matches_full_path(mode):
    c = small_case(mode, k=2, T=2, H=4, W=4, B=2, nh=2)
    T, H, W = c["T"], c["H"], c["W"]
    dq, dk, dv, out, lse = O.skiparse_bwd(c["q"], c["k"], c["v"], c["do"], T, H, W, 2, mode, THETA)
    for (b, h, s) in [(0, 0, 0), (1, 1, 1), (1, 0, 1)]:
        r = O.skiparse_scope(c["q"], c["k"], c["v"], c["do"], T, H, W, 2, mode, b, h, s, THETA)
        t = r["tokens"]
        for name, ref in (("out", out[b, t, h]), ("lse", lse[b, h, t]), ("dq", dq[b, t, h]),
                          ("dk", dk[b, t, h]), ("dv", dv[b, t, h])):
            assert np.max(np.abs(r[name] - ref)) < 1e-12, name
        rows = np.array([0, 3, 5])
        f = O.skiparse_scope(c["q"], c["k"], c["v"], None, T, H, W, 2, mode, b, h, s, THETA, rows=rows)
        assert np.max(np.abs(f["out"] - out[b, t[rows], h])) < 1e-12
        assert np.max(np.abs(f["lse"] - lse[b, h, t[rows]])) < 1e-12


# ---- planted mistakes: each must make at least one pin fail ------------------------

def _mutants():
    good_attn = O.softmax_attention_fwd
    good_bwd = O.softmax_attention_bwd
    good_rope = O.apply_rope
    good_single = O.single_skip_rearrange

    def wrong_scale(q, k, v, scale):
        return good_attn(q, k, v, scale * math.sqrt(q.shape[1]) / q.shape[1])

    def no_delta(q, k, v, o, lse, do, scale):
        return good_bwd(q, k, v, np.zeros_like(o), lse, do, scale)

    def dk_unscaled(q, k, v, o, lse, do, scale):
        dq, dk, dv = good_bwd(q, k, v, o, lse, do, scale)
        return dq, dk / scale, dv

    def rope_sign(x, T, H, W, theta, inverse=False):
        return good_rope(x, T, H, W, theta, inverse=not inverse)

    def rope_no_inverse(x, T, H, W, theta, inverse=False):
        return good_rope(x, T, H, W, theta, inverse=False)

    def single_b_outer(x, k):
        B, N = x.shape[:2]
        y = x.reshape((B, N // k, k) + x.shape[2:])
        y = np.moveaxis(y, 2, 1)   # b outer, k inner: '(b k)' instead of '(k b)'
        return y.reshape((k * B, N // k) + x.shape[2:])

    return [("softmax_attention_fwd", wrong_scale), ("softmax_attention_bwd", no_delta),
            ("softmax_attention_bwd", dk_unscaled), ("apply_rope", rope_sign),
            ("apply_rope", rope_no_inverse), ("single_skip_rearrange", single_b_outer)]


@pytest.mark.parametrize("i", range(6))
def test_planted_mistake_is_caught(monkeypatch, i):
    name, bad = _mutants()[i]
    monkeypatch.setattr(O, name, bad)
    caught = []
    for mode in MODES:
        c = small_case(mode, k=2, T=1, H=2, W=4, B=2, nh=1)
        caught.append(not pin_fwd_library(c))
        caught.append(not pin_bwd_autograd(c))
    # the batch order of the rearranged axis is pinned by the listing's pattern via einops
    ids = np.arange(2 * 16 * 3).reshape(2, 16, 3)
    caught.append(not np.array_equal(O.rearrange(ids, 2, O.SINGLE),
                                     einops.rearrange(ids, "b (g k) d -> (k b) g d", k=2)))
    assert any(caught), name


# ---- N the listings' rearrange cannot split: scopes from the prose (ragged lengths)

RAGGED = [((1, 5, 7), 3, O.SINGLE), ((1, 5, 7), 4, O.SINGLE), ((2, 3, 5), 4, O.GROUP),
          ((1, 6, 6), 5, O.GROUP), ((1, 3, 7), 2, O.GROUP), ((1, 2, 3), 4, O.GROUP)]


@pytest.mark.parametrize("grid,k,mode", RAGGED)
def test_ragged_equals_masked_dense(grid, k, mode):
    """For N not divisible by k (single) or k*k (group) the forward and backward
    equal dense attention under the prose mask, the oracle's independent path
    (which never forms scopes), including scopes one token or one partial group
    shorter than others, and empty scopes (N < k*k in the last case)."""
    T, H, W = grid
    c = small_case(mode, k=k, T=T, H=H, W=W, B=2, nh=2)
    q, kk, v, do = c["q"], c["k"], c["v"], c["do"]
    N, D = q.shape[1], q.shape[3]
    assert not O.divisible(N, k, mode)
    dq, dk, dv, out, lse = O.skiparse_bwd(q, kk, v, do, T, H, W, k, mode, THETA)
    out2, lse2 = O.skiparse_fwd(q, kk, v, T, H, W, k, mode, THETA)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    mask = O.skiparse_mask(N, k, mode)
    R = _rot_mats(N, T, H, W, D)
    for b in range(2):
        for h in range(2):
            qt = O.rope_closed_form(q, T, H, W, THETA)[b, :, h]
            kt = O.rope_closed_form(kk, T, H, W, THETA)[b, :, h]
            mo, ml = O.masked_dense_fwd(qt, kt, v[b, :, h], mask, 1 / math.sqrt(D))
            gq, gk, gv = O.masked_dense_bwd(qt, kt, v[b, :, h], do[b, :, h], mask, 1 / math.sqrt(D))
            gq = np.einsum("nji,nj->ni", R, gq)
            gk = np.einsum("nji,nj->ni", R, gk)
            assert np.max(np.abs(out[b, :, h] - mo)) < 1e-12
            assert np.max(np.abs(lse[b, h] - ml)) < 1e-12
            assert np.max(np.abs(dq[b, :, h] - gq)) < 1e-12
            assert np.max(np.abs(dk[b, :, h] - gk)) < 1e-12
            assert np.max(np.abs(dv[b, :, h] - gv)) < 1e-12


@pytest.mark.parametrize("grid,k,mode", RAGGED[:3])
def test_ragged_brute_force(grid, k, mode):
    """Ragged scopes against the unstabilised pure-Python formula, with scope
    membership written out from the prose (every k-th token, or every k-th
    group of k adjacent tokens)."""
    T, H, W = grid
    c = small_case(mode, k=k, T=T, H=H, W=W, B=1, nh=1)
    q, kk, v = c["q"], c["k"], c["v"]
    N, D = q.shape[1], q.shape[3]
    out, lse = O.skiparse_fwd(q, kk, v, T, H, W, k, mode, THETA)
    qt = O.rope_closed_form(q, T, H, W, THETA)[0, :, 0].tolist()
    kt = O.rope_closed_form(kk, T, H, W, THETA)[0, :, 0].tolist()
    if mode == O.SINGLE:
        same = lambda i, j: (i - j) % k == 0
    else:
        same = lambda i, j: (i // k - j // k) % k == 0
    bo, bl = _brute_force(qt, kt, v[0, :, 0].tolist(), same, 1 / math.sqrt(D))
    assert np.max(np.abs(out[0, :, 0] - bo)) < 1e-10
    assert np.max(np.abs(lse[0, 0] - bl)) < 1e-10


@pytest.mark.parametrize("mode", MODES)
def test_ragged_scope_sampler_matches_full_path(mode):
    T, H, W, k = 2, 5, 7, 3
    c = small_case(mode, k=k, T=T, H=H, W=W, B=1, nh=2)
    dq, dk, dv, out, lse = O.skiparse_bwd(c["q"], c["k"], c["v"], c["do"], T, H, W, k, mode, THETA)
    for s in range(k):
        r = O.skiparse_scope(c["q"], c["k"], c["v"], c["do"], T, H, W, k, mode, 0, 1, s, THETA)
        tok = r["tokens"]
        assert np.max(np.abs(r["out"] - out[0, tok, 1])) < 1e-12
        assert np.max(np.abs(r["dq"] - dq[0, tok, 1])) < 1e-12
        assert np.max(np.abs(r["dk"] - dk[0, tok, 1])) < 1e-12
        assert np.max(np.abs(r["dv"] - dv[0, tok, 1])) < 1e-12
