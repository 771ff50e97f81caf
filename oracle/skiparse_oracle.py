"""Plain CPU float64 oracle for Skiparse attention.

TEST INFRASTRUCTURE ONLY. Only the tests, `__graft_entry__.smoke()` and the
CPU-baseline / reference legs of `bench.py` may import or call this module.
The library under `sparse_spatiotemporal_attention_gb300/` never touches it, and
this module imports nothing from there (the seeded input generator lives in a
module of its own and is passed in as arrays).

What it computes follows "Open-Sora Plan" (docs page), section "Skiparse
Attention", its "Single Skip Implementation" and "Group Skip Implementation"
listings, step by step in the order given there:

  1. q, k are rotated by 3D RoPE at each token's ORIGINAL position (the
     section's implementation note: RoPE comes before the rearrange, because the
     rearrange loses the spatial positions);
  2. q, k, v are rearranged into sparse scopes (single: 'b (g k) d -> (k b) g d';
     group: 'b (n m k) d -> (m b) (n k) d' with m = k = sparse_k), written here
     as an explicit reshape/transpose of the token axis;
  3. plain softmax attention (non-causal, unmasked, no dropout, scale 1/sqrt(D))
     runs on every rearranged batch row and head, i.e. inside every scope;
  4. the result is rearranged back by the inverse pattern.

Everything is float64 from the bf16-valued inputs; no rounding is modelled.
The backward pass is the exact analytic gradient of that float64 forward pass.

Readings taken where the page is silent:
  * tokens are flattened t-major, then h, then w: i = (t*H + h)*W + w;
  * multi-head: the rearrange acts on the token axis only, identically per head,
    and the softmax scale is 1/sqrt(D) with D the head dimension;
  * 3D RoPE: the head's D channels are split in order into a t-chunk of D/4,
    an h-chunk of 3D/8 and a w-chunk of 3D/8 channels; inside a chunk of size d,
    channel pair (2j, 2j+1) is rotated by angle pos * theta**(-2j/d), with pos
    the 0-based integer coordinate on that axis;
  * LSE is the natural-log log-sum-exp of the scaled scores of each query row,
    stored in original token order as (B, heads, N);
  * N not divisible by k (single) or k*k (group), where the listings' rearrange
    has no shape: the section's prose still defines the scopes for any N
    (single: every k-th token, i.e. i mod k = s; group: every k-th group of k
    adjacent tokens, i.e. (i div k) mod k = s, the
    last group holding the N mod k leftover tokens). Scope s then holds exactly
    those tokens in ascending order, and scopes differ in length by at most one
    token (single) or one group (group); nothing is padded. When N is
    divisible this is the listings' rearrange exactly (a pinned property).

Parity: every function here is pinned by tests in tests/test_oracle_*.py
against library routines (einops.rearrange with the page's patterns, torch's
scaled_dot_product_attention and autograd in float64), closed forms,
invariants, brute force on tiny grids and a hand-written golden fixture.
"""
from __future__ import annotations

import math

import numpy as np

SINGLE = 0
GROUP = 1


# ---------------------------------------------------------------------------
# Token grid (reading: t-major flatten; the page's listings only say x is (B, N, C))
# ---------------------------------------------------------------------------

def token_coords(N: int, T: int, H: int, W: int):
    """(t, h, w) of every token i in [0, N), for i = (t*H + h)*W + w."""
    assert N == T * H * W
    i = np.arange(N, dtype=np.int64)
    t = i // (H * W)
    h = (i // W) % H
    w = i % W
    return t, h, w


# ---------------------------------------------------------------------------
# Sparse rearrange (Skiparse Attention: Single Skip / Group Skip Implementation)
# Arrays carry the token axis at position 1: (B, N, ...) with any trailing axes.
# ---------------------------------------------------------------------------

def single_skip_rearrange(x: np.ndarray, sparse_k: int) -> np.ndarray:
    """'b (g k) d -> (k b) g d': split N as (g, k) with k innermost, then put k
    outermost in the new batch axis, ahead of b."""
    B, N = x.shape[:2]
    rest = x.shape[2:]
    assert N % sparse_k == 0
    g = N // sparse_k
    y = x.reshape((B, g, sparse_k) + rest)          # b, g, k, ...
    y = np.moveaxis(y, 2, 0)                        # k, b, g, ...
    return y.reshape((sparse_k * B, g) + rest)      # (k b), g, ...


def single_skip_reverse(y: np.ndarray, sparse_k: int) -> np.ndarray:
    """'(k b) g d -> b (g k) d', the inverse of single_skip_rearrange."""
    KB, g = y.shape[:2]
    rest = y.shape[2:]
    B = KB // sparse_k
    x = y.reshape((sparse_k, B, g) + rest)          # k, b, g, ...
    x = np.moveaxis(x, 0, 2)                        # b, g, k, ...
    return x.reshape((B, g * sparse_k) + rest)


def group_skip_rearrange(x: np.ndarray, sparse_k: int) -> np.ndarray:
    """'b (n m k) d -> (m b) (n k) d' with m = k = sparse_k: split N as (n, m, k),
    move m outermost into the new batch axis, and keep (n, k) as the position."""
    B, N = x.shape[:2]
    rest = x.shape[2:]
    m = kk = sparse_k
    assert N % (m * kk) == 0
    n = N // (m * kk)
    y = x.reshape((B, n, m, kk) + rest)             # b, n, m, k, ...
    y = np.moveaxis(y, 2, 0)                        # m, b, n, k, ...
    return y.reshape((m * B, n * kk) + rest)        # (m b), (n k), ...


def group_skip_reverse(y: np.ndarray, sparse_k: int) -> np.ndarray:
    """'(m b) (n k) d -> b (n m k) d', the inverse of group_skip_rearrange."""
    MB, nk = y.shape[:2]
    rest = y.shape[2:]
    m = kk = sparse_k
    B = MB // m
    n = nk // kk
    x = y.reshape((m, B, n, kk) + rest)             # m, b, n, k, ...
    x = np.moveaxis(x, 0, 2)                        # b, n, m, k, ...
    return x.reshape((B, n * m * kk) + rest)


def rearrange(x, sparse_k, mode):
    return single_skip_rearrange(x, sparse_k) if mode == SINGLE else group_skip_rearrange(x, sparse_k)


def divisible(N: int, sparse_k: int, mode: int) -> bool:
    """True when the listings' rearrange applies: k | N (single), k*k | N (group)."""
    return N % (sparse_k if mode == SINGLE else sparse_k * sparse_k) == 0


def prose_scope_tokens(N: int, sparse_k: int, mode: int, s: int) -> np.ndarray:
    """Scope s for any N from the section's prose: the tokens i with
    i mod k = s (single skip) or (i div k) mod k = s (group skip), ascending."""
    i = np.arange(N, dtype=np.int64)
    a = i % sparse_k if mode == SINGLE else (i // sparse_k) % sparse_k
    return i[a == s]


def reverse(y, sparse_k, mode):
    return single_skip_reverse(y, sparse_k) if mode == SINGLE else group_skip_reverse(y, sparse_k)


def index_maps(N: int, sparse_k: int, mode: int):
    """scope_of_token[i], pos_of_token[i] as read off the rearrange itself:
    rearranging the token ids 0..N-1 (B = 1) gives, at [s, p], the token that
    lands at position p of scope s (rearranged batch row s*B + b). For N the
    rearrange cannot split, from the prose scopes (prose_scope_tokens)."""
    if not divisible(N, sparse_k, mode):
        scope = np.empty(N, dtype=np.int64)
        pos = np.empty(N, dtype=np.int64)
        for s in range(sparse_k):
            tok = prose_scope_tokens(N, sparse_k, mode, s)
            scope[tok] = s
            pos[tok] = np.arange(len(tok))
        return scope, pos
    ids = np.arange(N, dtype=np.int64)[None, :]
    r = rearrange(ids, sparse_k, mode)              # (k, N/k)
    scope = np.empty(N, dtype=np.int64)
    pos = np.empty(N, dtype=np.int64)
    kk, L = r.shape
    for s in range(kk):
        scope[r[s]] = s
        pos[r[s]] = np.arange(L)
    return scope, pos


def scope_tokens(N: int, sparse_k: int, mode: int, s: int) -> np.ndarray:
    """Token ids of scope s in in-scope order (row s of the rearranged ids; for N
    the rearrange cannot split, the prose scope)."""
    if not divisible(N, sparse_k, mode):
        return prose_scope_tokens(N, sparse_k, mode, s)
    ids = np.arange(N, dtype=np.int64)[None, :]
    return rearrange(ids, sparse_k, mode)[s]


# ---------------------------------------------------------------------------
# 3D RoPE at original positions (reading stated in the module docstring)
# ---------------------------------------------------------------------------

def rope_chunks(D: int):
    """Channel chunks (start, size) for the t, h and w axes: D/4, 3D/8, 3D/8."""
    assert D % 16 == 0
    dt = D // 4
    dh = 3 * D // 8
    dw = D - dt - dh
    return [(0, dt), (dt, dh), (dt + dh, dw)]


def apply_rope(x: np.ndarray, T: int, H: int, W: int, theta: float, inverse: bool = False) -> np.ndarray:
    """Rotate x (B, N, heads, D) float64 by each token's (t, h, w); inverse=True
    applies the transpose rotation (used for the gradient, R^T g). theta = 0
    means no rotation: q and k arrive already rotated (the listings rotate the
    projections' outputs, so a projection with a RoPE epilogue has done it)."""
    if theta == 0:
        return np.array(x, dtype=np.float64, copy=True)
    B, N, nh, D = x.shape
    coords = token_coords(N, T, H, W)
    out = np.array(x, dtype=np.float64, copy=True)
    sign = -1.0 if inverse else 1.0
    for (c0, d), pos in zip(rope_chunks(D), coords):
        for j in range(d // 2):
            omega = theta ** (-2.0 * j / d)
            ang = sign * pos.astype(np.float64) * omega            # (N,)
            c = np.cos(ang)[None, :, None]
            s = np.sin(ang)[None, :, None]
            a = x[..., c0 + 2 * j]
            b = x[..., c0 + 2 * j + 1]
            out[..., c0 + 2 * j] = a * c - b * s
            out[..., c0 + 2 * j + 1] = a * s + b * c
    return out


def rope_closed_form(x: np.ndarray, T: int, H: int, W: int, theta: float) -> np.ndarray:
    """Same rotation written independently as complex multiplication: each
    channel pair is z = x0 + i x1, multiplied by exp(i * pos * omega)."""
    B, N, nh, D = x.shape
    t, h, w = token_coords(N, T, H, W)
    out = np.empty_like(x, dtype=np.float64)
    for (c0, d), pos in zip(rope_chunks(D), (t, h, w)):
        half = d // 2
        freqs = np.power(float(theta), -np.arange(0, d, 2, dtype=np.float64) / d)   # (half,)
        phase = np.exp(1j * np.outer(pos.astype(np.float64), freqs))               # (N, half)
        z = x[..., c0:c0 + d:2] + 1j * x[..., c0 + 1:c0 + d:2]                      # (B, N, nh, half)
        zr = z * phase[None, :, None, :]
        out[..., c0:c0 + d:2] = zr.real
        out[..., c0 + 1:c0 + d:2] = zr.imag
        assert zr.shape[-1] == half
    return out


# ---------------------------------------------------------------------------
# Attention inside one rearranged batch row (the page's scaled_dot_product_attention call)
# ---------------------------------------------------------------------------

def softmax_attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """One (L, D) problem: S = scale q k^T, P = row softmax (max-subtracted),
    O = P v, lse = log sum exp of the scaled scores of each row."""
    S = scale * (q @ k.T)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    P = E / l
    O = P @ v
    lse = (m + np.log(l))[:, 0]
    return O, lse


def softmax_attention_bwd(q, k, v, o, lse, do, scale):
    """Exact gradient of softmax_attention_fwd for loss <dO, O>:
    P = exp(S - lse), dV = P^T dO, dP = dO V^T, delta = rowsum(dO * O),
    dS = P * (dP - delta), dq = scale dS k, dk = scale dS^T q."""
    S = scale * (q @ k.T)
    P = np.exp(S - lse[:, None])
    dv = P.T @ do
    dP = do @ v.T
    delta = (do * o).sum(axis=1)
    dS = P * (dP - delta[:, None])
    dq = scale * (dS @ k)
    dk = scale * (dS.T @ q)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# The whole path: RoPE -> rearrange -> attention per scope -> reverse rearrange
# ---------------------------------------------------------------------------

def _by_scopes(q, k, v, do, T, H, W, sparse_k, mode, theta):
    """The same steps for N the listings' rearrange cannot split: RoPE at the
    original positions, then each prose scope gathered, attended and scattered
    back. Returns (out, lse (B, N, heads), and dq, dk, dv when do is given)."""
    B, N, nh, D = q.shape
    scale = 1.0 / math.sqrt(D)
    qr = apply_rope(q, T, H, W, theta)
    kr = apply_rope(k, T, H, W, theta)
    vv = np.asarray(v, dtype=np.float64)
    out = np.empty_like(qr)
    lse = np.empty((B, N, nh))
    grads = None if do is None else [np.empty_like(qr) for _ in range(3)]
    for s in range(sparse_k):
        tok = prose_scope_tokens(N, sparse_k, mode, s)
        if len(tok) == 0:
            continue
        for b in range(B):
            for h in range(nh):
                o, l = softmax_attention_fwd(qr[b, tok, h], kr[b, tok, h], vv[b, tok, h], scale)
                out[b, tok, h], lse[b, tok, h] = o, l
                if do is not None:
                    g = softmax_attention_bwd(qr[b, tok, h], kr[b, tok, h], vv[b, tok, h], o, l,
                                              np.asarray(do[b, tok, h], dtype=np.float64), scale)
                    for a, gg in zip(grads, g):
                        a[b, tok, h] = gg
    if do is None:
        return out, lse
    dq = apply_rope(grads[0], T, H, W, theta, inverse=True)
    dk = apply_rope(grads[1], T, H, W, theta, inverse=True)
    return out, lse, dq, dk, grads[2]


def skiparse_fwd(q, k, v, T, H, W, sparse_k, mode, theta=10000.0):
    """q, k, v: (B, N, heads, D) float64 (bf16-valued). Returns out (B, N, heads, D)
    and lse (B, heads, N), both float64."""
    B, N, nh, D = q.shape
    if not divisible(N, sparse_k, mode):
        out, lse = _by_scopes(q, k, v, None, T, H, W, sparse_k, mode, theta)
        return out, np.ascontiguousarray(np.transpose(lse, (0, 2, 1)))
    scale = 1.0 / math.sqrt(D)
    qr = rearrange(apply_rope(q, T, H, W, theta), sparse_k, mode)
    kr = rearrange(apply_rope(k, T, H, W, theta), sparse_k, mode)
    vr = rearrange(np.asarray(v, dtype=np.float64), sparse_k, mode)
    o_r = np.empty_like(qr)
    lse_r = np.empty(qr.shape[:3], dtype=np.float64)               # (kB, L, heads)
    for r in range(qr.shape[0]):
        for h in range(nh):
            o, lse = softmax_attention_fwd(qr[r, :, h], kr[r, :, h], vr[r, :, h], scale)
            o_r[r, :, h] = o
            lse_r[r, :, h] = lse
    out = reverse(o_r, sparse_k, mode)
    lse = reverse(lse_r, sparse_k, mode)                            # (B, N, heads)
    return out, np.ascontiguousarray(np.transpose(lse, (0, 2, 1)))


def skiparse_bwd(q, k, v, do, T, H, W, sparse_k, mode, theta=10000.0):
    """Gradients of <dO, out> w.r.t. the pre-RoPE q, k and v. Returns
    (dq, dk, dv, out, lse) in the layouts of skiparse_fwd."""
    B, N, nh, D = q.shape
    if not divisible(N, sparse_k, mode):
        out, lse, dq, dk, dv = _by_scopes(q, k, v, do, T, H, W, sparse_k, mode, theta)
        return dq, dk, dv, out, np.ascontiguousarray(np.transpose(lse, (0, 2, 1)))
    scale = 1.0 / math.sqrt(D)
    qr = rearrange(apply_rope(q, T, H, W, theta), sparse_k, mode)
    kr = rearrange(apply_rope(k, T, H, W, theta), sparse_k, mode)
    vr = rearrange(np.asarray(v, dtype=np.float64), sparse_k, mode)
    dor = rearrange(np.asarray(do, dtype=np.float64), sparse_k, mode)
    o_r = np.empty_like(qr)
    lse_r = np.empty(qr.shape[:3], dtype=np.float64)
    dq_r = np.empty_like(qr)
    dk_r = np.empty_like(qr)
    dv_r = np.empty_like(qr)
    for r in range(qr.shape[0]):
        for h in range(nh):
            o, lse = softmax_attention_fwd(qr[r, :, h], kr[r, :, h], vr[r, :, h], scale)
            dq, dk, dv = softmax_attention_bwd(qr[r, :, h], kr[r, :, h], vr[r, :, h], o, lse,
                                               dor[r, :, h], scale)
            o_r[r, :, h], lse_r[r, :, h] = o, lse
            dq_r[r, :, h], dk_r[r, :, h], dv_r[r, :, h] = dq, dk, dv
    # RoPE came first, so its backward comes last: d(pre-RoPE) = R^T d(post-RoPE).
    dq = apply_rope(reverse(dq_r, sparse_k, mode), T, H, W, theta, inverse=True)
    dk = apply_rope(reverse(dk_r, sparse_k, mode), T, H, W, theta, inverse=True)
    dv = reverse(dv_r, sparse_k, mode)
    out = reverse(o_r, sparse_k, mode)
    lse = np.ascontiguousarray(np.transpose(reverse(lse_r, sparse_k, mode), (0, 2, 1)))
    return dq, dk, dv, out, lse


def skiparse_scope(q, k, v, do, T, H, W, sparse_k, mode, b, head, s, theta=10000.0,
                   rows=None):
    """One scope of one (batch, head), for checks on large inputs.

    q, k, v, do are the full (B, N, heads, D) arrays (any float dtype holding
    bf16 values); only the scope's tokens are read. Returns a dict with
    'tokens' (token ids in scope order) and out, lse (and dq, dk, dv when do is
    given) for those tokens, float64. With `rows` (indices into the scope) and
    do=None, only those query rows' out/lse are formed.
    """
    N = q.shape[1]
    D = q.shape[3]
    scale = 1.0 / math.sqrt(D)
    tok = scope_tokens(N, sparse_k, mode, s)
    # RoPE at the ORIGINAL positions, then gather the scope (step 1 before step 2).
    qh = np.asarray(q[b, :, head], dtype=np.float64)
    kh = np.asarray(k[b, :, head], dtype=np.float64)
    t, h, w = token_coords(N, T, H, W)
    qt = _rope_rows(qh[tok], t[tok], h[tok], w[tok], theta)
    kt = _rope_rows(kh[tok], t[tok], h[tok], w[tok], theta)
    vt = np.asarray(v[b, :, head], dtype=np.float64)[tok]
    res = {"tokens": tok}
    if do is None:
        sel = np.arange(len(tok)) if rows is None else np.asarray(rows)
        S = scale * (qt[sel] @ kt.T)
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        l = E.sum(axis=1, keepdims=True)
        res["rows"] = sel
        res["out"] = (E / l) @ vt
        res["lse"] = (m + np.log(l))[:, 0]
        return res
    dot = np.asarray(do[b, :, head], dtype=np.float64)[tok]
    o, lse = softmax_attention_fwd(qt, kt, vt, scale)
    dq, dk, dv = softmax_attention_bwd(qt, kt, vt, o, lse, dot, scale)
    res["out"], res["lse"] = o, lse
    res["dq"] = _rope_rows(dq, t[tok], h[tok], w[tok], theta, inverse=True)
    res["dk"] = _rope_rows(dk, t[tok], h[tok], w[tok], theta, inverse=True)
    res["dv"] = dv
    return res


def _rope_rows(x, t, h, w, theta, inverse=False):
    """apply_rope for a list of rows x (n, D) whose coordinates are given."""
    if theta == 0:
        return np.array(x, dtype=np.float64, copy=True)
    D = x.shape[1]
    out = np.array(x, dtype=np.float64, copy=True)
    sign = -1.0 if inverse else 1.0
    for (c0, d), pos in zip(rope_chunks(D), (t, h, w)):
        for j in range(d // 2):
            ang = sign * pos.astype(np.float64) * theta ** (-2.0 * j / d)
            c, s_ = np.cos(ang), np.sin(ang)
            a = x[:, c0 + 2 * j]
            bb = x[:, c0 + 2 * j + 1]
            out[:, c0 + 2 * j] = a * c - bb * s_
            out[:, c0 + 2 * j + 1] = a * s_ + bb * c
    return out


# ---------------------------------------------------------------------------
# Independent second path: dense attention under the boolean scope mask.
# Shares no code with the rearrange path above.
# ---------------------------------------------------------------------------

def skiparse_mask(N: int, sparse_k: int, mode: int) -> np.ndarray:
    """M[i, j] = True when tokens i and j share a scope, from the section's prose:
    single skip pairs tokens whose distance is a multiple of k (i = j mod k);
    group skip pairs groups of k adjacent tokens whose group indices differ by a
    multiple of k
    ((i div k) = (j div k) mod k)."""
    i = np.arange(N)
    if mode == SINGLE:
        a = i % sparse_k
    else:
        a = (i // sparse_k) % sparse_k
    return a[:, None] == a[None, :]


def masked_dense_fwd(qt, kt, v, mask, scale):
    """Dense attention over all N tokens with disallowed pairs removed.
    qt, kt are already rotated; (N, D) each. Returns out (N, D), lse (N,)."""
    S = scale * (qt @ kt.T)
    S = np.where(mask, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.where(mask, np.exp(S - m), 0.0)
    l = E.sum(axis=1, keepdims=True)
    return (E / l) @ v, (m + np.log(l))[:, 0]


def masked_dense_bwd(qt, kt, v, do, mask, scale):
    """Gradient of <do, masked_dense_fwd> w.r.t. qt, kt, v."""
    out, lse = masked_dense_fwd(qt, kt, v, mask, scale)
    S = scale * (qt @ kt.T)
    P = np.where(mask, np.exp(np.where(mask, S, 0.0) - lse[:, None]), 0.0)
    dv = P.T @ do
    dP = do @ v.T
    delta = np.einsum("id,id->i", do, out)
    dS = P * (dP - delta[:, None])
    return scale * dS @ kt, scale * dS.T @ qt, dv


def skiparse_fwd_flops(B, heads, N, D, sparse_k):
    """Algorithmic forward FLOPs: two L x L x D products per scope, k scopes."""
    return 4.0 * B * heads * N * N * D / sparse_k
