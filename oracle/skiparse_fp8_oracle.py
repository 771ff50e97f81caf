"""Plain CPU float64 oracle for the 8-bit Skiparse attention forward pass.

TEST INFRASTRUCTURE ONLY: imported by tests and bench.py's CPU legs, never by
the library. It builds on skiparse_oracle.py (RoPE, rearrange) and shares no
code with the GPU path.

The method is the Wan 2.1 report's ("Open and Advanced Large-Scale Video
Generative Models") section 4.4.3 "Quantization", paragraph "8-Bit
FlashAttention", applied inside each Skiparse scope:

  * "Mixed 8-Bit optimization": S = Q K^T is computed from INT8 q and k, and
    O = P V from FP8 (E4M3) P and v (recipe "int8"). The page contrasts it with
    FlashAttention-3's native FP8, which feeds E4M3 q, k and v to both
    products and which the page reports to degrade quality (recipe "e4m3",
    kept as the comparison);
  * "FP32 accumulation for cross-block reduction": P V is formed block by
    block of keys with 8-bit operands, and the blocks' products are summed in
    a wider accumulator (fp32 on the page; float64 here).

Readings taken where the page leaves a step open (it describes a Hopper
kernel and gives no formulas):

  * q and k are quantized after RoPE (RoPE precedes the rearrange): q per
    (token, head) row, k per block of 128 consecutive keys of a scope (one
    scale per key block, the granularity of SageAttention, which the page
    cites); v per (batch, head, channel) over all N tokens, so its scale
    factors out of O = P V column by column;
  * symmetric scaling: code = round(x * Q / max|x|), scale = max|x| / Q, with
    Q = 127 for INT8 (round to nearest, ties to even, clamped to +-127) and
    Q = 448 for E4M3 (nearest finite value, ties to the even code,
    saturating); all-zero data gives scale 1 and codes 0;
  * INT8 products are exact integers: S_int = sum_d qc_d kc_d, and
    S = S_int * s_q * s_k;
  * online softmax over blocks of 128 keys in scope order, in base 2:
    t = S * log2(e) / sqrt(D). The running row reference is an integer,
    M_b = max(M_(b-1), ceil(max_j t_j over block b)), so P = 2^(t - M_b) <= 1
    and every change of reference multiplies by an exact power of two;
  * P enters P V as E4M3(2^8 P) (at most 256 < 448, never saturating, and
    small P keep E4M3's normal precision down to 2^-14): block b adds
    E4M3(2^8 P_b) @ vc_b to O after O is multiplied by 2^(M_(b-1) - M_b);
    the row sum l adds the unquantized P the same way;
  * out = O * s_v / (2^8 l), lse = (M + log2 l) * ln 2.

Where floating point decides a code (the quantized q, k, v and P), the value
rounded is a float32 number, the precision of the kernel: q and k after RoPE
and v are float32, the scaled value x * (Q / max|x|) is formed in float32 from
them, and 2^8 P is the float32 nearest to its exact value. Everything else
(RoPE, the products, the sums, the rescaling, the output) is float64.
Parity pins: tests/test_oracle_fp8.py.
"""
from __future__ import annotations

import math

import numpy as np

from . import skiparse_oracle as O

E4M3_MAX = 448.0
INT8_MAX = 127.0
P_SHIFT = 8           # P is quantized as E4M3(2^8 P) with P <= 1
BLOCK = 128
RECIPES = ("int8", "e4m3")


def e4m3_values() -> np.ndarray:
    """All finite non-negative E4M3 (fn) values, ascending, from the format's
    definition: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent field 0
    is subnormal (m/8 * 2^-6); the all-ones code (S.1111.111) is NaN, so the
    largest finite value is 1.75 * 2^8 = 448."""
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue                      # NaN
            if e == 0:
                vals.append(m / 8.0 * 2.0 ** -6)
            else:
                vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_GRID = e4m3_values()


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest finite E4M3 value, ties to the even code,
    saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    idx = np.searchsorted(_GRID, a)                      # first grid value >= a
    idx = np.clip(idx, 1, len(_GRID) - 1)
    lo, hi = _GRID[idx - 1], _GRID[idx]
    take_hi = (hi - a) < (a - lo)
    tie = (hi - a) == (a - lo)
    # codes are consecutive integers along the grid: the even code is the even index
    take_hi = take_hi | (tie & ((idx % 2) == 0))
    r = np.where(take_hi, hi, lo)
    r = np.where(a <= _GRID[0], 0.0, r)
    return np.copysign(r, x)


def round_int8(x: np.ndarray) -> np.ndarray:
    """Round to the nearest integer, ties to even, clamped to [-127, 127]."""
    return np.clip(np.rint(np.asarray(x, dtype=np.float64)), -INT8_MAX, INT8_MAX)


def _fmt(recipe_operand: str):
    """(largest code magnitude Q, rounding function) of an operand format."""
    return (INT8_MAX, round_int8) if recipe_operand == "int8" else (E4M3_MAX, round_e4m3)


def _codes(x, amax, fmt):
    """Codes of x * (Q / amax), the scaled value formed in float32."""
    qmax, rnd = _fmt(fmt)
    x32 = np.asarray(x, dtype=np.float32)
    a32 = np.asarray(amax, dtype=np.float32)
    inv = np.where(a32 > 0, np.float32(qmax) / np.where(a32 > 0, a32, np.float32(1)), np.float32(0)).astype(np.float32)
    return rnd((x32 * inv).astype(np.float64))


def quantize_rows(x: np.ndarray, fmt: str = "e4m3"):
    """Per-row codes and scales over the last axis: x ~ codes * scale."""
    qmax, _ = _fmt(fmt)
    x32 = np.asarray(x, dtype=np.float32).astype(np.float64)
    amax = np.abs(x32).max(axis=-1, keepdims=True)
    codes = _codes(x32, amax, fmt)
    scale = np.where(amax > 0, amax / qmax, 1.0)
    return codes, scale[..., 0]


def quantize_blocks(x: np.ndarray, fmt: str = "e4m3", block: int = BLOCK):
    """x (L, D) in scope order: per block of `block` rows, codes and one scale
    (returned per row, constant within a block)."""
    codes = np.empty_like(np.asarray(x, dtype=np.float64))
    scale = np.empty(x.shape[0])
    for j0 in range(0, x.shape[0], block):
        c, s_ = quantize_rows(x[j0:j0 + block].reshape(1, -1), fmt)
        codes[j0:j0 + block] = c.reshape(-1, x.shape[1])
        scale[j0:j0 + block] = s_[0]
    return codes, scale


def quantize_channels(v: np.ndarray):
    """v (B, N, heads, D): per (b, head, channel) E4M3 codes and scales over N."""
    v32 = np.asarray(v, dtype=np.float32).astype(np.float64)
    amax = np.abs(v32).max(axis=1, keepdims=True)                 # (B, 1, heads, D)
    codes = _codes(v32, amax, "e4m3")
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    return codes, scale[:, 0]                                       # (B, heads, D)


def blocked_attention(sq, sk, qc, kc, vc, sv, scale, quantize_p=True):
    """One scope problem: qc (Lq, D) codes with row scales sq (Lq,), kc (L, D)
    with per-row (block-constant) scales sk (L,), vc (L, D) with channel scales
    sv (D,). Returns (out (Lq, D), lse (Lq,), l (Lq,)), l the row sum of P
    relative to the final reference 2^M (1/2 < max_j P_j <= 1, so l > 1/2).
    Query rows are independent, so qc may hold any subset of the scope's rows.
    quantize_p=False uses P itself in P V (with exact operands, exact softmax
    attention)."""
    Lq, D = qc.shape
    L = kc.shape[0]
    log2e = 1.0 / math.log(2.0)
    # exact: integer dot products, or sums of products of E4M3 values
    t = (qc @ kc.T) * (sq[:, None] * sk[None, :]) * (scale * log2e)   # (Lq, L), base-2 units
    M = np.zeros(Lq)
    l = np.zeros(Lq)
    acc = np.zeros((Lq, D))
    for j0 in range(0, L, BLOCK):
        tb = t[:, j0:j0 + BLOCK]
        mb = np.ceil(tb.max(axis=1))
        Mn = mb if j0 == 0 else np.maximum(M, mb)
        if j0 > 0:
            f = np.exp2(M - Mn)                      # exact powers of two
            acc *= f[:, None]
            l *= f
        M = Mn
        P = np.exp2(tb - M[:, None])
        l += P.sum(axis=1)
        if quantize_p:
            Pq = round_e4m3((P * 2.0 ** P_SHIFT).astype(np.float32).astype(np.float64))
        else:
            Pq = P * 2.0 ** P_SHIFT
        acc += Pq @ vc[j0:j0 + BLOCK]
    out = acc * sv[None, :] / (2.0 ** P_SHIFT * l[:, None])
    lse = (M + np.log2(l)) * math.log(2.0)
    return out, lse, l


def _quantize_qk(qr, kr_scope, recipe):
    fmt = "int8" if recipe == "int8" else "e4m3"
    q8, sq = quantize_rows(qr, fmt)
    k8, sk = quantize_blocks(kr_scope, fmt)
    return q8, sq, k8, sk


def _by_scopes(q8, sq, kr, v8, sv, sparse_k, mode, scale, fmt, quantize):
    """The same per-scope steps with each scope gathered by its token ids (the
    section's prose scopes; for N the listings' rearrange cannot split): q codes
    and v codes as quantized over the whole tensors, k quantized per block of
    128 consecutive keys of the scope (the last block partial), the blocked
    attention, results scattered back to the tokens' rows. Returns out
    (B, N, heads, D), lse and l (B, heads, N)."""
    B, N, nh, D = q8.shape
    out = np.empty((B, N, nh, D))
    lse = np.empty((B, nh, N))
    lsum = np.empty((B, nh, N))
    for s in range(sparse_k):
        tok = O.scope_tokens(N, sparse_k, mode, s)
        if len(tok) == 0:
            continue
        for b in range(B):
            for h in range(nh):
                if quantize:
                    k8, sk = quantize_blocks(kr[b, tok, h], fmt)
                else:
                    k8, sk = kr[b, tok, h], np.ones(len(tok))
                o, ls, l = blocked_attention(sq[b, tok, h], sk, q8[b, tok, h], k8, v8[b, tok, h], sv[b, h], scale,
                                             quantize_p=quantize)
                out[b, tok, h] = o
                lse[b, h, tok] = ls
                lsum[b, h, tok] = l
    return out, lse, lsum


def skiparse_fwd_fp8(q, k, v, T, H, W, sparse_k, mode, theta=10000.0, quantize=True, recipe="int8",
                     with_l=False):
    """q, k, v: (B, N, heads, D) float64 (bf16-valued). Returns out (B, N, heads, D)
    and lse (B, heads, N) (and l (B, heads, N) with with_l). quantize=False
    replaces every rounding by the identity (then the result is exact softmax
    attention)."""
    assert recipe in RECIPES
    B, N, nh, D = q.shape
    scale = 1.0 / math.sqrt(D)
    qr = O.apply_rope(q, T, H, W, theta)
    kr = O.apply_rope(k, T, H, W, theta)
    vv = np.asarray(v, dtype=np.float64)
    fmt = "int8" if recipe == "int8" else "e4m3"
    if quantize:
        q8, sq = quantize_rows(qr, fmt)
        v8, sv = quantize_channels(vv)
    else:
        q8, sq = qr, np.ones(qr.shape[:-1])
        v8, sv = vv, np.ones((B, nh, D))
    if not O.divisible(N, sparse_k, mode):
        out, lse, l = _by_scopes(q8, sq, kr, v8, sv, sparse_k, mode, scale, fmt, quantize)
        return (out, lse, l) if with_l else (out, lse)
    q8r, v8r = (O.rearrange(a, sparse_k, mode) for a in (q8, v8))
    krr = O.rearrange(kr, sparse_k, mode)                              # k blocks are scope blocks
    sqr = O.rearrange(sq[..., None], sparse_k, mode)[..., 0]          # (kB, L, heads)
    o_r = np.empty_like(q8r)
    lse_r = np.empty(q8r.shape[:3])
    l_r = np.empty(q8r.shape[:3])
    for r in range(q8r.shape[0]):
        b = r % B                                    # rearranged batch row r = s * B + b
        for h in range(nh):
            if quantize:
                k8, sk = quantize_blocks(krr[r, :, h], fmt)
            else:
                k8, sk = krr[r, :, h], np.ones(krr.shape[1])
            o, lse, l = blocked_attention(sqr[r, :, h], sk, q8r[r, :, h], k8, v8r[r, :, h],
                                          sv[b, h], scale, quantize_p=quantize)
            o_r[r, :, h] = o
            lse_r[r, :, h] = lse
            l_r[r, :, h] = l
    out = O.reverse(o_r, sparse_k, mode)
    lse = np.ascontiguousarray(np.transpose(O.reverse(lse_r, sparse_k, mode), (0, 2, 1)))
    if with_l:
        return out, lse, np.ascontiguousarray(np.transpose(O.reverse(l_r, sparse_k, mode), (0, 2, 1)))
    return out, lse


def skiparse_fwd_fp8_scope(q, k, v, T, H, W, sparse_k, mode, b, head, s, rows, theta=10000.0, recipe="int8"):
    """The 8-bit forward for chosen query rows of one scope of one (batch, head),
    for checks on large inputs. q, k, v are the full (B, N, heads, D) arrays
    (bf16-valued); only the scope's k rows, the chosen q rows and v[b, :, head]
    (whose per-channel scales span all N tokens) are read. `rows` index the
    scope in scope order. Returns (tokens of those rows, out (n, D), lse (n,),
    l (n,)), the same numbers skiparse_fwd_fp8 gives for those rows."""
    assert recipe in RECIPES
    N, D = q.shape[1], q.shape[3]
    scale = 1.0 / math.sqrt(D)
    fmt = "int8" if recipe == "int8" else "e4m3"
    tok = O.scope_tokens(N, sparse_k, mode, s)
    t, h, w = O.token_coords(N, T, H, W)
    rows = np.asarray(rows)
    qt = tok[rows]
    qr = O._rope_rows(np.asarray(q[b, qt, head], dtype=np.float64), t[qt], h[qt], w[qt], theta)
    kr = O._rope_rows(np.asarray(k[b, tok, head], dtype=np.float64), t[tok], h[tok], w[tok], theta)
    q8, sq = quantize_rows(qr, fmt)
    k8, sk = quantize_blocks(kr, fmt)
    vh = np.asarray(v[b:b + 1, :, head:head + 1], dtype=np.float64)
    v8, sv = quantize_channels(vh)
    out, lse, l = blocked_attention(sq, sk, q8, k8, v8[0, tok, 0], sv[0, 0], scale)
    return qt, out, lse, l
