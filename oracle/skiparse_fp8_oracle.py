"""Plain CPU float64 oracle for the 8-bit Skiparse attention forward pass.

TEST INFRASTRUCTURE ONLY: imported by tests and bench.py's CPU legs, never by
the library. It builds on skiparse_oracle.py (RoPE, rearrange) and shares no
code with the GPU path.

The method follows the Wan 2.1 report ("Open and Advanced Large-Scale Video
Generative Models"), section 4 "Model Design and Acceleration", 4.4.3
"Quantization", paragraph "8-Bit FlashAttention":
attention inputs are quantized to 8 bits for the two products S = Q K^T and
O = P V, and the products of successive key blocks are accumulated in fp32.
Readings taken here (the page gives the recipe for Hopper and no formulas):

  * both products use FP8 E4M3 operands. The page's INT8 for S = Q K^T is not
    a fast path on the target (its INT8 tensor rate is far below its FP8 rate);
    E4M3 keeps the page's point of 8-bit operands with per-row scales;
  * q and k are quantized after RoPE: q per (token, head) row, k per block of
    128 consecutive keys of a scope (a per-block scale, as SageAttention's),
    with scale s = max|x| / 448 over the row or block (448 = largest finite
    E4M3) and codes RNE(x * 448 / max|x|) (all-zero data: scale 1, codes 0);
  * v is quantized per (batch, head, channel) over all N tokens with the same
    rule, so its scale factors out of O = P V column by column;
  * attention runs per scope over blocks of 128 keys (scope order) with an
    online softmax in base 2: the running row max m (of S * scale * log2 e) is
    set by the first block and raised only when a later block's max exceeds it
    by more than 2 (then O and l are rescaled by 2^(m_old - m_new)), the lazy
    rescaling of the fp32 kernel with a threshold of 2^2 instead of 2^8, so
    that P = 2^(S * scale * log2 e - m) stays below 2^2;
  * P is quantized as RNE_E4M3(P * 2^6) for O += P V (fp32 cross-block
    accumulation): 2^2 * 2^6 = 256 < 448 keeps every code below saturation
    (with the fp32 kernel's 2^8 threshold, P * 2^8 would saturate and the
    error grows with the number of key blocks), while small P stay normal
    down to 2^-12; the row sum l adds the unquantized P;
  * out = O * s_v / (2^6 * l) (bf16 on the GPU), lse = (m + log2 l) * ln 2.

Where floating point decides a code, it is decided in the kernel's precision
(float32): the values handed to the E4M3 rounding (q, k, v times 448 / max|x|,
and P * 2^6 with P = 2^t, t = S * c - m + 6 formed as one float32 fused
multiply-add and 2^t in float32) are float32 numbers; everything else
(RoPE, the products, the sums, the rescaling, the output) is float64.
Parity pins: tests/test_oracle_fp8.py.
"""
from __future__ import annotations

import math

import numpy as np

from . import skiparse_oracle as O

E4M3_MAX = 448.0
P_SCALE = 64.0        # 2^6
BLOCK = 128
LAZY_LOG2 = 2.0       # rescale when a block's row max exceeds the running max by more than 2^2


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
    saturating at +-448 (the GPU's cvt.rn.satfinite)."""
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


def _f32_codes(x: np.ndarray, amax: np.ndarray) -> np.ndarray:
    """E4M3 codes of x * (448 / amax), the product formed in float32."""
    x32 = np.asarray(x, dtype=np.float32)
    a32 = np.asarray(amax, dtype=np.float32)
    inv = np.where(a32 > 0, np.float32(E4M3_MAX) / np.where(a32 > 0, a32, np.float32(1)), np.float32(0))
    return round_e4m3((x32 * inv.astype(np.float32)).astype(np.float64))


def quantize_rows(x: np.ndarray):
    """Per-row E4M3 codes and scales over the last axis: x ~ codes * scale."""
    x32 = np.asarray(x, dtype=np.float32).astype(np.float64)
    amax = np.abs(x32).max(axis=-1, keepdims=True)
    codes = _f32_codes(x32, amax)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    return codes, scale[..., 0]


def quantize_blocks(x: np.ndarray, block: int = BLOCK):
    """x (L, D) in scope order: per block of `block` rows, E4M3 codes and one
    scale (returned per row, constant within a block)."""
    codes = np.empty_like(x)
    scale = np.empty(x.shape[0])
    for j0 in range(0, x.shape[0], block):
        c, s_ = quantize_rows(x[j0:j0 + block].reshape(1, -1))
        codes[j0:j0 + block] = c.reshape(-1, x.shape[1])
        scale[j0:j0 + block] = s_[0]
    return codes, scale


def quantize_channels(v: np.ndarray):
    """v (B, N, heads, D): per (b, head, channel) E4M3 codes and scales over N."""
    v32 = np.asarray(v, dtype=np.float32).astype(np.float64)
    amax = np.abs(v32).max(axis=1, keepdims=True)                 # (B, 1, heads, D)
    codes = _f32_codes(v32, amax)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    return codes, scale[:, 0]                                       # (B, heads, D)


def blocked_attention(sq, sk, q8, k8, v8, sv, scale, quantize_p=True):
    """One scope problem: q8 (Lq, D) codes with row scales sq (Lq,), k8 (L, D) with
    sk (L,), v8 (L, D) with channel scales sv (D,). Online softmax over blocks of
    128 keys with the lazy rule; returns (out (Lq, D), lse (Lq,)). Query rows are
    independent, so q8 may hold any subset of the scope's rows (Lq <= L)."""
    Lq, D = q8.shape
    L = k8.shape[0]
    log2e = 1.0 / math.log(2.0)
    raw = q8 @ k8.T                                                  # exact: sums of E4M3 products
    if quantize_p:
        # per-row and per-block factor c = sq * sk * scale * log2 e and the scores
        # in float32, as the kernel forms the values its codes are decided on
        c = (np.float32(scale * log2e) * sq.astype(np.float32))[:, None] * sk.astype(np.float32)[None, :]
        c = c.astype(np.float32).astype(np.float64)
        S = raw.astype(np.float32).astype(np.float64) * c            # (Lq, L), base-2 units
    else:
        S = (sq[:, None] * sk[None, :]) * raw * scale * log2e
    m = np.zeros(Lq)
    l = np.zeros(Lq)
    acc = np.zeros((Lq, D))
    for j0 in range(0, L, BLOCK):
        Sb = S[:, j0:j0 + BLOCK]
        mx = Sb.max(axis=1)
        if j0 == 0:
            m = mx.copy()
        else:
            up = mx > m + LAZY_LOG2
            m_new = np.where(up, mx, m)
            f = np.exp2(m - m_new)
            acc *= f[:, None]
            l *= f
            m = m_new
        if quantize_p:
            # 2^6 P = 2^t, t = S * c + (6 - m) as one float32 fused multiply-add, 2^t in float32
            shift = (np.float32(math.log2(P_SCALE)) - m.astype(np.float32)).astype(np.float64)
            t = (raw[:, j0:j0 + BLOCK].astype(np.float32).astype(np.float64) * c[:, j0:j0 + BLOCK]
                 + shift[:, None]).astype(np.float32)
            Ps = np.exp2(t).astype(np.float64)                       # 2^6 P
            l += Ps.sum(axis=1) / P_SCALE
            Pq = round_e4m3(Ps)
        else:
            P = np.exp2(Sb - m[:, None])
            l += P.sum(axis=1)
            Pq = P * P_SCALE
        acc += Pq @ v8[j0:j0 + BLOCK]
    out = acc * sv[None, :] / (P_SCALE * l[:, None])
    lse = (m + np.log2(l)) * math.log(2.0)
    return out, lse


def skiparse_fwd_fp8(q, k, v, T, H, W, sparse_k, mode, theta=10000.0, quantize=True):
    """q, k, v: (B, N, heads, D) float64 (bf16-valued). Returns out (B, N, heads, D)
    and lse (B, heads, N). quantize=False replaces every E4M3 rounding by the
    identity (then the result is exact softmax attention)."""
    B, N, nh, D = q.shape
    scale = 1.0 / math.sqrt(D)
    qr = O.apply_rope(q, T, H, W, theta)
    kr = O.apply_rope(k, T, H, W, theta)
    vv = np.asarray(v, dtype=np.float64)
    if quantize:
        q8, sq = quantize_rows(qr)
        v8, sv = quantize_channels(vv)
    else:
        q8, sq = qr, np.ones(qr.shape[:-1])
        v8, sv = vv, np.ones((B, nh, D))
    q8r, v8r = (O.rearrange(a, sparse_k, mode) for a in (q8, v8))
    krr = O.rearrange(kr, sparse_k, mode)                              # k blocks are scope blocks
    sqr = O.rearrange(sq[..., None], sparse_k, mode)[..., 0]          # (kB, L, heads)
    o_r = np.empty_like(q8r)
    lse_r = np.empty(q8r.shape[:3])
    for r in range(q8r.shape[0]):
        b = r % B                                    # rearranged batch row r = s * B + b
        for h in range(nh):
            if quantize:
                k8, sk = quantize_blocks(krr[r, :, h])
            else:
                k8, sk = krr[r, :, h], np.ones(krr.shape[1])
            o, lse = blocked_attention(sqr[r, :, h], sk, q8r[r, :, h], k8, v8r[r, :, h],
                                       sv[b, h], scale, quantize_p=quantize)
            o_r[r, :, h] = o
            lse_r[r, :, h] = lse
    out = O.reverse(o_r, sparse_k, mode)
    lse = O.reverse(lse_r, sparse_k, mode)
    return out, np.ascontiguousarray(np.transpose(lse, (0, 2, 1)))


def skiparse_fwd_fp8_scope(q, k, v, T, H, W, sparse_k, mode, b, head, s, rows, theta=10000.0):
    """The 8-bit forward for chosen query rows of one scope of one (batch, head),
    for checks on large inputs. q, k, v are the full (B, N, heads, D) arrays
    (bf16-valued); only the scope's k rows, the chosen q rows and v[b, :, head]
    (whose per-channel scales span all N tokens) are read. `rows` index the
    scope in scope order. Returns (tokens of those rows, out (n, D), lse (n,)),
    the same numbers skiparse_fwd_fp8 gives for those rows."""
    N, D = q.shape[1], q.shape[3]
    scale = 1.0 / math.sqrt(D)
    tok = O.scope_tokens(N, sparse_k, mode, s)
    t, h, w = O.token_coords(N, T, H, W)
    rows = np.asarray(rows)
    qt = tok[rows]
    qr = O._rope_rows(np.asarray(q[b, qt, head], dtype=np.float64), t[qt], h[qt], w[qt], theta)
    kr = O._rope_rows(np.asarray(k[b, tok, head], dtype=np.float64), t[tok], h[tok], w[tok], theta)
    q8, sq = quantize_rows(qr)
    k8, sk = quantize_blocks(kr)
    vh = np.asarray(v[b:b + 1, :, head:head + 1], dtype=np.float64)
    v8, sv = quantize_channels(vh)
    out, lse = blocked_attention(sq, sk, q8, k8, v8[0, tok, 0], sv[0, 0], scale)
    return qt, out, lse
