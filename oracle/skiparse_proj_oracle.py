"""Plain CPU float64 oracle for the Q/K/V projection with RoPE.

TEST INFRASTRUCTURE ONLY: imported by tests and bench.py's CPU legs, never by
the library. It builds on skiparse_oracle.py's RoPE and shares no code with
the GPU path.

The Skiparse listings ("Open-Sora Plan" docs, section "Skiparse Attention",
single- and group-skip implementations) compute q, k, v = Q(x), K(x), V(x)
and then rotate q and k by RoPE before the rearrange. Readings taken here
(the listings show the calls only):

  * Q, K and V are linear layers, y = x W^T + b, on x of shape (B, N, C), with
    heads * D outputs each; the three weights are stacked into one
    (3 heads D, C) matrix in the order Q, K, V, and b is optional;
  * the outputs are split per head into (B, N, heads, D) (head h owns columns
    h D .. h D + D - 1 of its block), the layout the attention takes;
  * RoPE is skiparse_oracle.apply_rope (the same 3D RoPE the attention
    applies) on q and k, at each token's original (t, h, w); v is not rotated.

Everything is float64 from the bf16-valued inputs; the GPU rounds each output
to bf16 once. Parity pins: tests/test_oracle_proj.py.
"""
from __future__ import annotations

import numpy as np

from . import skiparse_oracle as O


def qkv_rope(x, w, bias, heads, D, T, H, W, theta=10000.0):
    """x (B, N, C), w (3 heads D, C), bias (3 heads D,) or None, float64.
    Returns q, k, v of shape (B, N, heads, D)."""
    B, N, C = x.shape
    hd = heads * D
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, None, :]
    q = y[..., 0:hd].reshape(B, N, heads, D)
    k = y[..., hd:2 * hd].reshape(B, N, heads, D)
    v = y[..., 2 * hd:3 * hd].reshape(B, N, heads, D)
    return O.apply_rope(q, T, H, W, theta), O.apply_rope(k, T, H, W, theta), np.array(v)


def qkv_rope_rows(x, w, bias, heads, D, T, H, W, rows, theta=10000.0):
    """The same for selected rows only: rows is a list of (b, n); returns q, k,
    v of shape (len(rows), heads, D) (for full-size samples)."""
    hd = heads * D
    b_idx = np.array([r[0] for r in rows])
    n_idx = np.array([r[1] for r in rows])
    xs = np.asarray(x, dtype=np.float64)[b_idx, n_idx]                  # (R, C)
    y = xs @ np.asarray(w, dtype=np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    t, h, ww = O.token_coords(x.shape[1], T, H, W)
    out = []
    for blk in range(3):
        part = y[:, blk * hd:(blk + 1) * hd].reshape(len(rows), heads, D)
        if blk < 2:
            part = np.stack([O._rope_rows(part[:, hh], t[n_idx], h[n_idx], ww[n_idx], theta)
                             for hh in range(heads)], axis=1)
        out.append(part)
    return tuple(out)
