"""Shared helpers for the parity tests: seeded inputs on the device, calls
through the C ABI, and the oracle comparison with the stated tolerances.

Tolerances (bf16 outputs and gradients vs the float64 oracle): max-abs 2e-2,
mean-abs 2e-3; fp32 RoPE: max-abs 1e-5; fp32 LSE: max-abs 1e-2. A relative RMS
error gate of 1e-2 is applied on top, because N(0,1) inputs give outputs of
order 1/sqrt(L), for which the absolute bounds alone would be loose.
"""
from __future__ import annotations

import numpy as np

from sparse_spatiotemporal_attention_gb300 import synthetic

TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_RMS_REL = 1e-2
TOL_LSE = 1e-2
TOL_ROPE = 1e-5
SENTINEL = 0x7FC1  # a bf16 NaN pattern, never produced by the kernels


def to_device(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def guarded_empty(shape, dtype, dev, pad=4096):
    """A tensor of `shape` inside a larger buffer whose margins hold a sentinel."""
    import torch
    n = int(np.prod(shape))
    if dtype == torch.bfloat16:
        buf = torch.full((n + 2 * pad,), SENTINEL, dtype=torch.int16, device=dev).view(torch.bfloat16)
    else:
        buf = torch.full((n + 2 * pad,), float("nan"), dtype=dtype, device=dev)
    return buf, buf[pad:pad + n].view(shape)


def guards_intact(buf, pad=4096):
    import torch
    head, tail = buf[:pad], buf[-pad:]
    if buf.dtype == torch.bfloat16:
        return bool((head.view(torch.int16) == SENTINEL).all() and (tail.view(torch.int16) == SENTINEL).all())
    return bool(torch.isnan(head).all() and torch.isnan(tail).all())


def compare(name, got, ref, tol_max=TOL_MAX, tol_mean=TOL_MEAN, tol_rel=TOL_RMS_REL):
    """Max-abs and mean-abs bars, and the relative RMS bar wherever the
    reference has a size to be relative to (a gradient that is zero by
    construction, as dq and dk of one-token scopes, is held to the absolute
    bars alone; real outputs here have RMS of order 1e-2 and up)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    rel = np.sqrt(np.sum(err ** 2) / max(np.sum(ref ** 2), 1e-300))
    sized = np.sqrt(np.mean(ref ** 2)) > 1e-5
    msg = f"{name}: max {err.max():.3e} mean {err.mean():.3e} relrms {rel:.3e}"
    assert err.max() <= tol_max and err.mean() <= tol_mean and (rel <= tol_rel or not sized), msg
    return msg


def run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode, theta=10000.0, guard=True, pad=4096):
    """pad: elements before (and after) the guarded bf16 output, e.g. 4104 puts
    its base 16 bytes past a 32-byte boundary."""
    import torch
    q, kk, v = (to_device(ins[n], dev) for n in ("q", "k", "v"))
    if guard:
        obuf, out = guarded_empty((B, N, heads, D), torch.bfloat16, dev, pad)
        lbuf, lse = guarded_empty((B, heads, N), torch.float32, dev)
    else:
        obuf = lbuf = None
        out = torch.empty((B, N, heads, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
    skp.skiparse_attn_fwd(q, kk, v, out, lse, T, H, W, k, mode, theta)
    torch.cuda.synchronize()
    if guard:
        assert guards_intact(obuf, pad) and guards_intact(lbuf), "forward wrote outside its outputs"
    return dict(q=q, k=kk, v=v, out=out, lse=lse)


def run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode, theta=10000.0, guard=True, pad=4096):
    import torch
    do = to_device(ins["do"], dev)
    nbytes = skp.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    bufs, outs = [], []
    for _ in range(3):
        if guard:
            b, t = guarded_empty((B, N, heads, D), torch.bfloat16, dev, pad)
        else:
            b, t = None, torch.empty((B, N, heads, D), dtype=torch.bfloat16, device=dev)
        bufs.append(b)
        outs.append(t)
    dq, dk, dv = outs
    skp.skiparse_attn_bwd(fw["q"], fw["k"], fw["v"], fw["out"], fw["lse"], do, dq, dk, dv, ws,
                          T, H, W, k, mode, theta)
    torch.cuda.synchronize()
    if guard:
        assert all(guards_intact(b, pad) for b in bufs), "backward wrote outside its outputs"
    return dict(dq=dq, dk=dk, dv=dv, do=do)


def host(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy().astype(np.float64)


def f64_inputs(ins):
    return {n: synthetic.bf16_bits_to_f64(a) for n, a in ins.items()}
