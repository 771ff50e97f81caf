"""GPU parity of the 8-bit forward pass (skiparse_attn_fwd_fp8) through the C
ABI against the 8-bit oracle (oracle/skiparse_fp8_oracle.py), which applies the
same quantization, deciding every E4M3 code on float32 values as the kernel
does. The two differ by the final bf16 rounding and, rarely, by one code where
a value lies within an ulp of a rounding midpoint, so the bf16 path's bars
apply (out mean-abs 2e-3, relative RMS 1e-2, max-abs 2e-2 for all but one
element in 10^4 and 0.1 for every element; LSE max-abs 1e-2). Against exact attention (the
main oracle) the kernel's error must not exceed the 8-bit method's own (the
oracle's) beyond bf16 rounding, and the method's error stays of the size E4M3
operands give (relative RMS < 8 %; about 5 % on these inputs)."""
import numpy as np
import pytest

from oracle import skiparse_fp8_oracle as F
from oracle import skiparse_oracle as O
from sparse_spatiotemporal_attention_gb300 import synthetic
import skiparse_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import sparse_spatiotemporal_attention_gb300 as skp
    assert torch.cuda.is_available()
    return skp, torch.device("cuda:0")


# (B, heads, T, H, W, k, mode); D = 128
CASES = [
    (1, 2, 3, 10, 10, 2, O.GROUP),      # L = 150: two tiles, ragged tail
    (2, 2, 3, 20, 24, 4, O.SINGLE),     # L = 360: three tiles (odd: tile B of the last pair past the scope)
    (1, 2, 2, 8, 16, 1, O.SINGLE),      # k = 1: dense, L = 256
    (1, 1, 2, 16, 32, 8, O.GROUP),      # k = 8, L = 128
    (1, 1, 8, 32, 32, 4, O.SINGLE),     # L = 2048, 16 tiles
]


def _ids(c):
    B, h, T, H, W, k, m = c
    return f"B{B}h{h}_{T}x{H}x{W}_k{k}_{'single' if m == O.SINGLE else 'group'}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_fp8_forward_parity(env, case):
    import torch
    skp, dev = env
    B, heads, T, H, W, k, mode = case
    D, N = 128, T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D)
    q, kk, v = (tl.to_device(ins[n], dev) for n in ("q", "k", "v"))
    obuf, out = tl.guarded_empty((B, N, heads, D), torch.bfloat16, dev)
    lbuf, lse = tl.guarded_empty((B, heads, N), torch.float32, dev)
    skp.skiparse_attn_fwd_fp8(q, kk, v, out, lse, T, H, W, k, mode)
    torch.cuda.synchronize()
    assert tl.guards_intact(obuf) and tl.guards_intact(lbuf), "8-bit forward wrote outside its outputs"
    f = tl.f64_inputs(ins)
    rout, rlse = F.skiparse_fwd_fp8(f["q"], f["k"], f["v"], T, H, W, k, mode)
    got = tl.host(out)
    # both sides decide every E4M3 code on float32 values, but sin / cos and 2^x
    # are different float32 implementations on the two sides, so a value within
    # an ulp of a rounding midpoint can take the neighbouring code: an isolated
    # element may then miss the max-abs bar (one in 10^4 allowed, none past 0.1)
    err = np.abs(got - rout)
    assert np.all(np.isfinite(got))
    assert err.mean() <= tl.TOL_MEAN, err.mean()
    assert np.sqrt(np.sum(err ** 2) / np.sum(rout ** 2)) <= tl.TOL_RMS_REL
    assert np.count_nonzero(err > tl.TOL_MAX) <= max(1, err.size // 10000), np.count_nonzero(err > tl.TOL_MAX)
    assert err.max() <= 0.1, err.max()
    tl.compare("lse", tl.host(lse), rlse, tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    # against exact attention the kernel adds nothing to the method's own error
    eout, _ = O.skiparse_fwd(f["q"], f["k"], f["v"], T, H, W, k, mode)
    rel_gpu = np.sqrt(np.sum((got - eout) ** 2) / np.sum(eout ** 2))
    rel_method = np.sqrt(np.sum((rout - eout) ** 2) / np.sum(eout ** 2))
    assert rel_gpu <= 1.05 * rel_method + 2e-3, (rel_gpu, rel_method)
    assert rel_method < 0.08, rel_method
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


# the 8-bit workloads the bench times: (B, heads, (T, H, W), k, mode); D = 128
FULL = [
    ("group_16x45x80_k4", 1, 24, (16, 45, 80), 4, O.GROUP),
    ("group_24x22x40_k4", 2, 24, (24, 22, 40), 4, O.GROUP),
    ("single_8x32x32_k4", 1, 24, (8, 32, 32), 4, O.SINGLE),
]


@pytest.mark.parametrize("name,B,heads,grid,k,mode", FULL, ids=[f[0] for f in FULL])
def test_fp8_full_size_sampled(env, name, B, heads, grid, k, mode):
    """Full size, launched as the bench launches it (its workspace, a side
    stream): the first and last 64 rows and 64 random rows of three scopes
    against the 8-bit oracle's scope routine, with the parity cases' bars."""
    import torch
    skp, dev = env
    T, H, W = grid
    D, N = 128, T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D)
    q, kk, v = (tl.to_device(ins[n], dev) for n in ("q", "k", "v"))
    out = torch.empty((B, N, heads, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
    ws = torch.empty(skp.skiparse_attn_fwd_fp8_workspace_bytes(B, heads, N, D, T, H, W, k, mode),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    skp.skiparse_attn_fwd_fp8(q, kk, v, out, lse, T, H, W, k, mode, stream=stream, workspace=ws)
    stream.synchronize()
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)
    got, glse = tl.host(out), tl.host(lse)
    assert np.all(np.isfinite(got)) and np.all(np.isfinite(glse))
    L = N // k
    rng = np.random.default_rng(31)
    gsel, rsel, gl, rl = [], [], [], []
    for b, h, s in [(0, 0, 0), (B - 1, heads - 1, k - 1), (B - 1, 7, k // 2)]:
        rows = np.unique(np.concatenate([np.arange(64), np.arange(L - 64, L), rng.integers(0, L, 64)]))
        sub = {n: synthetic.bf16_bits_to_f64(ins[n][b:b + 1, :, h:h + 1]) for n in ("q", "k", "v")}
        tok, ro, rlse = F.skiparse_fwd_fp8_scope(sub["q"], sub["k"], sub["v"], T, H, W, k, mode, 0, 0, s, rows)
        gsel.append(got[b, tok, h])
        rsel.append(ro)
        gl.append(glse[b, h, tok])
        rl.append(rlse)
    g_, r_ = np.concatenate(gsel), np.concatenate(rsel)
    err = np.abs(g_ - r_)
    assert err.mean() <= tl.TOL_MEAN, err.mean()
    assert np.sqrt(np.sum(err ** 2) / np.sum(r_ ** 2)) <= tl.TOL_RMS_REL
    assert np.count_nonzero(err > tl.TOL_MAX) <= max(1, err.size // 10000), np.count_nonzero(err > tl.TOL_MAX)
    assert err.max() <= 0.1, err.max()
    tl.compare("lse", np.concatenate(gl), np.concatenate(rl), tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE,
               tol_rel=1e-3)


def test_fp8_rejects_d64_and_small_workspace(env):
    import torch
    skp, dev = env
    q = torch.zeros((1, 256, 2, 64), dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    lse = torch.zeros((1, 2, 256), dtype=torch.float32, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(skp.SkiparseError) as e:
        skp.skiparse_attn_fwd_fp8(q, q, q, out, lse, 4, 8, 8, 2, 0, workspace=ws)
    assert e.value.status == -3
    q = torch.zeros((1, 256, 2, 128), dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    with pytest.raises(skp.SkiparseError) as e:
        skp.skiparse_attn_fwd_fp8(q, q, q, out, lse, 4, 8, 8, 2, 0, workspace=ws[:1024])
    assert e.value.status == -6


def test_fp8_forward_prerotated_inputs(env):
    """rope_theta = 0: q and k are taken as already rotated (no rotation in the
    prep kernel), against the 8-bit oracle with the same convention."""
    import torch
    skp, dev = env
    B, heads, T, H, W, k, mode = 1, 2, 3, 10, 10, 2, O.GROUP
    D, N = 128, T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D)
    q, kk, v = (tl.to_device(ins[n], dev) for n in ("q", "k", "v"))
    obuf, out = tl.guarded_empty((B, N, heads, D), torch.bfloat16, dev)
    lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
    skp.skiparse_attn_fwd_fp8(q, kk, v, out, lse, T, H, W, k, mode, rope_theta=0.0)
    torch.cuda.synchronize()
    assert tl.guards_intact(obuf)
    f = tl.f64_inputs(ins)
    rout, rlse = F.skiparse_fwd_fp8(f["q"], f["k"], f["v"], T, H, W, k, mode, theta=0.0)
    err = np.abs(tl.host(out) - rout)
    assert err.mean() <= tl.TOL_MEAN and err.max() <= 0.1
    assert np.sqrt(np.sum(err ** 2) / np.sum(rout ** 2)) <= tl.TOL_RMS_REL
    tl.compare("lse", tl.host(lse), rlse, tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


def test_rope_table_limit_rejected_on_the_host(env):
    """16 T + 24 (H + W) = 8200 RoPE pairs exceed the 8192 every entry point
    accepts: both forwards refuse the call before any launch (UNSUPPORTED) and
    leave their outputs untouched."""
    import torch
    skp, dev = env
    T, H, W, heads, D = 1, 1, 340, 1, 128
    N = T * H * W
    q = torch.zeros((1, N, heads, D), dtype=torch.bfloat16, device=dev)
    out = torch.full_like(q, 3.0)
    lse = torch.full((1, heads, N), 5.0, dtype=torch.float32, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    for call in (skp.skiparse_attn_fwd_fp8, skp.skiparse_attn_fwd):
        with pytest.raises(skp.SkiparseError) as e:
            call(q, q, q, out, lse, T, H, W, 1, 0, workspace=ws)
        assert e.value.status == -3
    torch.cuda.synchronize()
    assert bool((out == 3.0).all()) and bool((lse == 5.0).all())
