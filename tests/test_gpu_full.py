"""Parity at the full workload sizes, in the launch configuration bench.py
times (same shapes, seeds and entry points), on sampled outputs the oracle
computes scope by scope.

Workloads (latent grids shaped like video DiT tokens):
  single skip  B=1 heads=24 D=128 grid 8x32x32  (N=8192)  k=4, forward
  group skip   B=2 heads=24 D=128 grid 24x22x40 (N=21120) k=4, forward (+k=1)
  group skip   B=1 heads=24 D=128 grid 16x45x80 (N=57600) k=4, forward (+k=1)
  training     B=2 heads=24 D=128 grid 24x22x40 (N=21120) k=4, forward+backward
Sampling: whole scopes for the backward (every token of the scope); query
rows for the forward: the first and last 64 rows of a scope (the last ones
cover the ragged tail tile) plus 64 random rows.
"""
import numpy as np
import pytest

from oracle import skiparse_oracle as O
from sparse_spatiotemporal_attention_gb300 import synthetic
import skiparse_testlib as tl

pytestmark = pytest.mark.gpu

_INPUT_CACHE = {}


def inputs(B, N, heads, D, with_grad):
    key = (B, N, heads, D, with_grad)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = synthetic.attention_inputs(B, N, heads, D, with_grad=with_grad)
    return _INPUT_CACHE[key]


@pytest.fixture(scope="module")
def env():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import sparse_spatiotemporal_attention_gb300 as skp
    assert torch.cuda.is_available()
    return skp, torch.device("cuda:0")


def _slice(bits, b, head):
    return synthetic.bf16_bits_to_f64(bits[b:b + 1, :, head:head + 1])


def _rows(L, rng):
    r = np.unique(np.concatenate([np.arange(min(64, L)), np.arange(max(0, L - 64), L),
                                  rng.integers(0, L, 64)]))
    return r


FWD = [
    ("single_8x32x32_k4", 1, 24, 128, (8, 32, 32), 4, O.SINGLE),
    ("group_24x22x40_k4", 2, 24, 128, (24, 22, 40), 4, O.GROUP),
    ("group_24x22x40_k1", 2, 24, 128, (24, 22, 40), 1, O.GROUP),
    ("group_16x45x80_k4", 1, 24, 128, (16, 45, 80), 4, O.GROUP),
    ("group_16x45x80_k1", 1, 24, 128, (16, 45, 80), 1, O.GROUP),
]


@pytest.mark.parametrize("name,B,heads,D,grid,k,mode", FWD, ids=[f[0] for f in FWD])
def test_full_forward_sampled(env, name, B, heads, D, grid, k, mode):
    skp, dev = env
    T, H, W = grid
    N = T * H * W
    ins = inputs(B, N, heads, D, False)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode, guard=False)
    out = fw["out"].float().cpu().numpy()
    lse = fw["lse"].cpu().numpy()
    rng = np.random.default_rng(123)
    picks = [(0, 0, 0), (B - 1, heads - 1, k - 1), (B - 1, 7 % heads, (k // 2))]
    for b, h, s in picks:
        L = N // k
        rows = _rows(L, rng)
        sub = {n: _slice(ins[n], b, h) for n in ("q", "k", "v")}
        r = O.skiparse_scope(sub["q"], sub["k"], sub["v"], None, T, H, W, k, mode, 0, 0, s, rows=rows)
        tok = r["tokens"][rows]
        tl.compare(f"{name} out b{b} h{h} s{s}", out[b, tok, h], r["out"])
        tl.compare(f"{name} lse b{b} h{h} s{s}", lse[b, h, tok], r["lse"], tol_max=tl.TOL_LSE,
                   tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


def test_full_training_step_sampled(env):
    skp, dev = env
    B, heads, D, (T, H, W), k, mode = 2, 24, 128, (24, 22, 40), 4, O.GROUP
    N = T * H * W
    ins = inputs(B, N, heads, D, True)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode, guard=False)
    bw = tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode, guard=False)
    got = {n: bw[n].float().cpu().numpy() for n in ("dq", "dk", "dv")}
    got["out"] = fw["out"].float().cpu().numpy()
    for b, h, s in [(0, 0, 0), (1, 23, 3)]:
        sub = {n: _slice(ins[n], b, h) for n in ("q", "k", "v", "do")}
        r = O.skiparse_scope(sub["q"], sub["k"], sub["v"], sub["do"], T, H, W, k, mode, 0, 0, s)
        tok = r["tokens"]
        for n in ("out", "dq", "dk", "dv"):
            tl.compare(f"train {n} b{b} h{h} s{s}", got[n][b, tok, h], r[n])
    for n in ("dq", "dk", "dv"):
        assert np.all(np.isfinite(got[n])), n
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


def test_full_training_step_sampled_unequal_scopes(env):
    """The training step at a size next to the bench's with N that k^2 does not
    divide (23x22x41: N = 20,746, scopes of 5,188, 5,188, 5,186 and 5,184
    tokens): forward and backward through the scope-ordered copies, whole
    scopes of two (batch, head) pairs against the oracle."""
    skp, dev = env
    B, heads, D, (T, H, W), k, mode = 2, 24, 128, (23, 22, 41), 4, O.GROUP
    N = T * H * W
    assert not O.divisible(N, k, mode)
    ins = inputs(B, N, heads, D, True)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode, guard=False)
    bw = tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode, guard=False)
    got = {n: bw[n].float().cpu().numpy() for n in ("dq", "dk", "dv")}
    got["out"] = fw["out"].float().cpu().numpy()
    got_lse = fw["lse"].cpu().numpy()
    for b, h, s in [(0, 5, 0), (1, 17, 3)]:
        sub = {n: _slice(ins[n], b, h) for n in ("q", "k", "v", "do")}
        r = O.skiparse_scope(sub["q"], sub["k"], sub["v"], sub["do"], T, H, W, k, mode, 0, 0, s)
        tok = r["tokens"]
        assert len(tok) == len(O.prose_scope_tokens(N, k, mode, s))
        for n in ("out", "dq", "dk", "dv"):
            tl.compare(f"unequal {n} b{b} h{h} s{s}", got[n][b, tok, h], r[n])
        tl.compare(f"unequal lse b{b} h{h} s{s}", got_lse[b, h, tok], r["lse"], tol_max=tl.TOL_LSE,
                   tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    for n in ("dq", "dk", "dv"):
        assert np.all(np.isfinite(got[n])), n
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)
