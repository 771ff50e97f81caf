"""Seeded random small shapes through the C ABI against the float64 oracle:
grids of 1-4 frames of up to 12 x 24 tokens, either skip mode, k from 1 to 8
(single skip) or a power of two up to 8 (group skip), both head sizes and
batch 1 or 2. Many of them leave k (single) or k^2 (group) not dividing N, so
the scopes differ in length, some scopes hold a single token or none, and
most tiles are ragged. Forward and backward at the bars of the other parity
tests (out, dq, dk, dv: max-abs 2e-2, mean-abs 2e-3, relative RMS 1e-2; LSE
max-abs 1e-2, relative 1e-3, or 2^-8 where a scope holds one token).
"""
import numpy as np
import pytest

from oracle import skiparse_oracle as O
from sparse_spatiotemporal_attention_gb300 import synthetic
import skiparse_testlib as tl

pytestmark = pytest.mark.gpu


def _cases(n=16, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        mode = O.SINGLE if rng.integers(2) == 0 else O.GROUP
        k = int(rng.integers(1, 9)) if mode == O.SINGLE else int(rng.choice([1, 2, 4, 8]))
        T, H, W = int(rng.integers(1, 5)), int(rng.integers(1, 13)), int(rng.integers(1, 25))
        B, heads, D = int(rng.integers(1, 3)), int(rng.integers(1, 4)), int(rng.choice([64, 128]))
        out.append((B, heads, D, T, H, W, k, mode))
    return out


CASES = _cases()


def _ids(c):
    B, h, D, T, H, W, k, m = c
    return f"B{B}h{h}D{D}_{T}x{H}x{W}_k{k}_{'single' if m == O.SINGLE else 'group'}"


@pytest.fixture(scope="module")
def env():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import sparse_spatiotemporal_attention_gb300 as skp
    assert torch.cuda.is_available()
    return skp, torch.device("cuda:0")


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_random_shape_forward_backward(env, case):
    skp, dev = env
    B, heads, D, T, H, W, k, mode = case
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode)
    bw = tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode)
    f = tl.f64_inputs(ins)
    rdq, rdk, rdv, rout, rlse = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
    tl.compare("out", tl.host(fw["out"]), rout)
    lens = [len(O.prose_scope_tokens(N, k, mode, s)) for s in range(k)]
    lse_rel = 2.0 ** -8 if min(n for n in lens if n) == 1 else 1e-3
    tl.compare("lse", tl.host(fw["lse"]), rlse, tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE, tol_rel=lse_rel)
    tl.compare("dv", tl.host(bw["dv"]), rdv)
    tl.compare("dk", tl.host(bw["dk"]), rdk)
    tl.compare("dq", tl.host(bw["dq"]), rdq)
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)
