"""Scope subsets (skiparse_attn_fwd_scopes / skiparse_attn_bwd_scopes) on one
GPU: G calls with the round-robin shards (g, G) of the scopes, as G ranks would
make them, each writing exactly the rows of its scopes' tokens (every other row
keeps a sentinel), and together the whole forward and backward of the oracle
within the parity bars. Scopes never interact, so this is the whole of the
multi-GPU scope split: no data moves between the calls."""
import numpy as np
import pytest

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


# (B, heads, D, T, H, W, k, mode, G)
CASES = [
    (1, 2, 128, 3, 20, 24, 4, O.SINGLE, 2),     # L = 360, two ranks of two scopes
    (2, 2, 128, 3, 10, 10, 4, O.GROUP, 3),      # ranks take {0, 3}, {1}, {2}
    (1, 2, 64, 5, 5, 41, 4, O.SINGLE, 4),       # unequal scopes (N = 1025), one scope per rank
    (1, 2, 128, 3, 7, 9, 4, O.GROUP, 2),        # unequal scopes with a partial group
]


def _ids(c):
    B, h, D, T, H, W, k, m, G = c
    return f"B{B}h{h}D{D}_{T}x{H}x{W}_k{k}_{'single' if m == O.SINGLE else 'group'}_G{G}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_scope_shards_cover_the_call(env, case):
    import torch
    skp, dev = env
    B, heads, D, T, H, W, k, mode, G = case
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True)
    q, kk, v, do = (tl.to_device(ins[n], dev) for n in ("q", "k", "v", "do"))
    sent = torch.tensor([tl.SENTINEL], dtype=torch.int16).view(torch.bfloat16).item()
    out = torch.full((B, N, heads, D), float("nan"), dtype=torch.bfloat16, device=dev)
    out.view(torch.int16).fill_(tl.SENTINEL)
    lse = torch.full((B, heads, N), float("nan"), dtype=torch.float32, device=dev)
    grads = [torch.empty_like(out) for _ in range(3)]
    for gt in grads:
        gt.view(torch.int16).fill_(tl.SENTINEL)
    scope_of, _ = O.index_maps(N, k, mode)
    fws = torch.empty(skp.skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode), dtype=torch.uint8,
                      device=dev)
    bws = torch.empty(skp.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode), dtype=torch.uint8,
                      device=dev)
    done = np.zeros(N, dtype=bool)
    for rank in range(G):
        first, step = skp.scope_shard(k, G, rank)
        skp.skiparse_attn_fwd_scopes(q, kk, v, out, lse, T, H, W, k, mode, first, step, workspace=fws)
        torch.cuda.synchronize()
        done |= (scope_of % step) == first
        written = (out.view(torch.int16) != tl.SENTINEL).any(dim=3).any(dim=2).any(dim=0).cpu().numpy()
        assert np.array_equal(written, done), f"rank {rank}: forward wrote other scopes' rows"
        assert np.array_equal(~torch.isnan(lse).any(dim=1).any(dim=0).cpu().numpy(), done)
    for rank in range(G):
        first, step = skp.scope_shard(k, G, rank)
        skp.skiparse_attn_bwd_scopes(q, kk, v, out, lse, do, *grads, bws, T, H, W, k, mode, first, step)
        torch.cuda.synchronize()
        for name, gt in zip(("dq", "dk", "dv"), grads):
            written = (gt.view(torch.int16) != tl.SENTINEL).any(dim=3).any(dim=2).any(dim=0).cpu().numpy()
            assert np.array_equal(written, (scope_of % G) <= rank), f"rank {rank}: {name} rows"
    f = tl.f64_inputs(ins)
    rdq, rdk, rdv, rout, rlse = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
    tl.compare("out", tl.host(out), rout)
    tl.compare("lse", tl.host(lse), rlse, tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    tl.compare("dq", tl.host(grads[0]), rdq)
    tl.compare("dk", tl.host(grads[1]), rdk)
    tl.compare("dv", tl.host(grads[2]), rdv)
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


# (B, heads, T, H, W, k, mode, G); D = 128
CASES8 = [
    (1, 2, 3, 20, 24, 4, O.SINGLE, 2),          # equal scopes, two ranks
    (1, 2, 3, 7, 9, 4, O.GROUP, 3),             # unequal scopes with a partial group, three ranks
]


@pytest.mark.parametrize("recipe", ["int8", "e4m3"])
@pytest.mark.parametrize("case", CASES8, ids=lambda c: f"{c[2]}x{c[3]}x{c[4]}_k{c[5]}_G{c[7]}")
def test_8bit_scope_shards_equal_the_full_call(env, case, recipe):
    """The 8-bit forwards' scope subsets: each shard writes exactly its scopes'
    rows, and the union equals the full call bit for bit (every scope's codes,
    scales and products are the full call's; v's scales span all tokens either
    way)."""
    import torch
    skp, dev = env
    B, heads, T, H, W, k, mode, G = case
    D, N = 128, T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D)
    q, kk, v = (tl.to_device(ins[n], dev) for n in ("q", "k", "v"))
    full = skp.skiparse_attn_fwd_mixed8 if recipe == "int8" else skp.skiparse_attn_fwd_fp8
    part = skp.skiparse_attn_fwd_mixed8_scopes if recipe == "int8" else skp.skiparse_attn_fwd_fp8_scopes
    ref_out = torch.empty((B, N, heads, D), dtype=torch.bfloat16, device=dev)
    ref_lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
    full(q, kk, v, ref_out, ref_lse, T, H, W, k, mode)
    out = torch.empty_like(ref_out)
    out.view(torch.int16).fill_(tl.SENTINEL)
    lse = torch.full((B, heads, N), float("nan"), dtype=torch.float32, device=dev)
    scope_of, _ = O.index_maps(N, k, mode)
    done = np.zeros(N, dtype=bool)
    for rank in range(G):
        first, step = skp.scope_shard(k, G, rank)
        part(q, kk, v, out, lse, T, H, W, k, mode, first, step)
        torch.cuda.synchronize()
        done |= (scope_of % step) == first
        written = (out.view(torch.int16) != tl.SENTINEL).any(dim=3).any(dim=2).any(dim=0).cpu().numpy()
        assert np.array_equal(written, done), f"rank {rank}: wrote other scopes' rows"
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)
