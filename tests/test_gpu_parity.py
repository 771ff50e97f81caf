"""GPU parity through the C ABI against the float64 oracle (small and medium
shapes the oracle finishes in seconds). Each case spans one or more 128-row
tiles; several have a ragged last tile (L not a multiple of 128) or a scope
shorter than one tile.

Bars: index maps bit-exact; RoPE fp32 max-abs 1e-5; out, dq, dk, dv (bf16)
max-abs 2e-2, mean-abs 2e-3 and relative RMS 1e-2; LSE max-abs 1e-2.
"""
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


# (B, heads, D, T, H, W, k, mode)
CASES = [
    (1, 2, 64, 4, 8, 8, 2, O.SINGLE),        # the tiny correctness config, single skip
    (1, 2, 64, 4, 8, 8, 2, O.GROUP),         # the tiny correctness config, group skip
    (1, 2, 128, 3, 10, 10, 2, O.SINGLE),     # L = 150: two tiles, ragged tail of 22
    (1, 2, 128, 3, 10, 10, 2, O.GROUP),
    (2, 3, 64, 2, 8, 12, 2, O.SINGLE),       # B > 1, L = 96 < one tile
    (2, 2, 128, 2, 12, 20, 4, O.GROUP),      # B > 1, L = 120, merged batch rows in the tail
    (1, 2, 128, 1, 16, 24, 4, O.GROUP),      # T = 1 (an image), L = 96
    (1, 2, 128, 2, 8, 16, 1, O.SINGLE),      # k = 1: dense attention, L = 256
    (1, 1, 128, 2, 8, 16, 1, O.GROUP),
    (1, 2, 128, 4, 16, 16, 2, O.GROUP),      # L = 512: four full tiles
    (1, 1, 128, 2, 16, 32, 8, O.GROUP),      # k = 8
    (1, 2, 64, 3, 6, 8, 3, O.SINGLE),        # k = 3 (single skip takes any k), L = 48
    (1, 2, 128, 5, 9, 14, 5, O.SINGLE),      # k = 5, L = 126
    (2, 2, 128, 3, 20, 24, 4, O.SINGLE),     # L = 360: 3 tiles, tail 104, B = 2
    (1, 1, 128, 8, 32, 32, 4, O.SINGLE),     # the 8x32x32 grid with one head, L = 2048
]


def _ids(c):
    B, h, D, T, H, W, k, m = c
    return f"B{B}h{h}D{D}_{T}x{H}x{W}_k{k}_{'single' if m == O.SINGLE else 'group'}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_forward_parity(env, case):
    skp, dev = env
    B, heads, D, T, H, W, k, mode = case
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode)
    f = tl.f64_inputs(ins)
    rout, rlse = O.skiparse_fwd(f["q"], f["k"], f["v"], T, H, W, k, mode)
    tl.compare("out", tl.host(fw["out"]), rout)
    tl.compare("lse", tl.host(fw["lse"]), rlse, tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


# every case up to the 8x32x32 grid (one head, L = 2048: 16 query and 16 key tiles per scope)
BWD_CASES = [c for c in CASES if c[3] * c[4] * c[5] <= 8192]


@pytest.mark.parametrize("case", BWD_CASES, ids=_ids)
def test_backward_parity(env, case):
    skp, dev = env
    B, heads, D, T, H, W, k, mode = case
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode)
    bw = tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode)
    f = tl.f64_inputs(ins)
    rdq, rdk, rdv, rout, rlse = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
    tl.compare("out", tl.host(fw["out"]), rout)
    tl.compare("dv", tl.host(bw["dv"]), rdv)
    tl.compare("dk", tl.host(bw["dk"]), rdk)
    tl.compare("dq", tl.host(bw["dq"]), rdq)
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


# N that k (single) or k^2 (group) does not divide: scopes of unequal length,
# read from scope-ordered copies. Each case names its scope lengths.
RAGGED_CASES = [
    (1, 2, 128, 4, 8, 9, 5, O.SINGLE),       # N = 288: scopes 58, 58, 58, 57, 57
    (2, 2, 128, 5, 5, 41, 4, O.SINGLE),      # N = 1025: 257 (3 tiles), 256 x 3 (2 tiles), B = 2
    (1, 2, 64, 3, 10, 11, 4, O.SINGLE),      # D = 64, N = 330: 83, 83, 82, 82
    (1, 2, 128, 1, 27, 19, 4, O.GROUP),      # N = 513: 129 (2 tiles: a one-token group), 128 x 3
    (2, 2, 128, 3, 7, 9, 4, O.GROUP),        # N = 189: 48, 48, 48, 45 (a partial group), B = 2
    (1, 3, 64, 5, 5, 5, 2, O.GROUP),         # D = 64, N = 125: 63, 62 (the last group holds one token)
    (1, 2, 128, 1, 8, 9, 8, O.GROUP),        # N = 72 < k^2 = 64 + 8: nine groups, scope 0 two (16), the rest one
    (1, 2, 64, 1, 2, 5, 4, O.GROUP),         # N = 10: scopes 4, 4, 2 and an empty one
    (2, 2, 128, 1, 1, 3, 4, O.SINGLE),       # N = 3 < k: one token per scope, scope 3 empty
]


@pytest.mark.parametrize("case", RAGGED_CASES, ids=_ids)
def test_ragged_forward_backward_parity(env, case):
    skp, dev = env
    B, heads, D, T, H, W, k, mode = case
    N = T * H * W
    assert not O.divisible(N, k, mode)
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode)
    bw = tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode)
    f = tl.f64_inputs(ins)
    rdq, rdk, rdv, rout, rlse = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
    tl.compare("out", tl.host(fw["out"]), rout)
    # with one-token scopes the LSE is the bare logit q~ . k~ / sqrt(D), whose bf16
    # operands carry a relative error up to 2^-8: no log L term dilutes it
    lens = [len(O.prose_scope_tokens(N, k, mode, s)) for s in range(k)]
    lse_rel = 2.0 ** -8 if min(n for n in lens if n) == 1 else 1e-3
    tl.compare("lse", tl.host(fw["lse"]), rlse, tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE, tol_rel=lse_rel)
    tl.compare("dv", tl.host(bw["dv"]), rdv)
    tl.compare("dk", tl.host(bw["dk"]), rdk)
    tl.compare("dq", tl.host(bw["dq"]), rdq)
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


SAVED_CASES = [(1, 2, 128, 3, 10, 10, 2, O.GROUP), (2, 3, 64, 2, 8, 12, 2, O.SINGLE), (2, 2, 128, 3, 20, 24, 4, O.SINGLE),
               (2, 2, 128, 3, 7, 9, 4, O.GROUP), (1, 2, 64, 3, 10, 11, 4, O.SINGLE)]


@pytest.mark.parametrize("case", SAVED_CASES, ids=_ids)
def test_backward_saved_bitwise_and_parity(env, case):
    """The backward that reuses the forward's rotated q / k gives the regular
    backward's dk and dv bit for bit (the same kernels read bitwise-equal
    rotated copies) and its dq up to the order of dq's fp32 accumulation: the
    key tiles' bulk reduce-adds into the accumulator land in an order set by
    timing, so the fp32 sums may differ in their last bits and a dq element by
    one bf16 step after rounding. Both match the oracle."""
    import torch
    skp, dev = env
    B, heads, D, T, H, W, k, mode = case
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True)
    q, kk, v, do = (tl.to_device(ins[n], dev) for n in ("q", "k", "v", "do"))
    out = torch.empty((B, N, heads, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
    fws = torch.empty(skp.skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode), dtype=torch.uint8,
                      device=dev)
    skp.skiparse_attn_fwd(q, kk, v, out, lse, T, H, W, k, mode, workspace=fws)
    nbytes = skp.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    g1 = [torch.empty_like(q) for _ in range(3)]
    g2 = [torch.full_like(q, float("nan")) for _ in range(3)]
    skp.skiparse_attn_bwd(q, kk, v, out, lse, do, *g1, ws, T, H, W, k, mode)
    skp.skiparse_attn_bwd_saved(fws, v, out, lse, do, *g2, ws, T, H, W, k, mode)
    torch.cuda.synchronize()
    for name, a, b in zip(("dk", "dv"), g1[1:], g2[1:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
    d1, d2 = tl.host(g1[0]), tl.host(g2[0])
    diff = np.abs(d1 - d2)
    worst = np.unravel_index(np.argmax(diff), diff.shape)
    msg = f"dq: {np.count_nonzero(diff)} elements differ, worst {diff[worst]:.3e} at {d1[worst]:.3e} / {d2[worst]:.3e}"
    print(msg)
    # one bf16 step is at most 2^-7 of the value (at the bottom of a binade)
    assert np.all(diff <= 2.0 ** -7 * np.maximum(np.abs(d1), np.abs(d2)) + 1e-7), msg
    f = tl.f64_inputs(ins)
    rdq, rdk, rdv, _, _ = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
    tl.compare("dq", tl.host(g2[0]), rdq)
    tl.compare("dk", tl.host(g2[1]), rdk)
    tl.compare("dv", tl.host(g2[2]), rdv)
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)


@pytest.mark.parametrize("case", [(1, 2, 128, 3, 10, 10, 2, O.GROUP), (1, 2, 64, 3, 10, 11, 4, O.SINGLE)],
                         ids=_ids)
def test_outputs_off_a_32_byte_boundary(env, case):
    """out, dq, dk and dv placed 16 bytes past a 32-byte boundary (the least
    alignment the library accepts) take the kernels' 16-byte store path; the
    results equal those of 32-byte-aligned outputs (32-byte stores): out, lse,
    dk and dv bit for bit, dq up to the order of its fp32 accumulation."""
    import torch
    skp, dev = env
    B, heads, D, T, H, W, k, mode = case
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True)
    fa = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode)
    fb = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode, pad=4104)
    assert fa["out"].data_ptr() % 32 == 0 and fb["out"].data_ptr() % 32 == 16
    assert torch.equal(fa["out"].view(torch.int16), fb["out"].view(torch.int16))
    assert torch.equal(fa["lse"], fb["lse"])
    ba = tl.run_bwd(skp, dev, ins, fa, B, heads, N, D, T, H, W, k, mode)
    bb = tl.run_bwd(skp, dev, ins, fb, B, heads, N, D, T, H, W, k, mode, pad=4104)
    assert bb["dq"].data_ptr() % 32 == 16
    for name in ("dk", "dv"):
        assert torch.equal(ba[name].view(torch.int16), bb[name].view(torch.int16)), name
    d1, d2 = tl.host(ba["dq"]), tl.host(bb["dq"])
    assert np.all(np.abs(d1 - d2) <= 2.0 ** -7 * np.maximum(np.abs(d1), np.abs(d2)) + 1e-7)
    f = tl.f64_inputs(ins)
    rdq, rdk, rdv, rout, _ = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
    tl.compare("out", tl.host(fb["out"]), rout)
    tl.compare("dq", d2, rdq)
    tl.compare("dk", tl.host(bb["dk"]), rdk)
    tl.compare("dv", tl.host(bb["dv"]), rdv)


def test_peaky_softmax_rescale(env):
    """q scaled by 4 makes row maxima jump between key tiles, exercising the
    online-softmax rescale of O. Not a contract workload; its bound is derived
    from the operands' bf16 rounding instead. The rotated q~ and k~ are MMA
    operands in bf16: each element carries a relative rounding error of
    standard deviation 2^-8 / sqrt(12), so a logit q~.k~ / sqrt(D) moves by
    about sigma = 2^-8 / sqrt(12) * sqrt(2 sum_d q~_d^2 k~_d^2) / sqrt(D), here
    (|q~_d| ~ 4, |k~_d| ~ 1) about 0.0064. A softmax row split between keys
    moves its output by at most (e^(2 d) - 1) |v_j - O| for logit shifts d;
    with d = 5 sigma and |v_j - O| up to 2 max|v|, that is about 0.5 % of
    max|v|, and the gradients, formed from the same P, carry the same relative
    error. The bound, 2^-5 max|ref| per element (with relative RMS 1e-2),
    leaves a factor of about six over that estimate."""
    skp, dev = env
    B, heads, D, T, H, W, k, mode = 1, 2, 128, 4, 16, 16, 2, O.SINGLE
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True, q_scale=4.0)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode)
    bw = tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode)
    f = tl.f64_inputs(ins)
    rdq, rdk, rdv, rout, rlse = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
    tl.compare("lse", tl.host(fw["lse"]), rlse, tol_max=tl.TOL_LSE * 4, tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    for name, got, ref in (("out", fw["out"], rout), ("dv", bw["dv"], rdv), ("dk", bw["dk"], rdk),
                           ("dq", bw["dq"], rdq)):
        m = np.abs(ref).max()
        tl.compare(name, tl.host(got), ref, tol_max=m / 32, tol_mean=m / 256, tol_rel=1e-2)


@pytest.mark.parametrize("mode", [O.SINGLE, O.GROUP])
@pytest.mark.parametrize("N,k", [(256, 2), (4096, 4), (21120, 4), (57600, 4), (1024, 8), (300, 3), (512, 1),
                                 (1025, 4), (513, 4), (189, 4), (21525, 4), (77, 8), (7, 5)])
def test_index_map_bit_exact(env, mode, N, k):
    """Any N (scopes of unequal length where k or k^2 does not divide it)."""
    import torch
    skp, dev = env
    scope = torch.full((N,), -7, dtype=torch.int32, device=dev)
    pos = torch.full((N,), -7, dtype=torch.int32, device=dev)
    if mode == O.GROUP and 128 % k != 0:
        # a 128-row tile must hold whole groups: refused, nothing written
        with pytest.raises(skp.SkiparseError) as e:
            skp.skiparse_debug_index_map(scope, pos, N, k, mode)
        assert e.value.status == -3
        torch.cuda.synchronize()
        assert bool((scope == -7).all()) and bool((pos == -7).all())
        return
    skp.skiparse_debug_index_map(scope, pos, N, k, mode)
    torch.cuda.synchronize()
    rs, rp = O.index_maps(N, k, mode)
    assert np.array_equal(scope.cpu().numpy(), rs)
    assert np.array_equal(pos.cpu().numpy(), rp)


@pytest.mark.parametrize("D,grid", [(64, (4, 8, 8)), (128, (24, 22, 40)), (128, (16, 45, 80)), (128, (1, 3, 5))])
def test_rope_fp32(env, D, grid):
    import torch
    skp, dev = env
    T, H, W = grid
    N = T * H * W
    heads = 2
    x = synthetic.normal_bf16_bits(7, (1, N, heads, D))
    xd = tl.to_device(x, dev)
    out = torch.empty((1, N, heads, D), dtype=torch.float32, device=dev)
    skp.skiparse_debug_rope(xd, out, T, H, W, 10000.0)
    torch.cuda.synchronize()
    ref = O.apply_rope(synthetic.bf16_bits_to_f64(x), T, H, W, 10000.0)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref).max()
    assert err <= tl.TOL_ROPE, err


def test_trace_counts_launches(env):
    skp, dev = env
    B, heads, D, T, H, W, k, mode = 1, 2, 64, 4, 8, 8, 2, O.GROUP
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True)
    skp.skiparse_trace_begin()
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode, guard=False)
    tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode, guard=False)
    ms, cnt = skp.skiparse_trace_end(len(skp.KERNEL_NAMES))
    assert cnt[:5] == [1, 1, 1, 1, 1]
    assert all(c == 0 for c in cnt[5:])               # the 8-bit forwards and the projection did not run
    assert all(m > 0 for m in ms[:5]) and all(m == 0 for m in ms[5:])


def test_empty_and_invalid_calls_on_device(env):
    import torch
    skp, dev = env
    q = torch.zeros((1, 256, 2, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 2, 256), dtype=torch.float32, device=dev)
    out = torch.zeros_like(q)
    with pytest.raises(skp.SkiparseError) as e:
        skp.skiparse_attn_fwd(q, q, q, out, lse, 4, 8, 7, 2, 0)      # N != T*H*W
    assert e.value.status == -2
    with pytest.raises(skp.SkiparseError) as e:
        skp.skiparse_attn_fwd(q, q, q, q, lse, 4, 8, 8, 2, 0)        # out aliases q
    assert e.value.status == -9
    small = torch.empty(1024, dtype=torch.uint8, device=dev)
    with pytest.raises(skp.SkiparseError) as e:
        skp.skiparse_attn_fwd(q, q, q, out, lse, 4, 8, 8, 2, 0, workspace=small)   # workspace too small
    assert e.value.status == -6
    empty = torch.zeros((0, 256, 2, 64), dtype=torch.bfloat16, device=dev)
    skp.skiparse_attn_fwd(empty, empty, empty, empty, lse, 4, 8, 8, 2, 0)
    assert out.abs().sum().item() == 0


def test_bounded_wait_times_out_and_context_survives(env):
    """A wait on an mbarrier that nothing arrives at gives up after about one
    second, records its code in the device error word and lets the kernel exit;
    the context then still runs an attention call to parity."""
    import time
    import torch
    skp, dev = env
    assert skp.skiparse_device_error() == (0, 0)
    with pytest.raises(skp.SkiparseError):
        skp.skiparse_debug_wait_timeout(0)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    skp.skiparse_debug_wait_timeout(0x7e01)
    st, detail = skp.skiparse_device_error()
    elapsed = time.perf_counter() - t0
    assert st == -8 and detail == 0x7e01
    assert 0.9 < elapsed < 10.0
    assert skp.skiparse_device_error() == (0, 0)        # reading clears the word
    B, heads, D, T, H, W, k, mode = 1, 2, 64, 4, 8, 8, 2, O.GROUP
    N = T * H * W
    ins = synthetic.attention_inputs(B, N, heads, D)
    fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode)
    f = tl.f64_inputs(ins)
    rout, _ = O.skiparse_fwd(f["q"], f["k"], f["v"], T, H, W, k, mode)
    tl.compare("out", tl.host(fw["out"]), rout)
    assert skp.skiparse_device_error() == (0, 0)
