"""GPU parity of the Q/K/V projection with the RoPE epilogue (skiparse_qkv_rope)
through the C ABI against the float64 oracle (oracle/skiparse_proj_oracle.py).

Bar: every output is the exact value rounded to bf16 once, after fp32
accumulation, so |gpu - ref| <= 2^-8 |ref| (half a bf16 ulp is at most 2^-8 of
the value) plus fp32 arithmetic error, bounded here by 1e-4 of the outputs'
RMS (fp32 sums of C <= 3072 products of order 1/sqrt(C) err by ~1e-6)."""
import numpy as np
import pytest

from oracle import skiparse_proj_oracle as P
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


def _inputs(B, N, C, heads, D, with_bias):
    hd = heads * D
    x = synthetic.normal_bf16_bits(11, (B, N, C))
    w = synthetic.normal_bf16_bits(12, (3 * hd, C), 1.0 / np.sqrt(C))
    b = synthetic.normal_bf16_bits(13, (3 * hd,), 0.1) if with_bias else None
    return x, w, b


def _check(got, ref):
    err = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * rms
    assert np.all(np.isfinite(got))
    assert np.all(err <= bound), (err.max(), np.max(err - bound))
    assert err.mean() <= 2e-3 * rms


def _run(skp, dev, x, w, b, B, N, C, heads, D, T, H, W):
    import torch
    xd, wd = tl.to_device(x, dev), tl.to_device(w, dev)
    bd = tl.to_device(b, dev) if b is not None else None
    bufs = [tl.guarded_empty((B, N, heads, D), torch.bfloat16, dev) for _ in range(3)]
    skp.skiparse_qkv_rope(xd, wd, bd, bufs[0][1], bufs[1][1], bufs[2][1], T, H, W)
    torch.cuda.synchronize()
    for buf, _ in bufs:
        assert tl.guards_intact(buf), "projection wrote outside its outputs"
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)
    return [tl.host(t) for _, t in bufs]


# (B, T, H, W, C, heads, D, bias)
CASES = [
    (1, 4, 8, 8, 128, 2, 64, True),        # heads D = 128: 128-column tiles
    (2, 3, 10, 10, 200, 4, 64, False),     # 600 rows (ragged row tile), C = 200 (ragged channel stage)
    (1, 2, 16, 16, 3072, 2, 128, True),    # long channel loop (48 stages over 4 buffers)
    (3, 1, 5, 7, 64, 6, 128, True),        # T = 1, 105 rows, one stage, 3 heads D / 256 = 9 column tiles
]


def _ids(c):
    return f"B{c[0]}_{c[1]}x{c[2]}x{c[3]}_C{c[4]}_h{c[5]}_D{c[6]}{'_bias' if c[7] else ''}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_qkv_rope_parity(env, case):
    skp, dev = env
    B, T, H, W, C, heads, D, with_bias = case
    N = T * H * W
    x, w, b = _inputs(B, N, C, heads, D, with_bias)
    got = _run(skp, dev, x, w, b, B, N, C, heads, D, T, H, W)
    f = [synthetic.bf16_bits_to_f64(a) if a is not None else None for a in (x, w, b)]
    ref = P.qkv_rope(f[0], f[1], f[2], heads, D, T, H, W)
    for g_, r_ in zip(got, ref):
        _check(g_, r_)


def test_qkv_rope_full_size_sampled_rows(env):
    """The bench's launch configuration (training step sizes: B = 2, 24x22x40,
    C = heads D = 3072): 96 sampled rows against the oracle's row routine."""
    skp, dev = env
    B, T, H, W, heads, D = 2, 24, 22, 40, 24, 128
    N, C = T * H * W, heads * D
    x, w, b = _inputs(B, N, C, heads, D, True)
    got = _run(skp, dev, x, w, b, B, N, C, heads, D, T, H, W)
    rs = np.random.RandomState(5)
    rows = [(int(rs.randint(B)), int(rs.randint(N))) for _ in range(94)] + [(0, 0), (B - 1, N - 1)]
    f = [synthetic.bf16_bits_to_f64(a) for a in (x, w, b)]
    ref = P.qkv_rope_rows(f[0], f[1], f[2], heads, D, T, H, W, rows)
    for g_, r_ in zip(got, ref):
        sel = np.stack([g_[bi, n] for bi, n in rows])
        _check(sel, r_)


def test_qkv_rope_rejects(env):
    import torch
    skp, dev = env
    x = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((3 * 2 * 64, 128), dtype=torch.bfloat16, device=dev)
    q, k, v = (torch.zeros((1, 64, 2, 64), dtype=torch.bfloat16, device=dev) for _ in range(3))
    with pytest.raises(skp.SkiparseError) as e:                 # N != T H W
        skp.skiparse_qkv_rope(x, w, None, q, k, v, 2, 4, 4)
    assert e.value.status == -2
    with pytest.raises(skp.SkiparseError) as e:                 # q and k overlap
        skp.skiparse_qkv_rope(x, w, None, q, q, v, 4, 4, 4)
    assert e.value.status == -9
    x2 = torch.zeros((1, 64, 100), dtype=torch.bfloat16, device=dev)
    w2 = torch.zeros((3 * 2 * 64, 100), dtype=torch.bfloat16, device=dev)
    with pytest.raises(skp.SkiparseError) as e:                 # C % 8 != 0
        skp.skiparse_qkv_rope(x2, w2, None, q, k, v, 4, 4, 4)
    assert e.value.status == -3
    q1, k1, v1 = (torch.zeros((1, 64, 1, 64), dtype=torch.bfloat16, device=dev) for _ in range(3))
    w1 = torch.zeros((3 * 64, 128), dtype=torch.bfloat16, device=dev)
    with pytest.raises(skp.SkiparseError) as e:                 # heads D = 64 is not a multiple of 128
        skp.skiparse_qkv_rope(x, w1, None, q1, k1, v1, 4, 4, 4)
    assert e.value.status == -3


@pytest.mark.parametrize("mode", [0, 1], ids=["single", "group"])
def test_projection_then_attention_without_rotation(env, mode):
    """The listings' order with RoPE fused into the projection: x -> q~, k~, v
    (skiparse_qkv_rope) -> attention with rope_theta = 0 (no second rotation),
    forward and backward, against the oracle on the same bf16 q~, k~, v; and the
    composition against the oracle run from x."""
    import torch
    from oracle import skiparse_oracle as O
    skp, dev = env
    B, T, H, W, C, heads, D, k = 1, 3, 8, 16, 128, 2, 128, 2
    N = T * H * W
    x, w, b = _inputs(B, N, C, heads, D, True)
    xd, wd, bd = tl.to_device(x, dev), tl.to_device(w, dev), tl.to_device(b, dev)
    q, kk, v = (torch.empty((B, N, heads, D), dtype=torch.bfloat16, device=dev) for _ in range(3))
    skp.skiparse_qkv_rope(xd, wd, bd, q, kk, v, T, H, W)
    out = torch.empty_like(q)
    lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
    skp.skiparse_attn_fwd(q, kk, v, out, lse, T, H, W, k, mode, rope_theta=0.0)
    do = tl.to_device(synthetic.normal_bf16_bits(4, (B, N, heads, D)), dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(skp.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode), dtype=torch.uint8,
                     device=dev)
    skp.skiparse_attn_bwd(q, kk, v, out, lse, do, dq, dk, dv, ws, T, H, W, k, mode, rope_theta=0.0)
    torch.cuda.synchronize()
    st, detail = skp.skiparse_device_error()
    assert st == 0, hex(detail)
    qf, kf, vf, dof = (tl.host(t) for t in (q, kk, v, do))
    rout, rlse = O.skiparse_fwd(qf, kf, vf, T, H, W, k, mode, theta=0.0)
    tl.compare("out", tl.host(out), rout)
    tl.compare("lse", tl.host(lse), rlse, tol_max=tl.TOL_LSE, tol_mean=tl.TOL_LSE, tol_rel=1e-3)
    rdq, rdk, rdv = O.skiparse_bwd(qf, kf, vf, dof, T, H, W, k, mode, theta=0.0)[:3]
    tl.compare("dq", tl.host(dq), rdq)
    tl.compare("dk", tl.host(dk), rdk)
    tl.compare("dv", tl.host(dv), rdv)
    # the whole chain from x: the oracle projection (float64) then attention
    f = [synthetic.bf16_bits_to_f64(a) for a in (x, w, b)]
    pq, pk, pv = P.qkv_rope(f[0], f[1], f[2], heads, D, T, H, W)
    cout, _ = O.skiparse_fwd(pq, pk, pv, T, H, W, k, mode, theta=0.0)
    tl.compare("out (from x)", tl.host(out), cout)
    # the saved backward has no rotated copies to read when nothing was rotated
    fws = torch.empty(skp.skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode), dtype=torch.uint8,
                      device=dev)
    with pytest.raises(skp.SkiparseError) as e:
        skp.skiparse_attn_bwd_saved(fws, v, out, lse, do, dq, dk, dv, ws, T, H, W, k, mode, rope_theta=0.0)
    assert e.value.status == -1
