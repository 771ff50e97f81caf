"""The allocation-free backward entry point, skiparse_attn_bwd_noalloc.

It serves callers that cannot allocate device memory when they run the
backward; its scratch is a fixed array inside the library. This checks, through
the C ABI, that two calls in a row (different shapes, so the second call finds
the first one's leftovers in the shared array) give the same gradients as the
regular entry point with a caller-provided workspace and as the float64
oracle, within the parity tolerances used everywhere else, and that sizes
needing more scratch than the array holds are refused before anything runs.

The file is named to be collected last, so a run that stops at the first
failure has run every other test before this one.
"""
import pytest

from oracle import skiparse_oracle as O
from sparse_spatiotemporal_attention_gb300 import synthetic
import skiparse_testlib as tl

pytestmark = pytest.mark.gpu


def test_noalloc_backward_matches_workspace_backward_twice():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import sparse_spatiotemporal_attention_gb300 as skp
    lib = skp.load_library()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(1, 2, 64, 4, 8, 8, 2, O.GROUP), (2, 2, 128, 3, 10, 10, 2, O.SINGLE)]
    for call, (B, heads, D, T, H, W, k, mode) in enumerate(cases):
        N = T * H * W
        need = skp.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode)
        assert 0 < need <= skp.NOALLOC_SCRATCH_BYTES
        ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True, seeds={"q": 11 + call})
        fw = tl.run_fwd(skp, dev, ins, B, heads, N, D, T, H, W, k, mode, guard=False)
        ref = tl.run_bwd(skp, dev, ins, fw, B, heads, N, D, T, H, W, k, mode, guard=False)
        dq, dk, dv = (torch.full_like(fw["out"], float("nan")) for _ in range(3))
        st = lib.skiparse_attn_bwd_noalloc(fw["q"].data_ptr(), fw["k"].data_ptr(), fw["v"].data_ptr(),
                                           fw["out"].data_ptr(), fw["lse"].data_ptr(), ref["do"].data_ptr(),
                                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                           B, heads, N, D, T, H, W, k, mode, 10000.0, stream)
        assert st == 0, skp.status_string(st)
        torch.cuda.synchronize()
        f = tl.f64_inputs(ins)
        rdq, rdk, rdv, _, _ = O.skiparse_bwd(f["q"], f["k"], f["v"], f["do"], T, H, W, k, mode)
        for name, got, want in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
            tl.compare(f"call {call} {name}", tl.host(got), tl.host(ref[name]))
            tl.compare(f"call {call} {name} vs oracle", tl.host(got), want)
        st, detail = skp.skiparse_device_error()
        assert st == 0, hex(detail)

    # sizes beyond the array are refused with SKIPARSE_ERR_WORKSPACE, nothing launched
    B, heads, D, T, H, W, k = 2, 24, 128, 24, 22, 40, 4
    N = T * H * W
    assert skp.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, k, O.GROUP) > skp.NOALLOC_SCRATCH_BYTES
    A = 1 << 20
    st = lib.skiparse_attn_bwd_noalloc(A, 2 * A, 3 * A, 4 * A, 5 * A, 6 * A, 7 * A, 8 * A, 9 * A,
                                       B, heads, N, D, T, H, W, k, O.GROUP, 10000.0, stream)
    assert st == -6
