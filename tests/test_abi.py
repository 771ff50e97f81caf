"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/skiparse.h declares, and rejects bad arguments on the host before
touching the device (a valid call on a machine without a GPU reports
SKIPARSE_ERR_DEVICE)."""
import ctypes
import os
import re

import pytest

import sparse_spatiotemporal_attention_gb300 as skp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "skiparse.h")

OK, INVALID, SHAPE, UNSUP, ALIGN, DEVICE, WORKSPACE, LAUNCH, TIMEOUT, ALIAS = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9


@pytest.fixture(scope="module")
def lib():
    from sparse_spatiotemporal_attention_gb300 import _build
    _build.build()
    return skp.load_library()


def _header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(skiparse_[a-z0-9_]+)\s*\(", text)))


def test_header_exports_match(lib):
    names = _header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(skp.EXPORTS)


def test_status_strings(lib):
    for code in (OK, INVALID, SHAPE, UNSUP, ALIGN, DEVICE, WORKSPACE, LAUNCH, TIMEOUT, ALIAS):
        s = skp.status_string(code)
        assert s and s != "unknown status"
    assert skp.status_string(12345) == "unknown status"
    for i in range(len(skp.KERNEL_NAMES)):
        assert lib.skiparse_kernel_name(i).decode() == skp.KERNEL_NAMES[i]
    assert lib.skiparse_kernel_name(len(skp.KERNEL_NAMES)).decode() == "unknown"


A = 1 << 20  # fake, 16-byte-aligned device addresses: validation fails before any use


def _a256(x):
    return (x + 255) // 256 * 256


def fwd_parts(D, slots):
    """Forward workspace past the q / k copies: the split units' partial results,
    O (slots x 256 rows x D fp32) and (m, l) per row, with slots = min(160, the
    call's (unit, K tile) pairs), and the cos/sin table (8192 pairs of fp32)."""
    return _a256(slots * 256 * D * 4) + _a256(slots * 256 * 8) + 8192 * 8


FWD_WS = 2 * 256 * 2 * 64 * 2 + fwd_parts(64, 4)   # B=1, heads=2, N=256, D=64, k=2: 4 units of 1 tile


def fwd(lib, q=A, k=2 * A, v=3 * A, out=4 * A, lse=5 * A, ws=8 * A, ws_bytes=FWD_WS, B=1, heads=2, N=256, D=64,
        T=4, H=8, W=8, sk=2, mode=0, theta=10000.0):
    return lib.skiparse_attn_fwd(q, k, v, out, lse, ws, ws_bytes, B, heads, N, D, T, H, W, sk, mode, theta, None)


def test_fwd_validation(lib):
    assert fwd(lib, mode=2) == INVALID
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, sk=0) == INVALID
    assert fwd(lib, theta=-1.0) == INVALID
    assert fwd(lib, theta=0.0) == DEVICE                 # 0: q, k already rotated; valid, no GPU here
    assert fwd(lib, theta=float("inf")) == INVALID
    assert fwd(lib, N=255) == SHAPE                      # N != T*H*W
    assert fwd(lib, D=96) == UNSUP
    # k (single) or k^2 (group) need not divide N: scopes of unequal length, valid
    # (no GPU here), with the larger scope-ordered workspace
    ragged_ws = lib.skiparse_attn_fwd_workspace_bytes(1, 2, 192, 64, 3, 8, 8, 5, 0)
    assert fwd(lib, T=3, N=192, sk=5, ws_bytes=ragged_ws) == DEVICE
    assert fwd(lib, T=3, N=192, sk=5, ws_bytes=ragged_ws - 1) == WORKSPACE
    # group skip with k^2 > N: 8 scopes of one group each, 24 empty ones
    assert fwd(lib, N=256, sk=32, mode=1, ws_bytes=lib.skiparse_attn_fwd_workspace_bytes(1, 2, 256, 64, 4, 8, 8, 32,
                                                                                         1)) == DEVICE
    assert fwd(lib, T=9, H=6, W=6, N=324, sk=3, mode=1) == UNSUP   # group k must divide 128
    assert fwd(lib, T=2000, H=20, W=20, N=800000) == UNSUP         # RoPE table too large
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, lse=5 * A + 4) == ALIGN
    assert fwd(lib, out=A + 64) == ALIAS                 # out overlaps q
    assert fwd(lib, lse=4 * A + 128) == ALIAS            # lse overlaps out
    assert fwd(lib, ws=None) == WORKSPACE
    assert fwd(lib, ws_bytes=FWD_WS - 1) == WORKSPACE
    assert fwd(lib, ws=8 * A + 16) == ALIGN              # workspace: 256-byte aligned
    assert fwd(lib, ws=3 * A) == ALIAS                   # workspace overlaps v
    # empty calls are valid no-ops, pointers may be NULL
    assert fwd(lib, B=0, q=None, k=None, v=None, out=None, lse=None) == OK
    assert fwd(lib, T=0, N=0) == OK
    # a valid call with no GPU present reaches the device check
    assert fwd(lib) in (DEVICE,)


def test_fwd_workspace_bytes(lib):
    assert lib.skiparse_attn_fwd_workspace_bytes(1, 2, 256, 64, 4, 8, 8, 2, 0) == FWD_WS
    assert lib.skiparse_attn_fwd_workspace_bytes(0, 2, 256, 64, 4, 8, 8, 2, 0) == 0
    assert lib.skiparse_attn_fwd_workspace_bytes(1, 2, 256, 96, 4, 8, 8, 2, 0) == 0
    # each rotated copy is rounded up to 256 bytes: 1 x 1 x 3 tokens x 64 channels
    assert lib.skiparse_attn_fwd_workspace_bytes(1, 1, 3, 64, 1, 1, 3, 1, 0) == 2 * 512 + fwd_parts(64, 1)


def test_bwd_validation_and_workspace(lib):
    ws = lib.skiparse_attn_bwd_workspace_bytes(1, 2, 256, 64, 4, 8, 8, 2, 0)
    elems = 256 * 2 * 64
    assert ws >= elems * 4 + 2 * elems * 2
    assert lib.skiparse_attn_bwd_workspace_bytes(0, 2, 256, 64, 4, 8, 8, 2, 0) == 0
    assert lib.skiparse_attn_bwd_workspace_bytes(1, 2, 256, 96, 4, 8, 8, 2, 0) == 0
    big = lib.skiparse_attn_bwd_workspace_bytes(2, 24, 21120, 128, 24, 22, 40, 4, 1)
    assert big >= 2 * 24 * 21120 * 128 * 8

    def bwd(ws_ptr=10 * A, ws_bytes=ws, dq=7 * A, mode=0):
        return lib.skiparse_attn_bwd(A, 2 * A, 3 * A, 4 * A, 5 * A, 6 * A, dq, 8 * A, 9 * A, ws_ptr, ws_bytes,
                                     1, 2, 256, 64, 4, 8, 8, 2, mode, 10000.0, None)
    assert bwd(ws_ptr=None) == WORKSPACE
    assert bwd(ws_bytes=ws - 1) == WORKSPACE
    assert bwd(ws_ptr=10 * A + 16) == ALIGN
    assert bwd(dq=6 * A) == ALIAS
    assert bwd(ws_ptr=9 * A) == ALIAS
    assert bwd() == DEVICE


def test_bwd_saved_validation(lib):
    """The backward that reuses the forward's rotated q / k validates on the host first."""
    fws = lib.skiparse_attn_fwd_workspace_bytes(1, 2, 256, 64, 4, 8, 8, 2, 0)
    ws = lib.skiparse_attn_bwd_workspace_bytes(1, 2, 256, 64, 4, 8, 8, 2, 0)

    def bwd(fw_ptr=11 * A, fw_bytes=fws, ws_ptr=10 * A, ws_bytes=ws, dq=7 * A, B=1):
        return lib.skiparse_attn_bwd_saved(fw_ptr, fw_bytes, 3 * A, 4 * A, 5 * A, 6 * A, dq, 8 * A, 9 * A, ws_ptr,
                                           ws_bytes, B, 2, 256, 64, 4, 8, 8, 2, 0, 10000.0, None)
    assert bwd(fw_ptr=None) == INVALID
    assert bwd(fw_ptr=11 * A + 16) == ALIGN
    assert bwd(fw_bytes=fws - 1) == WORKSPACE
    assert bwd(ws_ptr=None) == WORKSPACE
    assert bwd(dq=3 * A) == ALIAS
    assert bwd(ws_ptr=11 * A) == ALIAS          # scratch over the forward's rotated q
    assert bwd(B=0, fw_ptr=None) == OK           # empty call
    assert bwd() == DEVICE
    # it needs less scratch than the regular backward (no rotated copies)
    assert bwd(ws_bytes=ws - 2 * 256 * 2 * 64 * 2) == DEVICE


def test_ragged_workspace_sizes(lib):
    """Scopes of unequal length read scope-ordered copies (k, B, Lp, heads, D) of
    q, k, v (forward, both 8-bit forwards too) and of q, k, v, dO (backward)."""
    B, heads, D, N, k = 1, 2, 64, 192, 5                 # single skip: L_0 = 39, Lp = 128
    copy = k * B * 128 * heads * D * 2
    assert lib.skiparse_attn_fwd_workspace_bytes(B, heads, N, D, 3, 8, 8, k, 0) == 3 * copy + fwd_parts(D, 10)
    stats = B * heads * k * 128
    want = stats * D * 4 + 4 * copy + 2 * stats * 4
    got = lib.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, 3, 8, 8, k, 0)
    assert want <= got <= want + 8 * 256 + 16 * 8192
    copy128 = k * 1 * 128 * 2 * 128 * 2                  # B = 1, heads = 2, D = 128
    for fn in ("skiparse_attn_fwd_fp8_workspace_bytes", "skiparse_attn_fwd_mixed8_workspace_bytes"):
        ws8 = getattr(lib, fn)(1, 2, 192, 128, 3, 8, 8, k, 0)
        equal = getattr(lib, fn)(1, 2, 192, 128, 3, 8, 8, 4, 0)   # k = 4 divides 192
        assert ws8 >= 3 * copy128 and equal > 0
    assert lib.skiparse_attn_fwd_fp8(A, 2 * A, 3 * A, 4 * A, 5 * A, 10 * A, 1 << 30, 1, 2, 192, 128, 3, 8, 8, 5, 0,
                                     10000.0, None) == DEVICE


def test_scope_subset_validation(lib):
    """The scope-subset calls validate like the full ones, then their subset."""
    def fwd_s(first, step, N=256, T=4):
        return lib.skiparse_attn_fwd_scopes(A, 2 * A, 3 * A, 4 * A, 5 * A, 8 * A, FWD_WS, 1, 2, N, 64, T, 8, 8, 2, 0,
                                            10000.0, first, step, None)
    assert fwd_s(0, 1) == DEVICE
    assert fwd_s(1, 2) == DEVICE
    assert fwd_s(-1, 2) == INVALID
    assert fwd_s(0, 0) == INVALID
    assert fwd_s(2, 2) == OK                      # no scope >= k: nothing to do
    assert fwd_s(0, 1, N=255) == SHAPE
    ws = lib.skiparse_attn_bwd_workspace_bytes(1, 2, 256, 64, 4, 8, 8, 2, 0)

    def bwd_s(first, step, ws_bytes=ws):
        return lib.skiparse_attn_bwd_scopes(A, 2 * A, 3 * A, 4 * A, 5 * A, 6 * A, 7 * A, 8 * A, 9 * A, 10 * A,
                                            ws_bytes, 1, 2, 256, 64, 4, 8, 8, 2, 0, 10000.0, first, step, None)
    assert bwd_s(0, 2) == DEVICE
    assert bwd_s(0, 0) == INVALID
    assert bwd_s(5, 1) == OK
    assert bwd_s(0, 2, ws_bytes=ws - 1) == WORKSPACE
    for name in ("skiparse_attn_fwd_fp8", "skiparse_attn_fwd_mixed8"):
        ws8 = getattr(lib, name + "_workspace_bytes")(1, 2, 256, 128, 4, 8, 8, 2, 0)
        fn = getattr(lib, name + "_scopes")

        def fwd8_s(first, step, D=128, ws_bytes=ws8):
            return fn(A, 2 * A, 3 * A, 4 * A, 5 * A, 10 * A, ws_bytes, 1, 2, 256, D, 4, 8, 8, 2, 0, 10000.0,
                      first, step, None)
        assert fwd8_s(0, 1) == DEVICE
        assert fwd8_s(1, 2) == DEVICE
        assert fwd8_s(-1, 1) == INVALID
        assert fwd8_s(0, 0) == INVALID
        assert fwd8_s(2, 1) == OK                 # no scope >= k
        assert fwd8_s(0, 1, D=64) == UNSUP
        assert fwd8_s(0, 2, ws_bytes=ws8 - 1) == WORKSPACE


def test_scope_shard_partition():
    """Round-robin shards of the scopes over ranks are disjoint and cover them."""
    for k in (1, 2, 3, 4, 8):
        for world in (1, 2, 3, 4, 8):
            seen = []
            for r in range(world):
                first, step = skp.scope_shard(k, world, r)
                seen += list(range(first, k, step))
            assert sorted(seen) == list(range(k))
    with pytest.raises(ValueError):
        skp.scope_shard(4, 2, 2)


def test_debug_hook_validation(lib):
    assert lib.skiparse_debug_index_map(A, 2 * A, 16, 3, 0, None) == DEVICE     # any N: unequal scopes
    assert lib.skiparse_debug_index_map(A, 2 * A, 16, 2, 2, None) == INVALID
    assert lib.skiparse_debug_index_map(A, A, 16, 2, 0, None) == ALIAS
    assert lib.skiparse_debug_index_map(None, None, 0, 2, 0, None) == OK
    assert lib.skiparse_debug_rope(A, 2 * A, 1, 1, 256, 64, 4, 8, 8, 10000.0, None) == DEVICE
    assert lib.skiparse_debug_rope(A, A + 16, 1, 1, 256, 64, 4, 8, 8, 10000.0, None) == ALIAS


def test_trace_without_gpu(lib):
    skp.skiparse_trace_begin()
    ms, cnt = skp.skiparse_trace_end(len(skp.KERNEL_NAMES))
    assert ms == [0.0] * len(skp.KERNEL_NAMES) and cnt == [0] * len(skp.KERNEL_NAMES)


def test_package_has_no_fallback():
    """The binding must not import the oracle or any CPU path."""
    src = open(os.path.join(ROOT, "sparse_spatiotemporal_attention_gb300", "__init__.py")).read()
    assert "oracle" not in src.replace("fallback", "")
    for f in os.listdir(os.path.join(ROOT, "sparse_spatiotemporal_attention_gb300")):
        if f.endswith(".py"):
            assert "import oracle" not in open(os.path.join(ROOT, "sparse_spatiotemporal_attention_gb300", f)).read()


def test_fwd_fp8_validation(lib):
    """The 8-bit forward validates on the host first (D = 128 only)."""
    ws = lib.skiparse_attn_fwd_fp8_workspace_bytes(1, 2, 256, 128, 4, 8, 8, 2, 0)
    assert ws > 0
    assert lib.skiparse_attn_fwd_fp8_workspace_bytes(1, 2, 256, 64, 4, 8, 8, 2, 0) == 0

    def fwd(ws_ptr=10 * A, ws_bytes=ws, D=128, out=4 * A, theta=10000.0, N=256):
        return lib.skiparse_attn_fwd_fp8(A, 2 * A, 3 * A, out, 5 * A, ws_ptr, ws_bytes, 1, 2, N, D, 4, 8, 8, 2, 0,
                                         theta, None)
    assert fwd(D=64) == UNSUP
    assert fwd(N=255) == SHAPE
    assert fwd(theta=-1.0) == INVALID
    assert fwd(ws_ptr=None) == WORKSPACE
    assert fwd(ws_bytes=ws - 1) == WORKSPACE
    assert fwd(out=A) == ALIAS
    assert fwd() == DEVICE
    assert fwd(theta=0.0) == DEVICE          # 0: q, k already rotated


def test_qkv_rope_validation(lib):
    """The projection validates on the host first: shapes, sizes, alignment, overlaps."""
    def proj(x=A, w=2 * A, bias=3 * A, q=4 * A, k=5 * A, v=6 * A, B=1, N=256, C=128, heads=2, D=64,
             T=4, H=8, W=8, theta=10000.0):
        return lib.skiparse_qkv_rope(x, w, bias, q, k, v, B, N, C, heads, D, T, H, W, theta, None)
    assert proj(N=255) == SHAPE
    assert proj(D=96) == UNSUP
    assert proj(C=100) == UNSUP                 # C % 8
    assert proj(heads=1) == UNSUP               # heads D = 64 not a multiple of 128
    assert proj(theta=-1.0) == INVALID
    assert proj(x=None) == INVALID
    assert proj(q=4 * A + 8) == ALIGN
    assert proj(k=4 * A) == ALIAS               # q and k overlap
    assert proj(q=A) == ALIAS                   # q over x
    assert proj(B=0, x=None) == OK              # empty call
    assert proj(bias=None) == DEVICE            # bias is optional
    assert proj() == DEVICE
    assert proj(theta=0.0) == DEVICE            # 0: no rotation
