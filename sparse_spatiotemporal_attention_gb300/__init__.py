"""GB300-native Skiparse attention (Open-Sora Plan), Python binding.

The library is `_lib/libskiparse.so`, a C ABI declared in include/skiparse.h
and built for sm_103a by `_build.build()`. This module only marshals arguments
(torch tensors -> device pointers, sizes, the current stream) and turns status
codes into exceptions: every step of the attention runs in the library's CUDA
kernels. If the library is missing, every call raises; there is no fallback.

Tensor layouts: q, k, v, out, dout, dq, dk, dv are bf16 (B, N, heads, D)
contiguous on the GPU; lse is fp32 (B, heads, N).
"""
from __future__ import annotations

import ctypes
import os

SINGLE = 0
GROUP = 1
KERNEL_NAMES = ("skiparse_fwd_kernel", "skiparse_bwd_pre_kernel", "skiparse_bwd_main_kernel",
                "skiparse_bwd_post_kernel", "skiparse_fwd_rope_kernel", "skiparse_fwd8_vmax_kernel",
                "skiparse_fwd8_prep_kernel", "skiparse_fwd8_kernel", "skiparse_qkv_rope_kernel",
                "skiparse_fwdm8_prep_kernel", "skiparse_fwdm8_kernel", "skiparse_fwd_merge_kernel")

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libskiparse.so")

EXPORTS = (
    "skiparse_attn_fwd_workspace_bytes", "skiparse_attn_fwd", "skiparse_attn_bwd_workspace_bytes", "skiparse_attn_bwd",
    "skiparse_debug_index_map", "skiparse_debug_rope", "skiparse_status_string",
    "skiparse_device_error", "skiparse_trace_begin", "skiparse_trace_end", "skiparse_kernel_name",
    "skiparse_attn_bwd_noalloc", "skiparse_debug_wait_timeout", "skiparse_attn_bwd_saved",
    "skiparse_attn_fwd_fp8_workspace_bytes", "skiparse_attn_fwd_fp8",
    "skiparse_attn_fwd_mixed8_workspace_bytes", "skiparse_attn_fwd_mixed8",
    "skiparse_attn_fwd_scopes", "skiparse_attn_bwd_scopes",
    "skiparse_attn_fwd_fp8_scopes", "skiparse_attn_fwd_mixed8_scopes",
    "skiparse_qkv_rope",
)


class SkiparseError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


_lib = None

_c_int, _c_size, _c_float, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libskiparse.so once. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libskiparse.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    sig = {
        "skiparse_attn_fwd_workspace_bytes": (_c_size, [_c_int] * 9),
        "skiparse_attn_fwd": (_c_int, [_vp] * 6 + [_c_size] + [_c_int] * 9 + [_c_float, _vp]),
        "skiparse_attn_bwd_workspace_bytes": (_c_size, [_c_int] * 9),
        "skiparse_attn_bwd": (_c_int, [_vp] * 10 + [_c_size] + [_c_int] * 9 + [_c_float, _vp]),
        "skiparse_debug_index_map": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp]),
        "skiparse_debug_rope": (_c_int, [_vp, _vp] + [_c_int] * 7 + [_c_float, _vp]),
        "skiparse_status_string": (ctypes.c_char_p, [_c_int]),
        "skiparse_device_error": (_c_int, [ctypes.POINTER(_c_int)]),
        "skiparse_trace_begin": (_c_int, []),
        "skiparse_trace_end": (_c_int, [ctypes.POINTER(_c_float), ctypes.POINTER(_c_int), _c_int]),
        "skiparse_kernel_name": (ctypes.c_char_p, [_c_int]),
        "skiparse_attn_bwd_noalloc": (_c_int, [_vp] * 9 + [_c_int] * 9 + [_c_float, _vp]),
        "skiparse_debug_wait_timeout": (_c_int, [_c_int, _vp]),
        "skiparse_qkv_rope": (_c_int, [_vp] * 6 + [_c_int] * 8 + [_c_float, _vp]),
        "skiparse_attn_fwd_fp8_workspace_bytes": (_c_size, [_c_int] * 9),
        "skiparse_attn_fwd_fp8": (_c_int, [_vp] * 6 + [_c_size] + [_c_int] * 9 + [_c_float, _vp]),
        "skiparse_attn_fwd_mixed8_workspace_bytes": (_c_size, [_c_int] * 9),
        "skiparse_attn_fwd_scopes": (_c_int, [_vp] * 6 + [_c_size] + [_c_int] * 9 + [_c_float, _c_int, _c_int, _vp]),
        "skiparse_attn_fwd_fp8_scopes": (_c_int, [_vp] * 6 + [_c_size] + [_c_int] * 9 + [_c_float, _c_int, _c_int, _vp]),
        "skiparse_attn_fwd_mixed8_scopes": (_c_int,
                                            [_vp] * 6 + [_c_size] + [_c_int] * 9 + [_c_float, _c_int, _c_int, _vp]),
        "skiparse_attn_bwd_scopes": (_c_int, [_vp] * 10 + [_c_size] + [_c_int] * 9 + [_c_float, _c_int, _c_int, _vp]),
        "skiparse_attn_fwd_mixed8": (_c_int, [_vp] * 6 + [_c_size] + [_c_int] * 9 + [_c_float, _vp]),
        "skiparse_attn_bwd_saved": (_c_int, [_vp, _c_size] + [_vp] * 8 + [_c_size] + [_c_int] * 9 + [_c_float, _vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().skiparse_status_string(int(status)).decode()


skiparse_status_string = status_string


def _check(status: int, what: str):
    if status != 0:
        raise SkiparseError(status, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _shape(q):
    B, N, heads, D = q.shape
    return int(B), int(heads), int(N), int(D)


def skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode) -> int:
    return int(load_library().skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode))


def skiparse_attn_fwd(q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta=10000.0, stream=None,
                      workspace=None, workspace_bytes=None):
    """Forward pass into caller-allocated out (bf16, like q) and lse (fp32 (B, heads, N)).
    `workspace` is a device buffer of at least skiparse_attn_fwd_workspace_bytes(...)
    bytes; when None, one is taken from torch's caching allocator for this call."""
    B, heads, N, D = _shape(q)
    if workspace is None:
        import torch
        nbytes = skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = load_library().skiparse_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                          _ptr(workspace), int(workspace_bytes),
                                          B, heads, N, D, T, H, W, sparse_k, mode,
                                          float(rope_theta), _stream(stream))
    _check(st, "skiparse_attn_fwd")


def skiparse_attn_fwd_fp8_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode) -> int:
    return int(load_library().skiparse_attn_fwd_fp8_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode))


def skiparse_attn_fwd_mixed8_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode) -> int:
    return int(load_library().skiparse_attn_fwd_mixed8_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode))


def _fwd8(name, q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta, stream, workspace, workspace_bytes,
          subset=None):
    lib = load_library()
    B, heads, N, D = _shape(q)
    if workspace is None:
        import torch
        nbytes = getattr(lib, name + "_workspace_bytes")(B, heads, N, D, T, H, W, sparse_k, mode)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
            B, heads, N, D, T, H, W, sparse_k, mode, float(rope_theta)]
    call = name
    if subset is not None:
        call = name + "_scopes"
        args += [int(subset[0]), int(subset[1])]
    st = getattr(lib, call)(*args, _stream(stream))
    _check(st, call)


def skiparse_attn_fwd_fp8(q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta=10000.0, stream=None,
                          workspace=None, workspace_bytes=None):
    """8-bit forward pass with E4M3 q, k, v and P (D = 128) into caller-allocated
    out and lse; `workspace` as for skiparse_attn_fwd, sized by
    skiparse_attn_fwd_fp8_workspace_bytes(...)."""
    _fwd8("skiparse_attn_fwd_fp8", q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta, stream, workspace,
          workspace_bytes)


def skiparse_attn_fwd_mixed8(q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta=10000.0, stream=None,
                             workspace=None, workspace_bytes=None):
    """8-bit forward pass with INT8 q, k for S and E4M3 P, v for P V (D = 128);
    `workspace` sized by skiparse_attn_fwd_mixed8_workspace_bytes(...)."""
    _fwd8("skiparse_attn_fwd_mixed8", q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta, stream, workspace,
          workspace_bytes)


def skiparse_attn_fwd_fp8_scopes(q, k, v, out, lse, T, H, W, sparse_k, mode, scope_first, scope_step,
                                 rope_theta=10000.0, stream=None, workspace=None, workspace_bytes=None):
    """skiparse_attn_fwd_fp8 over the scopes scope_first, scope_first +
    scope_step, ... only; the other rows of out and lse are left untouched."""
    _fwd8("skiparse_attn_fwd_fp8", q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta, stream, workspace,
          workspace_bytes, subset=(scope_first, scope_step))


def skiparse_attn_fwd_mixed8_scopes(q, k, v, out, lse, T, H, W, sparse_k, mode, scope_first, scope_step,
                                    rope_theta=10000.0, stream=None, workspace=None, workspace_bytes=None):
    """skiparse_attn_fwd_mixed8 over the scopes scope_first, scope_first +
    scope_step, ... only; the other rows of out and lse are left untouched."""
    _fwd8("skiparse_attn_fwd_mixed8", q, k, v, out, lse, T, H, W, sparse_k, mode, rope_theta, stream, workspace,
          workspace_bytes, subset=(scope_first, scope_step))


def skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode) -> int:
    return int(load_library().skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode))


def skiparse_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, workspace, T, H, W, sparse_k, mode,
                      rope_theta=10000.0, stream=None, workspace_bytes=None):
    """Backward pass into caller-allocated dq, dk, dv; `workspace` is a device
    buffer of at least skiparse_attn_bwd_workspace_bytes(...) bytes."""
    B, heads, N, D = _shape(q)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = load_library().skiparse_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                          _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes),
                                          B, heads, N, D, T, H, W, sparse_k, mode,
                                          float(rope_theta), _stream(stream))
    _check(st, "skiparse_attn_bwd")


def skiparse_attn_fwd_scopes(q, k, v, out, lse, T, H, W, sparse_k, mode, scope_first, scope_step,
                             rope_theta=10000.0, stream=None, workspace=None, workspace_bytes=None):
    """Forward over the scopes scope_first, scope_first + scope_step, ... only;
    the other rows of out and lse are left untouched."""
    B, heads, N, D = _shape(q)
    if workspace is None:
        import torch
        nbytes = skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = load_library().skiparse_attn_fwd_scopes(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace),
                                                 int(workspace_bytes), B, heads, N, D, T, H, W, sparse_k, mode,
                                                 float(rope_theta), int(scope_first), int(scope_step),
                                                 _stream(stream))
    _check(st, "skiparse_attn_fwd_scopes")


def skiparse_attn_bwd_scopes(q, k, v, out, lse, dout, dq, dk, dv, workspace, T, H, W, sparse_k, mode, scope_first,
                             scope_step, rope_theta=10000.0, stream=None, workspace_bytes=None):
    """Backward over the scopes scope_first, scope_first + scope_step, ... only;
    the other rows of dq, dk and dv are left untouched."""
    B, heads, N, D = _shape(q)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = load_library().skiparse_attn_bwd_scopes(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                                 _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes),
                                                 B, heads, N, D, T, H, W, sparse_k, mode, float(rope_theta),
                                                 int(scope_first), int(scope_step), _stream(stream))
    _check(st, "skiparse_attn_bwd_scopes")


def scope_shard(sparse_k, world, rank):
    """(scope_first, scope_step) of one rank when `world` ranks split the scopes
    round-robin: rank r computes the scopes s = r mod world. Ranks beyond
    sparse_k get none (scope_first >= sparse_k: their calls are no-ops)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must lie in [0, world)")
    return rank, world


def skiparse_attn_bwd_saved(fwd_workspace, v, out, lse, dout, dq, dk, dv, workspace, T, H, W, sparse_k, mode,
                            rope_theta=10000.0, stream=None, fwd_workspace_bytes=None, workspace_bytes=None):
    """Backward pass that reuses the rotated q and k the forward call left in
    `fwd_workspace` (same sizes, mode and rope_theta; unchanged since)."""
    B, heads, N, D = _shape(v)
    if fwd_workspace_bytes is None:
        fwd_workspace_bytes = fwd_workspace.numel() * fwd_workspace.element_size()
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = load_library().skiparse_attn_bwd_saved(_ptr(fwd_workspace), int(fwd_workspace_bytes), _ptr(v), _ptr(out),
                                                _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                                int(workspace_bytes), B, heads, N, D, T, H, W, sparse_k, mode,
                                                float(rope_theta), _stream(stream))
    _check(st, "skiparse_attn_bwd_saved")


def skiparse_attn_bwd_noalloc(q, k, v, out, lse, dout, dq, dk, dv, T, H, W, sparse_k, mode,
                              rope_theta=10000.0, stream=None):
    """Backward pass for callers that cannot allocate device memory: the scratch
    is a fixed array inside the library (SKIPARSE_NOALLOC_SCRATCH_BYTES, 64 MiB),
    shared by all calls, so calls must not overlap on the GPU. Larger sizes are
    rejected with status -6 (SKIPARSE_ERR_WORKSPACE)."""
    B, heads, N, D = _shape(q)
    st = load_library().skiparse_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                                  _ptr(dq), _ptr(dk), _ptr(dv), B, heads, N, D, T, H, W,
                                                  sparse_k, mode, float(rope_theta), _stream(stream))
    _check(st, "skiparse_attn_bwd_noalloc")


NOALLOC_SCRATCH_BYTES = 64 << 20


def skiparse_debug_index_map(scope_of_token, pos_of_token, N, sparse_k, mode, stream=None):
    st = load_library().skiparse_debug_index_map(_ptr(scope_of_token), _ptr(pos_of_token), N, sparse_k, mode,
                                                 _stream(stream))
    _check(st, "skiparse_debug_index_map")


def skiparse_debug_rope(x, x_rot, T, H, W, rope_theta=10000.0, stream=None):
    B, heads, N, D = _shape(x)
    st = load_library().skiparse_debug_rope(_ptr(x), _ptr(x_rot), B, heads, N, D, T, H, W,
                                            float(rope_theta), _stream(stream))
    _check(st, "skiparse_debug_rope")


def skiparse_debug_wait_timeout(code, stream=None):
    """Launches the bounded-wait check (about one second); read it with skiparse_device_error()."""
    _check(load_library().skiparse_debug_wait_timeout(int(code), _stream(stream)), "skiparse_debug_wait_timeout")


def skiparse_qkv_rope(x, w, bias, q, k, v, T, H, W, rope_theta=10000.0, stream=None):
    """[q | k | v] = x w^T (+ bias), RoPE on q and k (the Skiparse listings'
    projections before the attention). x (B, N, C), w (3 heads D, C), bias
    [3 heads D] or None, all bf16; q, k, v (B, N, heads, D) bf16 outputs."""
    B, N, C = x.shape
    Bq, Nq, heads, D = q.shape
    if (Bq, Nq) != (B, N) or tuple(k.shape) != tuple(q.shape) or tuple(v.shape) != tuple(q.shape):
        raise ValueError("q, k, v must be (B, N, heads, D) with x's B and N")
    if tuple(w.shape) != (3 * heads * D, C):
        raise ValueError("w must be (3 heads D, C)")
    if bias is not None and bias.numel() != 3 * heads * D:
        raise ValueError("bias must have 3 heads D elements")
    st = load_library().skiparse_qkv_rope(_ptr(x), _ptr(w), _ptr(bias), _ptr(q), _ptr(k), _ptr(v), B, N, C, heads,
                                          D, T, H, W, float(rope_theta), _stream(stream))
    _check(st, "skiparse_qkv_rope")


def skiparse_device_error():
    """(status, detail): reads and clears the device error word (synchronises)."""
    d = _c_int(0)
    st = load_library().skiparse_device_error(ctypes.byref(d))
    return int(st), int(d.value)


def skiparse_trace_begin():
    _check(load_library().skiparse_trace_begin(), "skiparse_trace_begin")


def skiparse_trace_end(n: int = len(KERNEL_NAMES)):
    """Returns ([ms per kernel id], [launches per kernel id])."""
    ms = (_c_float * n)()
    cnt = (_c_int * n)()
    _check(load_library().skiparse_trace_end(ms, cnt, n), "skiparse_trace_end")
    return [float(x) for x in ms], [int(x) for x in cnt]
