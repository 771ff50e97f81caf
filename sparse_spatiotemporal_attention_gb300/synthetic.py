"""Seeded synthetic inputs shaped like video-latent attention tensors.

This module is shared by the tests, the bench and the oracle harness. It holds
none of the attention arithmetic: it only draws numbers.

Recipe (the same on every machine, bit for bit):
  * a splitmix64 counter stream: draw n of seed s is mix(s + (n + 1) * 0x9E3779B97F4A7C15),
    where mix is the published splitmix64 finaliser (Steele, Lea, Flood 2014);
  * uniforms u = ((draw >> 11) + 1) * 2**-53, which lie in (0, 1];
  * standard normals by Box-Muller on consecutive pairs (u1, u2):
    r = sqrt(-2 ln u1), z0 = r cos(2 pi u2), z1 = r sin(2 pi u2), in float64;
  * float64 -> float32 (numpy, round to nearest even) -> bfloat16 (round to
    nearest even on the float32 bit pattern).

Tensors are (B, N, heads, D) contiguous, matching the layout the library takes.
Default seeds: q=1, k=2, v=3, dO=4.
"""
from __future__ import annotations

import os

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

SEEDS = {"q": 1, "k": 2, "v": 3, "do": 4}


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the splitmix64 stream of `seed` (uint64)."""
    with np.errstate(over="ignore"):
        z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z *= _GOLDEN
        z += np.uint64(seed)
        t = z >> np.uint64(30)
        z ^= t
        z *= _M1
        np.right_shift(z, np.uint64(27), out=t)
        z ^= t
        z *= _M2
        np.right_shift(z, np.uint64(31), out=t)
        z ^= t
    return z


def _normal_pairs(seed: int, p0: int, p1: int) -> np.ndarray:
    """Box-Muller values 2*p0 .. 2*p1-1 of stream `seed`."""
    z = splitmix64(seed, 2 * p0, 2 * (p1 - p0))
    u = ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * np.pi * u2
    blk = np.empty(2 * (p1 - p0), dtype=np.float64)
    blk[0::2] = r * np.cos(ang)
    blk[1::2] = r * np.sin(ang)
    return blk


def normal_f64(seed: int, count: int, chunk: int = 1 << 21) -> np.ndarray:
    """`count` N(0,1) float64 values of stream `seed` (Box-Muller on draw pairs).
    Chunks are independent (counter-based stream), so they run on a thread pool;
    the result does not depend on the chunking."""
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2

    def work(p0):
        p1 = min(npairs, p0 + chunk)
        blk = _normal_pairs(seed, p0, p1)
        o0, o1 = 2 * p0, min(count, 2 * p1)
        out[o0:o1] = blk[: o1 - o0]

    starts = range(0, npairs, chunk)
    if npairs > chunk:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    else:
        for p0 in starts:
            work(p0)
    return out


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    nan = (b & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    rounded = np.where(nan, (b >> np.uint32(16)) | np.uint32(0x40), rounded)
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def normal_bf16_bits_numpy(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) values rounded to bfloat16, as a uint16 array of `shape`
    (the definition of the recipe, in numpy)."""
    count = int(np.prod(shape))
    x = normal_f64(seed, count)
    if scale != 1.0:
        x = x * scale
    return f32_to_bf16_bits(x.astype(np.float32)).reshape(shape)


_CLIB = None


def _c_generator():
    """The same recipe in C (csrc/synthetic_gen.c), built on demand with gcc."""
    global _CLIB
    if _CLIB is None:
        import ctypes
        from . import _build
        path = _build.build_synthetic()
        lib = ctypes.CDLL(path)
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                          ctypes.c_void_p, ctypes.c_int]
        lib.synth_normal_bf16.restype = None
        _CLIB = lib
    return _CLIB


def normal_bf16_bits(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) values rounded to bfloat16, as a uint16 array of `shape`.
    Uses the threaded C implementation of the recipe; falls back to numpy when
    no C compiler is available."""
    count = int(np.prod(shape))
    try:
        lib = _c_generator()
    except Exception:
        return normal_bf16_bits_numpy(seed, shape, scale)
    out = np.empty(count, dtype=np.uint16)
    lib.synth_normal_bf16(seed, count, float(scale), out.ctypes.data, os.cpu_count() or 1)
    return out.reshape(shape)


def attention_inputs(B: int, N: int, heads: int, D: int, with_grad: bool = False,
                     q_scale: float = 1.0, seeds: dict | None = None) -> dict:
    """q, k, v (and dO) as uint16 bf16 bit arrays of shape (B, N, heads, D)."""
    s = dict(SEEDS)
    if seeds:
        s.update(seeds)
    shape = (B, N, heads, D)
    out = {
        "q": normal_bf16_bits(s["q"], shape, q_scale),
        "k": normal_bf16_bits(s["k"], shape),
        "v": normal_bf16_bits(s["v"], shape),
    }
    if with_grad:
        out["do"] = normal_bf16_bits(s["do"], shape)
    return out
