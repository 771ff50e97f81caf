"""The FMA-pipe 2^x that the forward kernels' softmax uses for a share of P.

CPU: the coefficients compiled into skiparse_dev.cuh are the float32 rounding
of a fresh Remez fit (exp2_poly_fit.py), and a float32 emulation of the whole
routine (clamp, round-to-nearest reduction with the 1.5 * 2^23 shifter, Horner
with one rounding per fused multiply-add, exponent added as an integer) stays
within the fit's relative error of float64 2^x over the kernels' argument range.
GPU: the device routine through the C ABI against float64 2^x and against the
hardware ex2.approx on the same inputs.
"""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_spatiotemporal_attention_gb300", "csrc")
REL_BOUND = 7.6e-5          # Remez level 7.48e-5 plus float32 evaluation


def _fit_module():
    spec = importlib.util.spec_from_file_location("exp2_poly_fit", os.path.join(CSRC, "exp2_poly_fit.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _compiled_coeffs():
    src = open(os.path.join(CSRC, "skiparse_dev.cuh")).read()
    line = re.search(r"constexpr float kC0 = [^;]*;", src).group(0)
    vals = dict(re.findall(r"(kC\d) = ([0-9a-fx.p+-]+)f", line))
    return np.array([float.fromhex(vals[f"kC{i}"]) for i in range(4)], dtype=np.float32)


def test_coefficients_are_the_float32_remez_fit():
    fit = _fit_module()
    c, E = fit.remez(3)
    assert 7.0e-5 < E < 7.6e-5
    assert np.array_equal(_compiled_coeffs(), c.astype(np.float32))


def _emulate(x):
    """The device routine in numpy float32 (no fused ops except where the device
    fuses: Horner steps are fused multiply-adds, emulated in float64 then rounded
    once, exact for float32 operands since the product fits in float64)."""
    c = _compiled_coeffs()
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-125.0))
    sh = (x + np.float32(12582912.0)).astype(np.float32)
    j = (sh - np.float32(12582912.0)).astype(np.float32)
    f = (x - j).astype(np.float32)
    f64 = f.astype(np.float64)
    p = ((np.float64(c[3]) * f64 + np.float64(c[2])).astype(np.float32)).astype(np.float64)
    p = ((p * f64 + np.float64(c[1])).astype(np.float32)).astype(np.float64)
    p = (p * f64 + np.float64(c[0])).astype(np.float32)
    bits = p.view(np.int32).astype(np.int64) + (sh.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32), f


def _inputs():
    rs = np.random.RandomState(17)
    return np.concatenate([
        rs.uniform(-130.0, 9.99, 200000), rs.uniform(-2.0, 2.0, 50000),
        np.arange(-125, 10, dtype=np.float64), np.arange(-125, 10) + 0.5, np.arange(-125, 10) - 0.5,
        [0.0, -0.0, 1e-30, -1e-30, -125.0, -126.0, -1000.0, 9.999, -124.5000001],
    ]).astype(np.float32)


def test_emulated_routine_within_the_fit_error():
    x = _inputs()
    y, f = _emulate(x)
    assert np.all(np.abs(f) <= 0.5)
    want = np.exp2(np.maximum(x.astype(np.float64), -125.0))
    rel = np.abs(y.astype(np.float64) / want - 1.0)
    assert rel.max() <= REL_BOUND, (rel.max(), x[np.argmax(rel)])
    # exact powers of two come out within the polynomial's error at f = 0
    k = np.arange(-125, 10, dtype=np.float32)
    yk, _ = _emulate(k)
    assert np.all(np.abs(yk.astype(np.float64) / np.exp2(k.astype(np.float64)) - 1.0) <= REL_BOUND)


def test_exp2_hook_validates_without_a_device():
    import sparse_spatiotemporal_attention_gb300 as skp
    lib = skp.load_library()
    assert lib.skiparse_debug_exp2(None, None, -1, 0, None) == -1
    assert lib.skiparse_debug_exp2(None, None, 4, 0, None) == -1
    assert lib.skiparse_debug_exp2(16, 32, 4, 2, None) == -1
    assert lib.skiparse_debug_exp2(None, None, 0, 0, None) == 0


@pytest.mark.gpu
def test_device_exp2_against_float64_and_mufu():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import sparse_spatiotemporal_attention_gb300 as skp
    dev = torch.device("cuda:0")
    x = _inputs()
    xd = torch.from_numpy(x).to(dev)
    yp = torch.empty_like(xd)
    ym = torch.empty_like(xd)
    skp.skiparse_debug_exp2(xd, yp)
    skp.skiparse_debug_exp2(xd, ym, mufu=True)
    torch.cuda.synchronize()
    yp, ym = yp.cpu().numpy().astype(np.float64), ym.cpu().numpy().astype(np.float64)
    want = np.exp2(np.maximum(x.astype(np.float64), -125.0))
    rel = np.abs(yp / want - 1.0)
    assert rel.max() <= REL_BOUND, (rel.max(), x[np.argmax(rel)])
    # the device agrees with the float32 emulation bit for bit
    ye, _ = _emulate(x)
    assert np.array_equal(yp.astype(np.float32).view(np.uint32), ye.view(np.uint32))
    # and with the hardware's own 2^x within the polynomial's error (normal range)
    sel = x >= -125.0
    assert np.max(np.abs(yp[sel] / ym[sel] - 1.0)) <= REL_BOUND + 2.0 ** -21
    # odd sizes: the tail element is written, nothing past it
    buf = torch.full((8,), -7.0, device=dev)
    skp.skiparse_debug_exp2(xd[:5], buf[:5])
    torch.cuda.synchronize()
    assert torch.all(buf[5:] == -7.0) and torch.all(buf[:5] > 0)
