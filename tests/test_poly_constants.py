"""CPU pins for the two polynomials the kernels evaluate on the FMA pipe.

The coefficients live in the CUDA sources (the tanh fit in the host code that
folds scale and cap into it, the 2^f fit in the kernel header).  Here they
are parsed from those files, evaluated in float32 Horner arithmetic as the
kernels do, and checked against numpy's tanh and exp2 within the bounds the
kernels rely on; the fitting script's defaults must reproduce them.  The
exp2 test also replays the kernel's Cody-Waite split (round-down add of a
magic constant, exponent bits from a shift) bit for bit in numpy.
"""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "flashattention_attn_fwd_gb300", "csrc")


def _fit_module():
    spec = importlib.util.spec_from_file_location("fit_poly", os.path.join(CSRC, "fit_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _tanh_coeffs():
    txt = open(os.path.join(CSRC, "api.cu")).read()
    m = re.search(r"kTanhP\[4\]\s*=\s*\{([^}]*)\}", txt)
    return np.array([float(x.strip().rstrip("f")) for x in m.group(1).split(",")], dtype=np.float32)


def _exp2_coeffs():
    txt = open(os.path.join(CSRC, "fused_attn.cuh")).read()
    return np.array([float(re.search(rf"kExp2E{i}\s*=\s*([0-9.eE+-]+)f", txt).group(1)) for i in range(4)],
                    dtype=np.float32)


def _horner(c, x):
    acc = np.float32(c[-1])
    for cj in c[-2::-1]:
        acc = (acc * x + np.float32(cj)).astype(np.float32)
    return acc


def test_tanh_polynomial_accuracy():
    c = _tanh_coeffs()
    y = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    t = (y * _horner(c, (y * y).astype(np.float32))).astype(np.float32)
    ref = np.tanh(y.astype(np.float64))
    nz = ref != 0
    assert np.max(np.abs(t[nz] - ref[nz]) / np.abs(ref[nz])) < 1e-6


def test_tanh_polynomial_folded_like_the_host():
    """The host folds cap*log2(e) and scale/cap into q_i = k p_i ya^(2i+1);
    s * Q(s^2) must then equal cap*log2(e)*tanh(s*scale/cap) in range."""
    c = _tanh_coeffs().astype(np.float64)
    scale, cap = 0.125, 30.0
    ya, k = scale / cap, cap * np.log2(np.e)
    q = np.float32([k * c[i] * ya ** (2 * i + 1) for i in range(4)])
    smax = 0.5 / ya
    s = np.linspace(-smax, smax, 100001).astype(np.float32)
    x = (s * _horner(q, (s * s).astype(np.float32))).astype(np.float32)
    ref = k * np.tanh(s.astype(np.float64) * ya)
    assert np.max(np.abs(x - ref)) < 1e-4  # log2 units; far below bf16 P rounding


def test_exp2_polynomial_accuracy():
    c = _exp2_coeffs()
    f = np.linspace(0, 1, 200001, endpoint=False).astype(np.float32)
    e = _horner(c, f)
    ref = np.exp2(f.astype(np.float64))
    assert np.max(np.abs(e - ref) / ref) < 1e-4


def test_exp2_cody_waite_split_bitwise():
    """Replays the kernel's 2^a for a in [-140, 8]: clamp at -127, t = a +
    magic rounded down, f = a - (t - magic), exponent bits (bits(t) << 23)."""
    c = _exp2_coeffs()
    magic = np.float32(12583039.0)  # 1.5 * 2^23 + 127
    a = np.concatenate([np.linspace(-140, 8, 300001), [-np.inf, 0.0, -127.0, -126.5, 7.99]]).astype(np.float32)
    ac = np.maximum(a, np.float32(-127.0))
    # round-down add: exact sum in float64, then the float32 at or below it
    exact = ac.astype(np.float64) + np.float64(magic)
    t = exact.astype(np.float32)
    t = np.where(t.astype(np.float64) > exact, np.nextafter(t, np.float32(-np.inf)), t).astype(np.float32)
    f = (ac - (t - magic)).astype(np.float32)
    assert np.all((f >= 0) & (f < 1))
    scale_bits = (t.view(np.uint32) << np.uint32(23)).astype(np.uint32)
    p = (_horner(c, f) * scale_bits.view(np.float32)).astype(np.float32)
    ref = np.exp2(np.maximum(a.astype(np.float64), -127.0))
    big = ref > 2.0 ** -126
    assert np.max(np.abs(p[big] - ref[big]) / ref[big]) < 1e-4
    assert np.all(p[~big] <= 2.0 ** -126)
    assert p[a == -np.inf][0] == 0.0


def test_fit_script_defaults_reproduce_the_constants():
    fit = _fit_module()
    ct, _ = fit.fit_tanh(0.5, 3)
    ce, _ = fit.fit_exp2(3)
    np.testing.assert_allclose(ct, _tanh_coeffs(), rtol=2e-6)
    np.testing.assert_allclose(ce, _exp2_coeffs(), rtol=2e-6)
