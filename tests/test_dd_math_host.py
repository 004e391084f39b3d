"""Accuracy of the CUDA library's double-float exponential (Tang's table-driven method,
used for the rows that are sampled by inverse CDF), compiled for the host and compared
with the C library's long-double expl. The GPU tests check that the device build gives
the same bits."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "smc_reweight_resample_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("ddprobe") / "libddprobe.so")
    subprocess.check_call(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-I", CSRC, os.path.join(ROOT, "tests", "support", "dd_math_probe.cpp"),
                           "-o", out])
    lib = ctypes.CDLL(out)
    P = ctypes.c_void_p
    lib.probe_exp_split.argtypes = [P, P, ctypes.c_int, P, P, P]
    lib.probe_dd_recip.argtypes = [P, P, ctypes.c_int, P, P]
    return lib


def _exp_split(lib, xh, xl):
    xh = np.ascontiguousarray(xh, np.float32)
    xl = np.ascontiguousarray(xl, np.float32)
    n = xh.size
    hi, lo, e = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.int32)
    lib.probe_exp_split(xh.ctypes.data, xl.ctypes.data, n, hi.ctypes.data, lo.ctypes.data, e.ctypes.data)
    return hi, lo, e


def _rel_err(hi, lo, e, xh, xl):
    ld = np.longdouble
    got = (hi.astype(ld) + lo.astype(ld)) * np.exp2(e.astype(ld))
    want = np.exp(xh.astype(ld) + xl.astype(ld))
    return np.abs(got / want - 1).astype(np.float64)


@pytest.mark.skipif(np.finfo(np.longdouble).eps > 1e-18, reason="needs extended long double")
@pytest.mark.parametrize("scale,tol", [(1.0, 2e-13), (20.0, 2e-13), (100.0, 1e-12), (700.0, 6e-12)])
def test_exp_split_accuracy(probe, scale, tol):
    rng = np.random.default_rng(int(scale))
    xh = (rng.uniform(-1, 1, 200000) * scale).astype(np.float32)
    xl = (xh * rng.uniform(-2 ** -25, 2 ** -25, xh.size)).astype(np.float32)
    hi, lo, e = _exp_split(probe, xh, xl)
    assert ((hi >= 1.0) & (hi < 2.0)).all()
    assert np.abs(lo).max() <= 2.0 ** -23
    assert _rel_err(hi, lo, e, xh, xl).max() < tol


@pytest.mark.skipif(np.finfo(np.longdouble).eps > 1e-18, reason="needs extended long double")
def test_exp_split_bf16_grid_and_edges(probe):
    # every bf16 value in [-64, 64] and the integers, where floor() boundaries sit
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    z = (bits << 16).view(np.float32)
    z = z[np.isfinite(z) & (np.abs(z) <= 64)]
    xs = np.concatenate([z, np.arange(-80, 81, dtype=np.float32), np.float32([0.0, -0.0, 1e-30, -1e-30])])
    hi, lo, e = _exp_split(probe, xs, np.zeros_like(xs))
    assert _rel_err(hi, lo, e, xs, np.zeros_like(xs)).max() < 2e-13


def test_dd_recip(probe):
    rng = np.random.default_rng(3)
    ah = rng.uniform(1, 3e5, 10000).astype(np.float32)
    al = (ah * rng.uniform(-2 ** -25, 2 ** -25, ah.size)).astype(np.float32)
    rh, rl = np.zeros_like(ah), np.zeros_like(ah)
    probe.probe_dd_recip(ah.ctypes.data, al.ctypes.data, ah.size, rh.ctypes.data, rl.ctypes.data)
    ld = np.longdouble
    err = np.abs((rh.astype(ld) + rl.astype(ld)) * (ah.astype(ld) + al.astype(ld)) - 1)
    assert err.max() < 1e-13


def _dd_div(lib, ah, al, bh, bl):
    lib.probe_dd_div.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_void_p] * 2
    args = [np.ascontiguousarray(x, np.float32) for x in (ah, al, bh, bl)]
    qh, ql = np.zeros_like(args[0]), np.zeros_like(args[0])
    lib.probe_dd_div(*[x.ctypes.data for x in args], args[0].size, qh.ctypes.data, ql.ctypes.data)
    return qh, ql


@pytest.mark.skipif(np.finfo(np.longdouble).eps > 1e-18, reason="needs extended long double")
def test_dd_div(probe):
    rng = np.random.default_rng(4)
    ah = rng.uniform(0.5, 3e4, 20000).astype(np.float32)
    al = (ah * rng.uniform(-2 ** -25, 2 ** -25, ah.size)).astype(np.float32)
    bh = rng.uniform(0.5, 3e4, ah.size).astype(np.float32)
    bl = (bh * rng.uniform(-2 ** -25, 2 ** -25, ah.size)).astype(np.float32)
    qh, ql = _dd_div(probe, ah, al, bh, bl)
    ld = np.longdouble
    want = (ah.astype(ld) + al.astype(ld)) / (bh.astype(ld) + bl.astype(ld))
    assert (np.abs((qh.astype(ld) + ql.astype(ld)) / want - 1)).max() < 1e-13
    # quotients that are floats come out exact (an ESS of N^2 / N against a threshold of N)
    n = np.arange(1, 1001, dtype=np.float32)
    qh, ql = _dd_div(probe, n * n, np.zeros_like(n), n, np.zeros_like(n))
    assert (qh == n).all() and (ql == 0).all()
    qh, ql = _dd_div(probe, np.float32([1.0, 3.0, 0.75]), np.zeros(3), np.float32([4.0, 8.0, 3.0]), np.zeros(3))
    assert qh.tolist() == [0.25, 0.375, 0.25] and (ql == 0).all()


@pytest.mark.parametrize("d", [1, 2, 3, 5, 7, 63, 64, 65, 126, 567, 1152, 4097, 72576, 1 << 20, 999983,
                               (1 << 30) + 3])
def test_fast_division(probe, d):
    """The launch-invariant division used to decode chunk indices equals n // d for n < 2^31."""
    probe.probe_fast_div_check.argtypes = [ctypes.c_uint] * 4
    probe.probe_fast_div_check.restype = ctypes.c_int
    assert probe.probe_fast_div_check(d, 0, 200000, 1) == 0
    assert probe.probe_fast_div_check(d, (1 << 31) - 200001, 200000, 1) == 0
    assert probe.probe_fast_div_check(d, 12345, 100000, 21473) == 0
