"""The streaming pass's chunk dealing (smcsd_deal.h), compiled for the host: every chunk of both
lists goes to exactly one block and one local position, a block's local sequence has no gaps, a
block's precise chunks are exactly items b, b + B, ... of the precise list, and with the phase-1
ratio the kernels use the precise chunks are used up before the last fifth of every block's
sequence (so that the draws they feed finish inside the pass)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "smc_reweight_resample_gb300", "csrc")
BIT = 0x80000000


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("dealprobe") / "libdealprobe.so")
    subprocess.check_call(["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-I", CSRC,
                           os.path.join(ROOT, "tests", "support", "deal_probe.cpp"), "-o", out])
    lib = ctypes.CDLL(out)
    lib.probe_deal.argtypes = [ctypes.c_longlong, ctypes.c_longlong, ctypes.c_int, ctypes.c_uint,
                               ctypes.c_uint, ctypes.c_void_p, ctypes.c_int]
    lib.probe_fper.argtypes = [ctypes.c_int]
    return lib


def deal(lib, n_precise, n_fast, fper, B, ring=32, max_local=4096):
    items = np.zeros(B * max_local, np.int64)
    most = lib.probe_deal(n_precise, n_fast, fper, B, ring, items.ctypes.data, max_local)
    assert most >= 0
    return items.reshape(B, max_local)[:, :max(most, 1)]


CASES = [
    # (S, fast rows per sampled row, cpr, B): the 8 x 16 step, the 4 x 64 power step, the draft
    # sampler (no fast rows), small and ragged shapes
    (128, 8, 63, 152), (256, 16, 75, 152), (512, 0, 63, 152), (12, 6, 3, 7), (5, 2, 1, 3),
    (1, 8, 63, 152), (33, 4, 2, 20),
]


@pytest.mark.parametrize("S,fslots,cpr,B", CASES)
def test_every_chunk_once(probe, S, fslots, cpr, B):
    n_precise, n_fast = S * cpr, S * fslots * cpr
    fper = probe.probe_fper(fslots)
    it = deal(probe, n_precise, n_fast, fper, B)
    prec, fast = [], []
    for b in range(B):
        row = it[b]
        n = int((row != -2).sum())
        assert (row[:n] != -2).all() and (row[n:] == -2).all()  # no gaps
        p = [int(x) & ~BIT for x in row[:n] if int(x) & BIT]
        f = [int(x) for x in row[:n] if not int(x) & BIT]
        assert p == list(range(b, n_precise, B))  # in list order
        assert f == list(range(B - 1 - b, n_fast, B))
        prec += p
        fast += f
        if p and f and fslots >= 4:
            last_p = max(k for k in range(n) if int(row[k]) & BIT)
            assert last_p < 0.85 * n, (b, last_p, n)
    assert sorted(prec) == list(range(n_precise))
    assert sorted(fast) == list(range(n_fast))


def test_fper(probe):
    assert [probe.probe_fper(f) for f in (0, 1, 2, 4, 8, 16)] == [0, 1, 1, 3, 6, 12]
