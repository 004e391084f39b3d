"""The CUDA library builds, loads and exports every entry point that include/smcsd.h declares;
the host-only entry points and argument checks work without a GPU (nothing is enqueued)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smcsd.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from smc_reweight_resample_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sd_verify", "smc_reweight", "smc_ess_resample", "kv_pagetable_remap",
              "pacer_block_stop", "smc_step", "smcsd_workspace_size", "smcsd_workspace_init",
              "smcsd_check_status", "smcsd_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_host_only_entry_points(lib):
    lib.smcsd_status_string.restype = ctypes.c_char_p
    assert lib.smcsd_status_string(0) == b"ok"
    assert b"range" in lib.smcsd_status_string(-6)
    lib.smcsd_workspace_size.restype = ctypes.c_size_t
    n3 = lib.smcsd_workspace_size(2, 128, 4, 128256)
    assert n3 > 0 and n3 % 256 == 0
    assert lib.smcsd_workspace_size(0, 0, 4, 100) == 0
    assert lib.smcsd_workspace_size(99, 4, 4, 100) == 0


def test_argument_checks_return_before_any_cuda_call(lib):
    P = ctypes.c_void_p
    lib.sd_verify.argtypes = [P, P, ctypes.c_int, P, P, P, ctypes.c_int, ctypes.c_int,
                              ctypes.c_int, ctypes.c_float, P, P, P, P, P, P, ctypes.c_size_t, P]
    fake = P(256)
    # unsupported dtype
    assert lib.sd_verify(fake, fake, 7, fake, None, None, 4, 2, 10, 1.0, fake, fake, fake, None,
                         None, fake, 1 << 20, None) == -2
    # null target logits
    assert lib.sd_verify(None, fake, 1, fake, None, None, 4, 2, 10, 1.0, fake, fake, fake, None,
                         None, fake, 1 << 20, None) == -1
    # temperature <= 0
    assert lib.sd_verify(fake, fake, 1, fake, None, None, 4, 2, 10, 0.0, fake, fake, fake, None,
                         None, fake, 1 << 20, None) == -1
    # one ragged offset array without the other
    assert lib.sd_verify(fake, fake, 1, fake, fake, None, 4, 2, 10, 1.0, fake, fake, fake, None,
                         None, fake, 1 << 20, None) == -1
    # workspace too small
    assert lib.sd_verify(fake, fake, 1, fake, None, None, 4, 2, 10, 1.0, fake, fake, fake, None,
                         None, fake, 16, None) == -3


def test_tilted_and_pos_emb_argument_checks(lib):
    P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.smc_reweight_tilted.argtypes = [P, P, i, P, i, i, i, f, f, i, P, f, P, P, P, P, P, P, sz, P]
    fake = P(256)

    def rw(target, reward, scale, alpha=2.0, ws_bytes=1 << 20):
        return lib.smc_reweight_tilted(fake, fake, 1, fake, 4, 2, 10, 1.0, alpha, target, reward,
                                       scale, fake, fake, fake, None, None, fake, ws_bytes, None)

    assert rw(2, None, 0.0) == -1                  # unknown target
    assert rw(-1, None, 0.0) == -1
    assert rw(1, fake, float("nan")) == -1         # reward given with a non-finite scale
    assert rw(1, fake, float("inf")) == -1
    assert rw(1, None, 0.0, alpha=0.0) == -1       # alpha <= 0
    assert rw(1, fake, 0.5, ws_bytes=16) == -3     # valid up to the workspace size
    lib.pacer_block_stop_pos.argtypes = [P, P, P, f, i, i, i, i, f, f, P, P, P, P, P, sz, P]
    # b above the kernel's limit of 64, and a null head, are refused with or without embeddings
    assert lib.pacer_block_stop_pos(fake, fake, fake, 0.0, 4, 65, 5, 16, 0.5, 1.1, fake, None,
                                    None, None, fake, 1 << 20, None) == -1
    assert lib.pacer_block_stop_pos(fake, None, fake, 0.0, 4, 4, 5, 16, 0.5, 1.1, fake, None,
                                    None, None, fake, 1 << 20, None) == -1


def test_draft_sample_argument_checks(lib):
    P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.draft_sample.argtypes = [P, i, i, i, f, P, P, P, P, P, sz, P]
    lib.smcsd_workspace_size.restype = ctypes.c_size_t
    fake = P(256)
    ok_ws = lib.smcsd_workspace_size(6, 8, 0, 100)
    assert ok_ws > 0 and ok_ws == lib.smcsd_workspace_size(6, 8, 5, 100)  # K is ignored
    assert lib.draft_sample(fake, 3, 8, 100, 1.0, fake, fake, None, None, fake, ok_ws, None) == -2
    assert lib.draft_sample(None, 1, 8, 100, 1.0, fake, fake, None, None, fake, ok_ws, None) == -1
    assert lib.draft_sample(fake, 1, 8, 100, 1.0, fake, None, None, None, fake, ok_ws, None) == -1
    assert lib.draft_sample(fake, 1, 0, 100, 1.0, fake, fake, None, None, fake, ok_ws, None) == -1
    assert lib.draft_sample(fake, 1, 8, 100, 0.0, fake, fake, None, None, fake, ok_ws, None) == -1
    assert lib.draft_sample(fake, 1, 8, 100, 1.0, fake, fake, None, None, fake, 64, None) == -3


def test_selftest_wait_argument_checks(lib):
    P, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.smcsd_selftest_wait.argtypes = [ctypes.c_uint, P, sz, P]
    fake = P(256)
    assert lib.smcsd_selftest_wait(0, fake, 1024, None) == -1          # no limit
    assert lib.smcsd_selftest_wait(2000001, fake, 1024, None) == -1    # above 2 s
    assert lib.smcsd_selftest_wait(1000, None, 1024, None) == -1       # no workspace
    assert lib.smcsd_selftest_wait(1000, fake, 2, None) == -3          # workspace too small
    assert lib.smcsd_selftest_wait(1000, P(260), 1024, None) == -3     # misaligned
