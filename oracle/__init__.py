"""Float64 CPU oracle: ctypes binding for ``smc_oracle.c``.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The product path (the CUDA library and its
Python binding) never imports it, and the two share no code.

Every wrapper takes numpy arrays: bf16 logits as ``uint16`` bit patterns, fp32 logits as
``float32``. The C functions cite the passages of the pages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smc_oracle.c")
_LIB = os.path.join(_HERE, "libsmc_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EDTYPE, ENONFINITE, ERANGE = 0, -1, -2, -5, -6


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable flags, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i, d, f, ll = ctypes.c_int, ctypes.c_double, ctypes.c_float, ctypes.c_longlong
            lib.oracle_row_lse.argtypes = [P, i, ll, i, d, P]
            lib.oracle_sample_inverse_cdf.argtypes = [P, i, d, P, P]
            lib.oracle_sd_verify.argtypes = [P, P, i, P, P, P, i, i, i, f, P, P, P, P, P, P, P]
            lib.oracle_smc_reweight.argtypes = [P, P, i, P, i, i, i, f, f, P, P, P, P, P, P, P]
            lib.oracle_smc_reweight_tilted.argtypes = [P, P, i, P, i, i, i, f, f, i, P, f, P, P, P,
                                                       P, P, P, P]
            lib.oracle_ess_resample.argtypes = [P, i, i, f, P, P, P, P, P, P]
            lib.oracle_draft_sample.argtypes = [P, i, i, i, f, P, P, P, P, P]
            lib.oracle_pagetable_remap.argtypes = [P, P, i, i, P, P, i, P, i]
            lib.oracle_pacer_block_stop.argtypes = [P, P, f, i, i, i, i, f, f, P, P, P]
            lib.oracle_pacer_block_stop_pos.argtypes = [P, P, P, f, i, i, i, i, f, f, P, P, P]
            for fn in (lib.oracle_row_lse, lib.oracle_sample_inverse_cdf, lib.oracle_sd_verify,
                       lib.oracle_smc_reweight, lib.oracle_smc_reweight_tilted,
                       lib.oracle_ess_resample, lib.oracle_pagetable_remap,
                       lib.oracle_pacer_block_stop, lib.oracle_pacer_block_stop_pos,
                       lib.oracle_draft_sample):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _q(a, offset):
    """Pointer to element `offset` of a contiguous array (None stays None)."""
    return None if a is None else ctypes.c_void_p(a.ctypes.data + int(offset) * a.itemsize)


def _blocks(n, threads):
    """Contiguous blocks [s0, s1) covering range(n), one per thread."""
    t = max(1, min(int(threads), n))
    edges = [n * i // t for i in range(t + 1)]
    return [(edges[i], edges[i + 1]) for i in range(t) if edges[i + 1] > edges[i]]


def _run_blocks(n, threads, fn):
    """Runs fn(s0, s1) over the blocks, in threads when threads > 1 (ctypes releases the GIL
    for the C call, so the blocks run in parallel), and returns the first nonzero status in
    block order, which is the status a single call over all of range(n) returns: every
    sequence or particle is computed on its own, so the split changes no result."""
    blocks = _blocks(n, threads)
    if len(blocks) == 1:
        return fn(*blocks[0])
    with ThreadPoolExecutor(max_workers=len(blocks)) as ex:
        rcs = list(ex.map(lambda b: fn(*b), blocks))
    for rc in rcs:
        if rc != OK:
            return rc
    return OK


def default_threads() -> int:
    """Threads for the heavy oracle calls of the tests: every host core."""
    return os.cpu_count() or 1


def _dtype_code(logits: np.ndarray) -> int:
    if logits.dtype == np.float32:
        return 0
    if logits.dtype == np.uint16:
        return 1
    raise TypeError("logits must be float32 or uint16 (bf16 bits)")


class OracleError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: oracle status {code}")
        self.code = code


def _check(rc: int, where: str):
    if rc != OK:
        raise OracleError(rc, where)


def row_lse(logits: np.ndarray, row: int, V: int, scale: float) -> float:
    lib = _load()
    logits = np.ascontiguousarray(logits)
    out = np.zeros(1, np.float64)
    _check(lib.oracle_row_lse(_p(logits), _dtype_code(logits), row, V, scale, _p(out)), "row_lse")
    return float(out[0])


def sample_inverse_cdf(r: np.ndarray, u: float):
    lib = _load()
    r = np.ascontiguousarray(r, dtype=np.float64)
    tok = np.zeros(1, np.int32)
    marg = np.zeros(1, np.float64)
    _check(lib.oracle_sample_inverse_cdf(_p(r), r.size, float(u), _p(tok), _p(marg)), "inverse_cdf")
    return int(tok[0]), float(marg[0])


def sd_verify(tgt, drf, draft_tokens, S, K, V, temperature, uniforms, tgt_offsets=None,
              drf_offsets=None, raise_on_error=True, threads=1):
    """Returns a dict with accept_len, out_token, lse_tgt, lse_drf, accept_margin,
    token_margin and status. ``threads`` > 1 splits the sequences into contiguous blocks run
    in parallel; the results are the same bits."""
    lib = _load()
    tgt = np.ascontiguousarray(tgt)
    drf = np.ascontiguousarray(drf)
    dt = _dtype_code(tgt)
    assert _dtype_code(drf) == dt
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    to = None if tgt_offsets is None else np.ascontiguousarray(tgt_offsets, dtype=np.int32)
    do = None if drf_offsets is None else np.ascontiguousarray(drf_offsets, dtype=np.int32)
    rows_t = tgt.size // V
    rows_d = max(drf.size // V, 1)
    out = dict(
        accept_len=np.full(S, -7, np.int32), out_token=np.full(S, -7, np.int32),
        lse_tgt=np.full(rows_t, np.nan), lse_drf=np.full(rows_d, np.nan),
        accept_margin=np.full(max(S * K, 1), -1.0), token_margin=np.full(S, np.nan),
    )
    ragged = to is not None

    def block(s0, s1):
        # fixed layout: row and token offsets follow s; ragged: the offsets stay absolute
        tr, dr = (0, 0) if ragged else (s0 * (K + 1) * V, s0 * K * V)
        tk = 0 if ragged else s0 * K
        lt, ld = (0, 0) if ragged else (s0 * (K + 1), s0 * K)
        return lib.oracle_sd_verify(
            _q(tgt, tr), _q(drf, dr), dt, _q(draft_tokens, tk), _q(to, s0), _q(do, s0), s1 - s0,
            K, V, float(temperature), _q(uniforms, s0 * (K + 1)), _q(out["accept_len"], s0),
            _q(out["out_token"], s0), _q(out["lse_tgt"], lt), _q(out["lse_drf"], ld),
            _q(out["accept_margin"], s0 * K), _q(out["token_margin"], s0))

    rc = _run_blocks(S, threads, block)
    out["status"] = rc
    if raise_on_error:
        _check(rc, "sd_verify")
    return out


def smc_reweight(tgt, drf, draft_tokens, S, K, V, temperature, alpha, uniforms, logw,
                 raise_on_error=True, threads=1):
    """``logw`` (float32 [S]) is copied, updated and returned in the dict. ``threads`` > 1
    splits the particles into contiguous blocks run in parallel; the results are the same
    bits."""
    lib = _load()
    tgt = np.ascontiguousarray(tgt)
    drf = np.ascontiguousarray(drf)
    dt = _dtype_code(tgt)
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    lw = np.array(logw, dtype=np.float32, copy=True)
    out = dict(
        logw=lw, bonus_token=np.full(S, -7, np.int32), lse_tgt=np.full(S * (K + 1), np.nan),
        lse_drf=np.full(max(S * K, 1), np.nan), bonus_margin=np.full(S, np.nan),
        dlogw=np.full(S, np.nan),
    )
    def block(s0, s1):
        return lib.oracle_smc_reweight(
            _q(tgt, s0 * (K + 1) * V), _q(drf, s0 * K * V), dt, _q(draft_tokens, s0 * K), s1 - s0,
            K, V, float(temperature), float(alpha), _q(uniforms, s0), _q(lw, s0),
            _q(out["bonus_token"], s0), _q(out["lse_tgt"], s0 * (K + 1)),
            _q(out["lse_drf"], s0 * K), _q(out["bonus_margin"], s0), _q(out["dlogw"], s0))

    rc = _run_blocks(S, threads, block)
    out["status"] = rc
    if raise_on_error:
        _check(rc, "smc_reweight")
    return out


TARGET_TOKEN, TARGET_SEQUENCE = 0, 1


def smc_reweight_tilted(tgt, drf, draft_tokens, S, K, V, temperature, alpha, uniforms, logw,
                        target_mode=TARGET_TOKEN, log_reward=None, reward_scale=0.0,
                        raise_on_error=True, threads=1):
    """Reweight with the per-position (TARGET_TOKEN) or whole-sequence (TARGET_SEQUENCE) power
    target and an optional additive log-reward; same dict as ``smc_reweight``."""
    lib = _load()
    tgt = np.ascontiguousarray(tgt)
    drf = np.ascontiguousarray(drf)
    dt = _dtype_code(tgt)
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    rw = None if log_reward is None else np.ascontiguousarray(log_reward, dtype=np.float32)
    lw = np.array(logw, dtype=np.float32, copy=True)
    out = dict(
        logw=lw, bonus_token=np.full(S, -7, np.int32), lse_tgt=np.full(S * (K + 1), np.nan),
        lse_drf=np.full(max(S * K, 1), np.nan), bonus_margin=np.full(S, np.nan),
        dlogw=np.full(S, np.nan),
    )
    def block(s0, s1):
        return lib.oracle_smc_reweight_tilted(
            _q(tgt, s0 * (K + 1) * V), _q(drf, s0 * K * V), dt, _q(draft_tokens, s0 * K), s1 - s0,
            K, V, float(temperature), float(alpha), int(target_mode), _q(rw, s0),
            float(reward_scale), _q(uniforms, s0), _q(lw, s0), _q(out["bonus_token"], s0),
            _q(out["lse_tgt"], s0 * (K + 1)), _q(out["lse_drf"], s0 * K),
            _q(out["bonus_margin"], s0), _q(out["dlogw"], s0))

    rc = _run_blocks(S, threads, block)
    out["status"] = rc
    if raise_on_error:
        _check(rc, "smc_reweight_tilted")
    return out


def draft_sample(logits, R, V, temperature, uniforms, raise_on_error=True, threads=1):
    """One token per row from softmax(z/T) by inverse CDF; dict with tokens, logq, lse, margin."""
    lib = _load()
    logits = np.ascontiguousarray(logits)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    out = dict(tokens=np.full(R, -7, np.int32), logq=np.full(R, np.nan), lse=np.full(R, np.nan),
               margin=np.full(R, np.nan))
    def block(r0, r1):
        return lib.oracle_draft_sample(
            _q(logits, r0 * V), _dtype_code(logits), r1 - r0, V, float(temperature),
            _q(uniforms, r0), _q(out["tokens"], r0), _q(out["logq"], r0), _q(out["lse"], r0),
            _q(out["margin"], r0))

    rc = _run_blocks(R, threads, block)
    out["status"] = rc
    if raise_on_error:
        _check(rc, "draft_sample")
    return out


def ess_resample(logw, G, N, ess_threshold, uniforms, raise_on_error=True):
    lib = _load()
    lw = np.array(logw, dtype=np.float32, copy=True)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    out = dict(
        logw=lw, ancestors=np.full(G * N, -7, np.int32), ess=np.full(G, np.nan, np.float32),
        resampled=np.full(G, -7, np.int32), ess_margin=np.full(G, np.nan),
        anc_margin=np.full(G * N, np.nan),
    )
    rc = lib.oracle_ess_resample(_p(lw), G, N, float(ess_threshold), _p(uniforms),
                                 _p(out["ancestors"]), _p(out["ess"]), _p(out["resampled"]),
                                 _p(out["ess_margin"]), _p(out["anc_margin"]))
    out["status"] = rc
    if raise_on_error:
        _check(rc, "ess_resample")
    return out


def pagetable_remap(ancestors, resampled, G, N, table_in, pages_per_seq, num_pages=0,
                    with_refcount=True, raise_on_error=True):
    lib = _load()
    anc = np.ascontiguousarray(ancestors, dtype=np.int32)
    res = None if resampled is None else np.ascontiguousarray(resampled, dtype=np.int32)
    tin = np.ascontiguousarray(table_in, dtype=np.int32)
    tout = np.full(G * N * pages_per_seq, -7, np.int32)
    rc_arr = np.full(max(num_pages, 1), -7, np.int32) if with_refcount else None
    rc = lib.oracle_pagetable_remap(_p(anc), _p(res), G, N, _p(tin), _p(tout), pages_per_seq,
                                    _p(rc_arr), num_pages)
    if raise_on_error:
        _check(rc, "pagetable_remap")
    return dict(table_out=tout, refcount=rc_arr, status=rc)


def pacer_block_stop(hidden, w, c, S, b, max_blocks, d, t0, rho, pos_emb=None,
                     raise_on_error=True):
    """``pos_emb``: optional bf16 bits [max_blocks*b, d] added to every sequence's hidden states."""
    lib = _load()
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    out = dict(lengths=np.full(S, -7, np.int32), block_scores=np.full(S * max_blocks, np.nan),
               margin=np.full(S, np.nan))
    if pos_emb is None:
        rc = lib.oracle_pacer_block_stop(_p(hidden), _p(w), float(c), S, b, max_blocks, d,
                                         float(t0), float(rho), _p(out["lengths"]),
                                         _p(out["block_scores"]), _p(out["margin"]))
    else:
        pe = np.ascontiguousarray(pos_emb, dtype=np.uint16)
        assert pe.size == max_blocks * b * d
        rc = lib.oracle_pacer_block_stop_pos(_p(hidden), _p(w), _p(pe), float(c), S, b, max_blocks,
                                             d, float(t0), float(rho), _p(out["lengths"]),
                                             _p(out["block_scores"]), _p(out["margin"]))
    out["status"] = rc
    if raise_on_error:
        _check(rc, "pacer_block_stop")
    return out
