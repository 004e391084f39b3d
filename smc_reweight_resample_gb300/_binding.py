"""ctypes binding of the C ABI in ``include/smcsd.h``.

Argument marshalling only: every step of the path runs in the CUDA library. Tensors must
already live on the CUDA device; outputs are allocated with torch when not supplied. The
library is loaded from this package directory and its absence is an error: there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsmcsd.so")

OK, ERR_INVALID_ARG, ERR_DTYPE, ERR_WORKSPACE, ERR_CUDA, ERR_NONFINITE, ERR_RANGE, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6, -7
F32, BF16 = 0, 1
TARGET_TOKEN, TARGET_SEQUENCE = 0, 1
(OP_SD_VERIFY, OP_SMC_REWEIGHT, OP_SMC_STEP, OP_ESS_RESAMPLE, OP_PAGETABLE_REMAP, OP_PACER_BLOCK_STOP,
 OP_DRAFT_SAMPLE) = range(7)

_lib = None


class SMCSDError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


def load(path: str = LIB_PATH):
    """Load the CUDA library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run smc_reweight_resample_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.smcsd_workspace_size.argtypes = [i, i, i, i]
    lib.smcsd_workspace_size.restype = sz
    lib.smcsd_workspace_init.argtypes = [P, sz, P]
    lib.smcsd_check_status.argtypes = [P, P]
    lib.smcsd_status_string.argtypes = [i]
    lib.smcsd_status_string.restype = ctypes.c_char_p
    lib.sd_verify.argtypes = [P, P, i, P, P, P, i, i, i, f, P, P, P, P, P, P, sz, P]
    lib.smc_reweight.argtypes = [P, P, i, P, i, i, i, f, f, P, P, P, P, P, P, sz, P]
    lib.smc_ess_resample.argtypes = [P, i, i, f, P, P, P, P, P, sz, P]
    lib.kv_pagetable_remap.argtypes = [P, P, i, i, P, P, i, P, i, P, sz, P]
    lib.pacer_block_stop.argtypes = [P, P, f, i, i, i, i, f, f, P, P, P, P, P, sz, P]
    lib.smc_step.argtypes = [P, P, i, P, i, i, i, i, f, f, P, P, P, f, P, P, P, P, P, P, i, P, i,
                             P, sz, P]
    lib.smc_step_static.argtypes = [P, P, i, P, i, i, i, i, f, f, P, P, P, f, P, P, P, P, P, P, i,
                                    P, i, P, P]
    lib.smc_step_logq.argtypes = [P, i, P, P, i, i, i, i, f, f, P, P, P, f, P, P, P, P, P, P, i, P,
                                  i, P, sz, P]
    lib.smc_reweight_tilted.argtypes = [P, P, i, P, i, i, i, f, f, i, P, f, P, P, P, P, P, P, sz, P]
    lib.smc_step_tilted.argtypes = [P, P, i, P, i, i, i, i, f, f, i, P, f, P, P, P, f, P, P, P, P,
                                    P, P, i, P, i, P, sz, P]
    lib.pacer_block_stop_pos.argtypes = [P, P, P, f, i, i, i, i, f, f, P, P, P, P, P, sz, P]
    lib.draft_sample.argtypes = [P, i, i, i, f, P, P, P, P, P, sz, P]
    lib.smcsd_selftest_wait.argtypes = [ctypes.c_uint, P, sz, P]
    for fn in ("smcsd_workspace_init", "smcsd_check_status", "sd_verify", "smc_reweight",
               "smc_ess_resample", "kv_pagetable_remap", "pacer_block_stop", "smc_step",
               "smc_step_static", "smc_step_logq", "smc_reweight_tilted", "smc_step_tilted",
               "pacer_block_stop_pos", "draft_sample", "smcsd_selftest_wait"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().smcsd_status_string(int(code)).decode()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits must be float32 or bfloat16, not {t.dtype}")


def _check(rc: int, where: str):
    if rc != OK:
        raise SMCSDError(rc, where)


def workspace_size(op: int, S: int, K: int = 0, V: int = 1) -> int:
    return int(load().smcsd_workspace_size(op, S, K, V))


class Workspace:
    """Scratch buffer for one stream of calls (zero-filled at creation, as the ABI requires)."""

    def __init__(self, op: int, S: int, K: int = 0, V: int = 1, device=None):
        n = workspace_size(op, S, K, V)
        if n == 0:
            raise ValueError("invalid workspace request")
        self.buf = torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        self.nbytes = n

    @property
    def args(self):
        return ctypes.c_void_p(self.ptr), ctypes.c_size_t(self.nbytes)


def selftest_wait(ws: Workspace, limit_us: int, stream=None):
    """Runs the bounded waits against nothing; check_status(ws) then reports ERR_TIMEOUT."""
    w, n = ws.args
    _check(load().smcsd_selftest_wait(int(limit_us), w, n, _stream(stream)), "smcsd_selftest_wait")


def check_status(ws: Workspace, stream=None) -> int:
    """Wait for the stream; return (and clear) the first device-side error recorded in ws."""
    return int(load().smcsd_check_status(ctypes.c_void_p(ws.ptr), _stream(stream)))


def _out(t, shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device) if t is None else t


def sd_verify(tgt_logits, drf_logits, draft_tokens, S, K, V, temperature, uniforms,
              tgt_offsets=None, drf_offsets=None, ws=None, accept_len=None, out_token=None,
              lse_tgt=None, lse_drf=None, stream=None):
    """Returns (accept_len, out_token) int32 tensors [S]."""
    dev = tgt_logits.device
    ws = ws or Workspace(OP_SD_VERIFY, S, K, V, dev)
    accept_len = _out(accept_len, (S,), torch.int32, dev)
    out_token = _out(out_token, (S,), torch.int32, dev)
    w, n = ws.args
    rc = load().sd_verify(_ptr(tgt_logits), _ptr(drf_logits), _dtype_code(tgt_logits),
                          _ptr(draft_tokens), _ptr(tgt_offsets), _ptr(drf_offsets), S, K, V,
                          float(temperature), _ptr(uniforms), _ptr(accept_len), _ptr(out_token),
                          _ptr(lse_tgt), _ptr(lse_drf), w, n, _stream(stream))
    _check(rc, "sd_verify")
    return accept_len, out_token


def smc_reweight(tgt_logits, drf_logits, draft_tokens, S, K, V, temperature, alpha, uniforms,
                 logw, ws=None, bonus_token=None, lse_tgt=None, lse_drf=None, stream=None):
    """Updates logw in place; returns bonus_token int32 [S]."""
    dev = tgt_logits.device
    ws = ws or Workspace(OP_SMC_REWEIGHT, S, K, V, dev)
    bonus_token = _out(bonus_token, (S,), torch.int32, dev)
    w, n = ws.args
    rc = load().smc_reweight(_ptr(tgt_logits), _ptr(drf_logits), _dtype_code(tgt_logits),
                             _ptr(draft_tokens), S, K, V, float(temperature), float(alpha),
                             _ptr(uniforms), _ptr(logw), _ptr(bonus_token), _ptr(lse_tgt),
                             _ptr(lse_drf), w, n, _stream(stream))
    _check(rc, "smc_reweight")
    return bonus_token


def smc_reweight_tilted(tgt_logits, drf_logits, draft_tokens, S, K, V, temperature, alpha,
                        uniforms, logw, target=TARGET_SEQUENCE, log_reward=None,
                        reward_scale=0.0, ws=None, bonus_token=None, lse_tgt=None, lse_drf=None,
                        stream=None):
    """smc_reweight toward the per-position (TARGET_TOKEN) or whole-sequence (TARGET_SEQUENCE)
    power target, with an optional additive log-reward float32 [S]. Updates logw in place;
    returns bonus_token int32 [S]."""
    dev = tgt_logits.device
    ws = ws or Workspace(OP_SMC_REWEIGHT, S, K, V, dev)
    bonus_token = _out(bonus_token, (S,), torch.int32, dev)
    w, n = ws.args
    rc = load().smc_reweight_tilted(_ptr(tgt_logits), _ptr(drf_logits), _dtype_code(tgt_logits),
                                    _ptr(draft_tokens), S, K, V, float(temperature), float(alpha),
                                    int(target), _ptr(log_reward), float(reward_scale),
                                    _ptr(uniforms), _ptr(logw), _ptr(bonus_token), _ptr(lse_tgt),
                                    _ptr(lse_drf), w, n, _stream(stream))
    _check(rc, "smc_reweight_tilted")
    return bonus_token


def draft_sample(logits, R, V, temperature, uniforms, ws=None, tokens=None, logq=None, lse=None,
                 stream=None):
    """One token per row of logits [R, V] from softmax(z/T). Returns (tokens int32 [R], logq
    float [R] or None); pass logq=False to skip it, lse (float [R]) to get the normalisers."""
    dev = logits.device
    ws = ws or Workspace(OP_DRAFT_SAMPLE, R, 0, V, dev)
    tokens = _out(tokens, (R,), torch.int32, dev)
    if logq is None:
        logq = torch.empty(R, dtype=torch.float32, device=dev)
    elif logq is False:
        logq = None
    w, n = ws.args
    rc = load().draft_sample(_ptr(logits), _dtype_code(logits), R, V, float(temperature),
                             _ptr(uniforms), _ptr(tokens), _ptr(logq), _ptr(lse), w, n,
                             _stream(stream))
    _check(rc, "draft_sample")
    return tokens, logq


def smc_ess_resample(logw, G, N, ess_threshold, uniforms, ws=None, ancestors=None, ess=None,
                     resampled=None, stream=None):
    """Updates logw in place; returns (ancestors [G*N], ess [G], resampled [G])."""
    dev = logw.device
    ws = ws or Workspace(OP_ESS_RESAMPLE, G, 0, 1, dev)
    ancestors = _out(ancestors, (G * N,), torch.int32, dev)
    ess = _out(ess, (G,), torch.float32, dev)
    resampled = _out(resampled, (G,), torch.int32, dev)
    w, n = ws.args
    rc = load().smc_ess_resample(_ptr(logw), G, N, float(ess_threshold), _ptr(uniforms),
                                 _ptr(ancestors), _ptr(ess), _ptr(resampled), w, n, _stream(stream))
    _check(rc, "smc_ess_resample")
    return ancestors, ess, resampled


def kv_pagetable_remap(ancestors, resampled, G, N, table_in, pages_per_seq, num_pages=0,
                       table_out=None, refcount=None, with_refcount=True, ws=None, stream=None):
    """Returns (table_out, refcount or None)."""
    dev = table_in.device
    ws = ws or Workspace(OP_PAGETABLE_REMAP, G, 0, 1, dev)
    table_out = _out(table_out, table_in.shape, torch.int32, dev)
    if with_refcount and refcount is None:
        refcount = torch.empty(num_pages, dtype=torch.int32, device=dev)
    w, n = ws.args
    rc = load().kv_pagetable_remap(_ptr(ancestors), _ptr(resampled), G, N, _ptr(table_in),
                                   _ptr(table_out), pages_per_seq, _ptr(refcount), num_pages, w, n,
                                   _stream(stream))
    _check(rc, "kv_pagetable_remap")
    return table_out, refcount


def pacer_block_stop(hidden, w, c, S, b, max_blocks, d, t0, rho, ws=None, lengths=None,
                     block_scores=None, offsets=True, stream=None):
    """hidden bf16 [S, max_blocks*b, d], w bf16 [d]. Returns (lengths, block_scores,
    tgt_offsets, drf_offsets); the offsets are None when offsets=False."""
    return pacer_block_stop_pos(hidden, w, None, c, S, b, max_blocks, d, t0, rho, ws, lengths,
                                block_scores, offsets, stream)


def pacer_block_stop_pos(hidden, w, pos_emb, c, S, b, max_blocks, d, t0, rho, ws=None,
                         lengths=None, block_scores=None, offsets=True, stream=None):
    """pacer_block_stop with position embeddings pos_emb bf16 [max_blocks*b, d] (None: none)."""
    dev = hidden.device
    ws = ws or Workspace(OP_PACER_BLOCK_STOP, S, 0, 1, dev)
    lengths = _out(lengths, (S,), torch.int32, dev)
    block_scores = _out(block_scores, (S * max_blocks,), torch.float32, dev)
    to = torch.empty(S + 1, dtype=torch.int32, device=dev) if offsets else None
    do = torch.empty(S + 1, dtype=torch.int32, device=dev) if offsets else None
    wp, n = ws.args
    if pos_emb is None:
        rc = load().pacer_block_stop(_ptr(hidden), _ptr(w), float(c), S, b, max_blocks, d,
                                     float(t0), float(rho), _ptr(lengths), _ptr(block_scores),
                                     _ptr(to), _ptr(do), wp, n, _stream(stream))
    else:
        rc = load().pacer_block_stop_pos(_ptr(hidden), _ptr(w), _ptr(pos_emb), float(c), S, b,
                                         max_blocks, d, float(t0), float(rho), _ptr(lengths),
                                         _ptr(block_scores), _ptr(to), _ptr(do), wp, n,
                                         _stream(stream))
    _check(rc, "pacer_block_stop")
    return lengths, block_scores, to, do


def _step_outputs(dev, G, N, table_in, num_pages, bonus_token, ancestors, ess, resampled,
                  table_out, refcount, with_refcount):
    S = G * N
    bonus_token = _out(bonus_token, (S,), torch.int32, dev)
    ancestors = _out(ancestors, (S,), torch.int32, dev)
    ess = _out(ess, (G,), torch.float32, dev)
    resampled = _out(resampled, (G,), torch.int32, dev)
    if table_in is not None:
        table_out = _out(table_out, table_in.shape, torch.int32, dev)
        if with_refcount and refcount is None:
            refcount = torch.empty(num_pages, dtype=torch.int32, device=dev)
    else:
        table_out = refcount = None
    return dict(bonus_token=bonus_token, ancestors=ancestors, ess=ess, resampled=resampled,
                table_out=table_out, refcount=refcount)


def smc_step_tilted(tgt_logits, drf_logits, draft_tokens, G, N, K, V, temperature, alpha,
                    bonus_uniforms, logw, ess_threshold, resample_uniforms, target=TARGET_SEQUENCE,
                    log_reward=None, reward_scale=0.0, table_in=None, pages_per_seq=0,
                    num_pages=0, ws=None, bonus_token=None, ancestors=None, ess=None,
                    resampled=None, table_out=None, refcount=None, with_refcount=True,
                    stream=None):
    """smc_step toward a tilted target (see smc_reweight_tilted). Updates logw in place.
    Returns a dict of output tensors."""
    dev = tgt_logits.device
    ws = ws or Workspace(OP_SMC_STEP, G * N, K, V, dev)
    o = _step_outputs(dev, G, N, table_in, num_pages, bonus_token, ancestors, ess, resampled,
                      table_out, refcount, with_refcount)
    w, n = ws.args
    rc = load().smc_step_tilted(_ptr(tgt_logits), _ptr(drf_logits), _dtype_code(tgt_logits),
                                _ptr(draft_tokens), G, N, K, V, float(temperature), float(alpha),
                                int(target), _ptr(log_reward), float(reward_scale),
                                _ptr(bonus_uniforms), _ptr(logw), _ptr(o["bonus_token"]),
                                float(ess_threshold), _ptr(resample_uniforms),
                                _ptr(o["ancestors"]), _ptr(o["ess"]), _ptr(o["resampled"]),
                                _ptr(table_in), _ptr(o["table_out"]), pages_per_seq,
                                _ptr(o["refcount"]), num_pages, w, n, _stream(stream))
    _check(rc, "smc_step_tilted")
    return o


def smc_step(tgt_logits, drf_logits, draft_tokens, G, N, K, V, temperature, alpha,
             bonus_uniforms, logw, ess_threshold, resample_uniforms, table_in=None,
             pages_per_seq=0, num_pages=0, ws=None, bonus_token=None, ancestors=None, ess=None,
             resampled=None, table_out=None, refcount=None, with_refcount=True, stream=None):
    """Fused SMC-SD step. Updates logw in place. Returns a dict of output tensors."""
    dev = tgt_logits.device
    S = G * N
    ws = ws or Workspace(OP_SMC_STEP, S, K, V, dev)
    bonus_token = _out(bonus_token, (S,), torch.int32, dev)
    ancestors = _out(ancestors, (S,), torch.int32, dev)
    ess = _out(ess, (G,), torch.float32, dev)
    resampled = _out(resampled, (G,), torch.int32, dev)
    if table_in is not None:
        table_out = _out(table_out, table_in.shape, torch.int32, dev)
        if with_refcount and refcount is None:
            refcount = torch.empty(num_pages, dtype=torch.int32, device=dev)
    else:
        table_out = refcount = None
    w, n = ws.args
    rc = load().smc_step(_ptr(tgt_logits), _ptr(drf_logits), _dtype_code(tgt_logits),
                         _ptr(draft_tokens), G, N, K, V, float(temperature), float(alpha),
                         _ptr(bonus_uniforms), _ptr(logw), _ptr(bonus_token), float(ess_threshold),
                         _ptr(resample_uniforms), _ptr(ancestors), _ptr(ess), _ptr(resampled),
                         _ptr(table_in), _ptr(table_out), pages_per_seq, _ptr(refcount), num_pages,
                         w, n, _stream(stream))
    _check(rc, "smc_step")
    return dict(bonus_token=bonus_token, ancestors=ancestors, ess=ess, resampled=resampled,
                table_out=table_out, refcount=refcount)


def smc_step_logq(tgt_logits, draft_tokens, drf_logq, G, N, K, V, temperature, alpha,
                  bonus_uniforms, logw, ess_threshold, resample_uniforms, table_in=None,
                  pages_per_seq=0, num_pages=0, ws=None, bonus_token=None, ancestors=None,
                  ess=None, resampled=None, table_out=None, refcount=None, with_refcount=True,
                  stream=None):
    """smc_step with the draft's log q(x_k) (float32 [G*N*K]) in place of the draft logits."""
    dev = tgt_logits.device
    S = G * N
    ws = ws or Workspace(OP_SMC_STEP, S, K, V, dev)
    bonus_token = _out(bonus_token, (S,), torch.int32, dev)
    ancestors = _out(ancestors, (S,), torch.int32, dev)
    ess = _out(ess, (G,), torch.float32, dev)
    resampled = _out(resampled, (G,), torch.int32, dev)
    if table_in is not None:
        table_out = _out(table_out, table_in.shape, torch.int32, dev)
        if with_refcount and refcount is None:
            refcount = torch.empty(num_pages, dtype=torch.int32, device=dev)
    else:
        table_out = refcount = None
    w, n = ws.args
    rc = load().smc_step_logq(_ptr(tgt_logits), _dtype_code(tgt_logits), _ptr(draft_tokens),
                              _ptr(drf_logq), G, N, K, V, float(temperature), float(alpha),
                              _ptr(bonus_uniforms), _ptr(logw), _ptr(bonus_token),
                              float(ess_threshold), _ptr(resample_uniforms), _ptr(ancestors),
                              _ptr(ess), _ptr(resampled), _ptr(table_in), _ptr(table_out),
                              pages_per_seq, _ptr(refcount), num_pages, w, n, _stream(stream))
    _check(rc, "smc_step_logq")
    return dict(bonus_token=bonus_token, ancestors=ancestors, ess=ess, resampled=resampled,
                table_out=table_out, refcount=refcount)


STATIC_SCRATCH_BYTES = 32 << 20


def smc_step_static(tgt_logits, drf_logits, draft_tokens, G, N, K, V, temperature, alpha,
                    bonus_uniforms, logw, ess_threshold, resample_uniforms, table_in=None,
                    pages_per_seq=0, num_pages=0, bonus_token=None, ancestors=None, ess=None,
                    resampled=None, table_out=None, refcount=None, with_refcount=True,
                    status=None, stream=None):
    """smc_step on the library's own scratch area (no workspace argument). Output tensors must
    be passed in by a caller that cannot allocate; missing ones are allocated here for
    convenience. `status` (int32 [1] on the device) receives the call's device-side status."""
    dev = tgt_logits.device
    S = G * N
    bonus_token = _out(bonus_token, (S,), torch.int32, dev)
    ancestors = _out(ancestors, (S,), torch.int32, dev)
    ess = _out(ess, (G,), torch.float32, dev)
    resampled = _out(resampled, (G,), torch.int32, dev)
    if table_in is not None:
        table_out = _out(table_out, table_in.shape, torch.int32, dev)
        if with_refcount and refcount is None:
            refcount = torch.empty(num_pages, dtype=torch.int32, device=dev)
    else:
        table_out = refcount = None
    rc = load().smc_step_static(_ptr(tgt_logits), _ptr(drf_logits), _dtype_code(tgt_logits),
                                _ptr(draft_tokens), G, N, K, V, float(temperature), float(alpha),
                                _ptr(bonus_uniforms), _ptr(logw), _ptr(bonus_token),
                                float(ess_threshold), _ptr(resample_uniforms), _ptr(ancestors),
                                _ptr(ess), _ptr(resampled), _ptr(table_in), _ptr(table_out),
                                pages_per_seq, _ptr(refcount), num_pages, _ptr(status),
                                _stream(stream))
    _check(rc, "smc_step_static")
    return dict(bonus_token=bonus_token, ancestors=ancestors, ess=ess, resampled=resampled,
                table_out=table_out, refcount=refcount)
