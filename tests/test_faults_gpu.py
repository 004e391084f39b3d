"""Device-side error reporting without any GPU fault: bad data is flagged in the workspace and
read back with smcsd_check_status; host-side argument errors return before anything is
enqueued."""
import numpy as np
import pytest
import torch

from smc_reweight_resample_gb300 import synth
from gpu_util import dev, dev_logits, host

pytestmark = pytest.mark.gpu


def _sd_inputs(seed=0):
    c = synth.sd_case(seed, 4, 3, 3000, 3.0, 1.0)
    return c, dev_logits(c.tgt), dev_logits(c.drf), dev(c.draft_tokens), dev(c.uniforms)


def test_nan_logit_reports_nonfinite(smcsd):
    c, t, d, toks, u = _sd_inputs()
    t.view(torch.int16).view(-1)[5 * c.V + 17] = 0x7FC0  # a NaN in target row 5
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, c.S, c.K, c.V)
    smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_NONFINITE
    assert smcsd.check_status(ws) == 0  # cleared by the read
    # the workspace is still usable
    _, t2, _, _, _ = _sd_inputs()
    smcsd.sd_verify(t2, d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)
    assert smcsd.check_status(ws) == 0


def test_all_masked_row_reports_nonfinite(smcsd):
    c, t, d, toks, u = _sd_inputs()
    t.view(torch.int16).view(-1)[2 * c.V: 3 * c.V] = -128  # 0xFF80 = -inf
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, c.S, c.K, c.V)
    smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_NONFINITE


def test_token_out_of_range(smcsd):
    c, t, d, toks, u = _sd_inputs()
    toks[3] = c.V + 5
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, c.S, c.K, c.V)
    smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_RANGE


def test_bad_ragged_offsets(smcsd):
    c, t, d, toks, u = _sd_inputs()
    to = dev(np.array([0, 4, 5, 9, 12], np.int32))   # sequence 1: 1 target row ...
    do = dev(np.array([0, 3, 5, 8, 11], np.int32))   # ... but 2 draft rows
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, c.S, c.K, c.V)
    smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, to, do, ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_RANGE


def test_remap_bad_page_id(smcsd):
    G, N, P = 2, 4, 8
    table = np.arange(G * N * P, dtype=np.int32)
    table[7] = 10_000
    ws = smcsd.Workspace(smcsd.OP_PAGETABLE_REMAP, G)
    smcsd.kv_pagetable_remap(dev(np.zeros(G * N, np.int32)), None, G, N, dev(table), P,
                             num_pages=G * N * P, ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_RANGE


def test_nan_weight(smcsd):
    lw = dev(np.array([0.0, np.nan, 0.0, 0.0], np.float32))
    ws = smcsd.Workspace(smcsd.OP_ESS_RESAMPLE, 1)
    smcsd.smc_ess_resample(lw, 1, 4, 2.0, dev(np.zeros(1, np.float32)), ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_NONFINITE


def test_host_argument_errors(smcsd):
    c, t, d, toks, u = _sd_inputs()
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, c.S, c.K, c.V)
    with pytest.raises(smcsd.SMCSDError) as e:
        smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 0.0, u, ws=ws)
    assert e.value.code == smcsd.ERR_INVALID_ARG
    small = smcsd.Workspace(smcsd.OP_SD_VERIFY, 1, 1, 1)
    with pytest.raises(smcsd.SMCSDError) as e:
        smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, ws=small)
    assert e.value.code == smcsd.ERR_WORKSPACE
    with pytest.raises(TypeError):
        smcsd.sd_verify(t.to(torch.float16), d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)


def test_bounded_wait_runs_out_and_the_context_survives(smcsd):
    """The pipeline's waits, run against a barrier and a slot tag that nothing completes, give
    up after their limit and record ERR_TIMEOUT; the workspace and the context then serve a
    normal verify, which matches the oracle."""
    import time

    import oracle

    c, t, d, toks, u = _sd_inputs(3)
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, c.S, c.K, c.V)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    smcsd.selftest_wait(ws, 20000)  # 20 ms per wait
    assert smcsd.check_status(ws) == smcsd.ERR_TIMEOUT
    dt = time.perf_counter() - t0
    assert 0.035 <= dt < 2.0, dt  # both waits ran their 20 ms, and no longer than a bound
    assert smcsd.check_status(ws) == 0
    acc, tok = smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)
    assert smcsd.check_status(ws) == 0
    o = oracle.sd_verify(c.tgt, c.drf, c.draft_tokens, c.S, c.K, c.V, 1.0, c.uniforms)
    np.testing.assert_array_equal(host(acc), o["accept_len"])
    np.testing.assert_array_equal(host(tok), o["out_token"])
