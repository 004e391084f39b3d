"""GPU parity of draft_sample ("Faster LLM Inference via Sequential Monte Carlo", sec. 2 step 1:
each draft token drawn from the draft's tempered distribution) against the float64 oracle
through the C ABI: tokens by the decision rule, log q and normalisers within 1e-4; then the
drawn drafts verified against an identical target are all accepted."""
import numpy as np
import pytest
import torch

import oracle
from smc_reweight_resample_gb300 import synth
from gpu_util import DecisionLedger, FLOAT_ATOL, dev, dev_logits, host

pytestmark = pytest.mark.gpu


def check_draft(smcsd, z, R, V, T, u, ledger):
    lse = torch.full((R,), float("nan"), device="cuda")
    ws = smcsd.Workspace(smcsd.OP_DRAFT_SAMPLE, R, 0, V)
    tok, logq = smcsd.draft_sample(dev_logits(z), R, V, T, dev(u), ws=ws, lse=lse)
    assert smcsd.check_status(ws) == 0
    o = oracle.draft_sample(z, R, V, T, u)
    ledger.compare("draft_token", host(tok), o["tokens"], o["margin"])
    same = host(tok) == o["tokens"]
    np.testing.assert_allclose(host(logq)[same], o["logq"][same], atol=FLOAT_ATOL, rtol=0)
    np.testing.assert_allclose(host(lse), o["lse"], atol=FLOAT_ATOL, rtol=0)
    return host(tok)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V,T", [(5003, 1.0), (32000, 0.7), (1000, 1.3), (7, 1.0)])
def test_draft_sample_small(smcsd, dtype, V, T):
    L = DecisionLedger()
    R = 24
    _, drf = synth.logits_pair(40 + V, R, 1, V, 3.0, 1.0, dtype)
    drf = drf[:R]
    check_draft(smcsd, drf, R, V, T, synth.uniforms(41, R), L)
    L.finish()


def test_draft_sample_full_size(smcsd):
    """The 512 draft rows of the 8 x 16 particle, K=4, V=128256 bf16 step."""
    cfg = synth.SMC_LLAMA3
    x = synth.smc_step_inputs(cfg, 0, 0)
    R = cfg.S * cfg.K
    L = DecisionLedger()
    check_draft(smcsd, x.drf, R, cfg.V, cfg.temperature, synth.uniforms(42, R), L)
    L.finish()


def test_drafted_tokens_accepted_by_identical_target(smcsd):
    S, K, V = 16, 4, 32000
    c = synth.sd_case(43, S, K, V, 3.0, 1.0)
    tok, _ = smcsd.draft_sample(dev_logits(c.drf), S * K, V, 1.0, dev(synth.uniforms(44, S * K)))
    tgt = c.tgt.reshape(S, K + 1, V).copy()
    tgt[:, :K] = c.drf.reshape(S, K, V)
    acc, _ = smcsd.sd_verify(dev_logits(tgt.reshape(S * (K + 1), V)), dev_logits(c.drf), tok, S, K,
                             V, 1.0, dev(c.uniforms))
    assert (host(acc) == K).all()


def test_masked_row_is_reported(smcsd):
    R, V = 4, 4096
    z = np.random.default_rng(0).normal(0, 1, (R, V)).astype(np.float32)
    z[2] = -np.inf
    ws = smcsd.Workspace(smcsd.OP_DRAFT_SAMPLE, R, 0, V)
    smcsd.draft_sample(dev(z), R, V, 1.0, dev(synth.uniforms(0, R)), ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_NONFINITE
