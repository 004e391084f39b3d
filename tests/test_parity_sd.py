"""GPU parity of sd_verify (speculative-decoding verify; "Faster LLM Inference via Sequential
Monte Carlo", sec. 1, ragged lengths from "PACER", Methodik 2) against the float64 oracle,
called through the C ABI on the seeded workloads and on edge shapes."""
import numpy as np
import pytest
import torch

import oracle
from smc_reweight_resample_gb300 import synth
from gpu_util import DecisionLedger, FLOAT_ATOL, dev, dev_logits, host

pytestmark = pytest.mark.gpu


def run_sd(smcsd, c, ledger, unaligned=False):
    S, K, V = c.S, c.K, c.V
    t = dev_logits(c.tgt)
    d = dev_logits(c.drf) if c.drf.size else dev_logits(np.zeros((1, V), c.tgt.dtype))
    if unaligned:  # shift the rows off 16-byte alignment: scalar-load path
        t = torch.cat([t.reshape(-1)[:1], t.reshape(-1)])[1:].reshape(t.shape)
        assert t.data_ptr() % 16 != 0
    toks = dev(c.draft_tokens) if c.draft_tokens.size else dev(np.zeros(1, np.int32))
    u = dev(c.uniforms)
    to = dev(c.tgt_offsets) if c.tgt_offsets is not None else None
    do = dev(c.drf_offsets) if c.drf_offsets is not None else None
    lse_t = torch.full((c.tgt.shape[0],), float("nan"), device="cuda")
    lse_d = torch.full((max(c.drf.shape[0], 1),), float("nan"), device="cuda")
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, S, K, V)
    acc, tok = smcsd.sd_verify(t, d, toks, S, K, V, c.temperature, u, to, do, ws=ws,
                               lse_tgt=lse_t, lse_drf=lse_d)
    assert smcsd.check_status(ws) == 0
    o = oracle.sd_verify(c.tgt, c.drf if c.drf.size else np.zeros((1, V), c.tgt.dtype),
                         c.draft_tokens if c.draft_tokens.size else np.zeros(1, np.int32), S, K, V,
                         c.temperature, c.uniforms, c.tgt_offsets, c.drf_offsets,
                         threads=oracle.default_threads())
    ga, gt = host(acc), host(tok)
    oa, ot = o["accept_len"], o["out_token"]
    if K > 0:
        am = o["accept_margin"].reshape(S, K)
        kf = np.minimum(np.minimum(ga, oa), K - 1)
        margin = np.where(ga == oa, 1.0, am[np.arange(S), kf])
    else:
        margin = np.ones(S)
    ledger.compare("accept_len", ga, oa, margin)
    same = ga == oa
    ledger.compare("out_token", gt[same], ot[same], o["token_margin"][same])
    np.testing.assert_allclose(host(lse_t), o["lse_tgt"], atol=FLOAT_ATOL, rtol=0)
    if c.drf.size:
        np.testing.assert_allclose(host(lse_d)[: c.drf.shape[0]], o["lse_drf"][: c.drf.shape[0]],
                                   atol=FLOAT_ATOL, rtol=0)
    return ga, gt


def test_sd_tiny_fp32_many_seeds(smcsd):
    L = DecisionLedger()
    for seed in range(24):
        run_sd(smcsd, synth.sd_tiny(seed), L)
    L.finish()


@pytest.mark.parametrize("K", [2, 4, 6])
def test_sd_mistral_vocab(smcsd, K):
    L = DecisionLedger()
    for seed in range(3):
        run_sd(smcsd, synth.sd_mistral(seed, K), L)
    L.finish()


@pytest.mark.parametrize("V", [1, 7, 8, 1000, 2048, 2049, 32003])
@pytest.mark.parametrize("K", [1, 3, 8])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_sd_edge_shapes(smcsd, V, K, dtype):
    L = DecisionLedger()
    for seed in range(2):
        c = synth.sd_case(100 + seed, 5, K, V, 3.0, 1.0, 0.8, dtype)
        run_sd(smcsd, c, L)
    L.finish()


def test_sd_unaligned_rows_use_scalar_path(smcsd):
    L = DecisionLedger()
    run_sd(smcsd, synth.sd_case(7, 6, 3, 4100, 3.0, 1.0, 1.0, "bf16"), L, unaligned=True)
    L.finish()


def test_sd_masked_tokens(smcsd):
    c = synth.sd_case(8, 8, 4, 5000, 3.0, 1.0)
    rng = np.random.default_rng(8)
    neg = synth.bf16_bits(np.array([-np.inf], np.float32))[0]
    for a in (c.tgt, c.drf):
        m = rng.random(a.shape) < 0.3
        a[m] = neg
    c.draft_tokens = synth.gumbel_draft_tokens(9, c.drf, c.V, 1.0)
    L = DecisionLedger()
    run_sd(smcsd, c, L)
    L.finish()


def test_sd_identical_models_accept_all(smcsd):
    S, K, V = 10, 5, 32000
    c = synth.sd_case(3, S, K, V, 3.0, 1.0)
    c.drf = c.tgt.reshape(S, K + 1, V)[:, :K].reshape(S * K, V).copy()
    L = DecisionLedger()
    ga, _ = run_sd(smcsd, c, L)
    assert (ga == K).all()
    L.finish()


def test_sd_ragged(smcsd):
    lengths = np.array([4, 8, 12, 16, 20, 4, 0, 7, 1, 20, 5, 9], np.int32)
    c = synth.ragged_sd_case(11, lengths, 32256, K_max=20)
    L = DecisionLedger()
    run_sd(smcsd, c, L)
    L.finish()


def test_sd_llama3_vocab_128_sequences(smcsd):
    """The benchmarked SD shape: 128 sequences, K=4, V=128256 bf16 (63 chunks per row in the
    final-token passes), two seeds."""
    L = DecisionLedger()
    for seed in range(2):
        run_sd(smcsd, synth.sd_case(40 + seed, 128, 4, 128256, 3.0, 1.0, 1.0, "bf16"), L)
    L.finish()


def test_sd_ragged_llama3_vocab(smcsd):
    """Ragged lengths 0..20 at V=128256."""
    lengths = np.array([4, 8, 12, 16, 20, 4, 0, 7, 1, 20, 5, 9, 13, 2, 17, 6], np.int32)
    c = synth.ragged_sd_case(12, lengths, 128256, K_max=20)
    L = DecisionLedger()
    run_sd(smcsd, c, L)
    L.finish()


def test_sd_two_calls_same_workspace_are_identical(smcsd):
    c = synth.sd_mistral(5, 4)
    t, d, toks, u = dev_logits(c.tgt), dev_logits(c.drf), dev(c.draft_tokens), dev(c.uniforms)
    ws = smcsd.Workspace(smcsd.OP_SD_VERIFY, c.S, c.K, c.V)
    a1, t1 = smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)
    a2, t2 = smcsd.sd_verify(t, d, toks, c.S, c.K, c.V, 1.0, u, ws=ws)
    assert smcsd.check_status(ws) == 0
    assert torch.equal(a1, a2) and torch.equal(t1, t2)
