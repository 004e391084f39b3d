"""GPU parity of smc_step_logq ("Faster LLM Inference via Sequential Monte Carlo", sec. 2 steps 1
and 3: the draft proposes each token from its own distribution, and the weight needs only the
probability the draft gave it): the draft sampler's tokens and log q, drawn on the GPU, feed a
step that reads the target logits only; the float64 oracle reweights the same tokens from the
full draft logits. Log-weights within 1e-4, bonus tokens, resampling flags and ancestors by the
decision rule, page tables and refcounts exact."""
import numpy as np
import pytest
import torch

import oracle
from smc_reweight_resample_gb300 import synth
from gpu_util import DecisionLedger, FLOAT_ATOL, dev, dev_logits, host

pytestmark = pytest.mark.gpu


def run_logq_steps(smcsd, cfg, steps, seed):
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    ws = smcsd.Workspace(smcsd.OP_SMC_STEP, S, K, V)
    wsd = smcsd.Workspace(smcsd.OP_DRAFT_SAMPLE, S * K, 0, V)
    lw = torch.from_numpy(np.random.default_rng(seed).normal(0, 1, S).astype(np.float32)).cuda()
    table = dev(synth.initial_page_table(S, P))
    L = DecisionLedger()
    nthr = oracle.default_threads()
    for step in range(steps):
        x = synth.smc_step_inputs(cfg, seed, step)
        ud = synth.uniforms(seed, S * K, stream=900 + step)
        toks, logq = smcsd.draft_sample(dev_logits(x.drf), S * K, V, cfg.temperature, dev(ud), ws=wsd)
        assert smcsd.check_status(wsd) == 0
        lw_before = host(lw).copy()
        table_before = host(table).copy()
        out = smcsd.smc_step_logq(dev_logits(x.tgt), toks, logq, G, N, K, V, cfg.temperature,
                                  cfg.alpha, dev(x.bonus_uniforms), lw, cfg.ess_threshold,
                                  dev(x.resample_uniforms), table_in=table, pages_per_seq=P,
                                  num_pages=S * P, ws=ws)
        assert smcsd.check_status(ws) == 0
        o = oracle.smc_reweight(x.tgt, x.drf, host(toks), S, K, V, cfg.temperature, cfg.alpha,
                                x.bonus_uniforms, lw_before, threads=nthr)
        L.compare("bonus_token", host(out["bonus_token"]), o["bonus_token"], o["bonus_margin"])
        r = oracle.ess_resample(o["logw"], G, N, cfg.ess_threshold, x.resample_uniforms)
        L.compare("resampled", host(out["resampled"]), r["resampled"], r["ess_margin"])
        np.testing.assert_allclose(host(out["ess"]), r["ess"], rtol=1e-5, atol=0)
        for g in np.nonzero(host(out["resampled"]) == r["resampled"])[0]:
            sl = slice(g * N, (g + 1) * N)
            m = r["anc_margin"][sl] if r["resampled"][g] else np.ones(N)
            L.compare("ancestors", host(out["ancestors"])[sl], r["ancestors"][sl], m)
            np.testing.assert_allclose(host(lw)[sl], r["logw"][sl], atol=FLOAT_ATOL, rtol=0)
        m = oracle.pagetable_remap(host(out["ancestors"]), host(out["resampled"]), G, N,
                                   table_before, P, num_pages=S * P)
        np.testing.assert_array_equal(host(out["table_out"]), m["table_out"])
        np.testing.assert_array_equal(host(out["refcount"]), m["refcount"])
        table = out["table_out"]
    L.finish()


def test_logq_step_small_several_steps(smcsd):
    cfg = synth.SMCConfig("logq_small", 6, 16, 3, 20000, 3.0, 1.0, 0.9, 1.0, 256)
    run_logq_steps(smcsd, cfg, 4, 7)


def test_logq_step_power_target(smcsd):
    cfg = synth.SMCConfig("logq_power", 3, 32, 2, 5003, 3.0, 1.5, 0.7, 4.0, 128)
    run_logq_steps(smcsd, cfg, 2, 8)


def test_logq_step_full_size(smcsd):
    """The 8 x 16 particle, K=4, V=128256 bf16 step, two consecutive steps."""
    run_logq_steps(smcsd, synth.SMC_LLAMA3, 2, 9)


def test_logq_equals_logits_when_log_q_is_exact(smcsd):
    """With the draft rows' log q computed by the step itself (smc_reweight's normalisers at the
    draft tokens), the two entry points agree within float rounding of log q."""
    cfg = synth.SMCConfig("logq_eq", 4, 16, 4, 8192, 3.0, 1.0, 1.0, 1.0, 128)
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    x = synth.smc_step_inputs(cfg, 10, 0)
    lse_d = torch.empty(S * K, device="cuda")
    tok = smcsd.smc_reweight(dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens), S, K, V,
                             1.0, 1.0, dev(x.bonus_uniforms), torch.zeros(S, device="cuda"),
                             lse_drf=lse_d)
    zd = synth.widen(x.drf).reshape(S * K, V)[np.arange(S * K), x.draft_tokens].astype(np.float32)
    logq = dev((zd - host(lse_d)).astype(np.float32))
    lw_a, lw_b = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
    table = dev(synth.initial_page_table(S, P))
    a = smcsd.smc_step(dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens), G, N, K, V, 1.0,
                       1.0, dev(x.bonus_uniforms), lw_a, N / 2.0, dev(x.resample_uniforms),
                       table_in=table, pages_per_seq=P, num_pages=S * P)
    b = smcsd.smc_step_logq(dev_logits(x.tgt), dev(x.draft_tokens), logq, G, N, K, V, 1.0, 1.0,
                            dev(x.bonus_uniforms), lw_b, N / 2.0, dev(x.resample_uniforms),
                            table_in=table, pages_per_seq=P, num_pages=S * P)
    assert torch.equal(a["bonus_token"], b["bonus_token"])
    np.testing.assert_allclose(host(a["ess"]), host(b["ess"]), rtol=1e-5)
    np.testing.assert_allclose(host(lw_a), host(lw_b), atol=1e-5, rtol=0)


def test_logq_needs_log_q(smcsd):
    t = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(8, dtype=torch.int32, device="cuda")
    f32 = torch.zeros(8, device="cuda")
    with pytest.raises(smcsd.SMCSDError) as e:
        smcsd.smc_step_logq(t, i32, None, 1, 4, 1, 2, 1.0, 1.0, f32, f32, 2.0, f32)
    assert e.value.code == smcsd.ERR_INVALID_ARG
