"""GPU parity of the tilted SMC targets ("Faster LLM Inference via Sequential Monte Carlo",
sec. 3 "flexibility": power sampling and reward-weighted decoding; sec. 5: reward
optimisation): smc_reweight_tilted and smc_step_tilted against the float64 oracle through the
C ABI, for the whole-sequence power target prod p^alpha and the additive log-reward, at small
shapes, at the full workload sizes and over consecutive fused steps."""
import numpy as np
import pytest
import torch

import oracle
from smc_reweight_resample_gb300 import synth
from gpu_util import DecisionLedger, FLOAT_ATOL, dev, dev_logits, host
from test_parity_smc import compare_resample

pytestmark = pytest.mark.gpu


def check_tilted(smcsd, c, u, lw0, T, alpha, target, reward, scale, ledger):
    S, K, V = c.S, c.K, c.V
    lw = dev(lw0.copy())
    lse_t = torch.full((S * (K + 1),), float("nan"), device="cuda")
    lse_d = torch.full((max(S * K, 1),), float("nan"), device="cuda")
    ws = smcsd.Workspace(smcsd.OP_SMC_REWEIGHT, S, K, V)
    tok = smcsd.smc_reweight_tilted(dev_logits(c.tgt), dev_logits(c.drf), dev(c.draft_tokens), S,
                                    K, V, T, alpha, dev(u), lw, target=target,
                                    log_reward=None if reward is None else dev(reward),
                                    reward_scale=scale, ws=ws, lse_tgt=lse_t, lse_drf=lse_d)
    assert smcsd.check_status(ws) == 0
    o = oracle.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, T, alpha, u, lw0,
                                   target_mode=target, log_reward=reward, reward_scale=scale)
    np.testing.assert_allclose(host(lw), o["logw"], atol=FLOAT_ATOL, rtol=0)
    ledger.compare("bonus_token", host(tok), o["bonus_token"], o["bonus_margin"])
    np.testing.assert_allclose(host(lse_t), o["lse_tgt"], atol=FLOAT_ATOL, rtol=0)
    if K > 0:
        np.testing.assert_allclose(host(lse_d), o["lse_drf"], atol=FLOAT_ATOL, rtol=0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("T,alpha,with_reward", [(1.0, 2.0, False), (0.7, 4.0, True),
                                                 (1.3, 0.5, True), (1.0, 1.0, False)])
def test_sequence_target_small(smcsd, dtype, T, alpha, with_reward):
    L = DecisionLedger()
    for seed in range(3):
        S, K, V = 12, 3, 5003
        c = synth.sd_case(60 + seed, S, K, V, 3.0, 1.0, T, dtype)
        u = synth.uniforms(60 + seed, S, stream=7)
        lw0 = np.random.default_rng(seed).normal(0, 2, S).astype(np.float32)
        r = synth.log_rewards(seed, S) if with_reward else None
        check_tilted(smcsd, c, u, lw0, T, alpha, smcsd.TARGET_SEQUENCE, r, 0.6, L)
    L.finish()


def test_reward_on_per_position_target(smcsd):
    L = DecisionLedger()
    S, K, V = 16, 4, 32000
    c = synth.sd_case(70, S, K, V, 3.0, 1.0, 0.7)
    u = synth.uniforms(70, S, stream=7)
    lw0 = np.zeros(S, np.float32)
    check_tilted(smcsd, c, u, lw0, 0.7, 4.0, smcsd.TARGET_TOKEN, synth.log_rewards(70, S), -1.5, L)
    L.finish()


def test_sequence_target_edge_shapes(smcsd):
    """K = 0 (the step is the (K+1)-th token alone), one particle, and a vocabulary that is not a
    multiple of the chunk with unaligned rows (the scalar path)."""
    L = DecisionLedger()
    for S, K, V in ((5, 0, 4099), (1, 2, 1000), (7, 2, 3001)):
        c = synth.sd_case(80 + V, S, K, V, 3.0, 1.0, 0.9)
        u = synth.uniforms(80 + V, S, stream=7)
        lw0 = np.random.default_rng(V).normal(0, 1, S).astype(np.float32)
        check_tilted(smcsd, c, u, lw0, 0.9, 3.0, smcsd.TARGET_SEQUENCE, synth.log_rewards(V, S),
                     0.5, L)
    L.finish()


def test_alpha_one_sequence_target_equals_smc_reweight(smcsd):
    S, K, V = 32, 4, 20000
    c = synth.sd_case(90, S, K, V, 3.0, 1.0)
    u = dev(synth.uniforms(90, S, stream=7))
    lw0 = np.random.default_rng(9).normal(0, 1, S).astype(np.float32)
    t, d, x = dev_logits(c.tgt), dev_logits(c.drf), dev(c.draft_tokens)
    lw_a, lw_b = dev(lw0.copy()), dev(lw0.copy())
    ta = smcsd.smc_reweight(t, d, x, S, K, V, 1.0, 1.0, u, lw_a)
    tb = smcsd.smc_reweight_tilted(t, d, x, S, K, V, 1.0, 1.0, u, lw_b, target=smcsd.TARGET_SEQUENCE)
    assert torch.equal(ta, tb)
    assert torch.equal(lw_a, lw_b)


@pytest.mark.parametrize("cfg", [synth.SMC_LLAMA3, synth.SMC_QWEN_POWER], ids=lambda c: c.name)
def test_sequence_target_full_size(smcsd, cfg):
    x = synth.smc_step_inputs(cfg, 0, 0)
    c = synth.SDCase(cfg.S, cfg.K, cfg.V, cfg.temperature, x.tgt, x.drf, x.draft_tokens,
                     x.bonus_uniforms)
    lw0 = np.random.default_rng(2).normal(0, 1, cfg.S).astype(np.float32)
    L = DecisionLedger()
    check_tilted(smcsd, c, x.bonus_uniforms, lw0, cfg.temperature, cfg.alpha,
                 smcsd.TARGET_SEQUENCE, synth.log_rewards(3, cfg.S), 0.25, L)
    L.finish()


def run_tilted_steps(smcsd, cfg, steps, target, scale, seed=0):
    """Fused tilted steps; each step the oracle starts from the GPU's state (teacher-forced)."""
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    ws = smcsd.Workspace(smcsd.OP_SMC_STEP, S, K, V)
    lw = torch.zeros(S, dtype=torch.float32, device="cuda")
    table = dev(synth.initial_page_table(S, P))
    L = DecisionLedger()
    resampled_any = False
    for step in range(steps):
        x = synth.smc_step_inputs(cfg, seed, step)
        r = synth.log_rewards(seed * 1000 + step, S)
        lw_before, table_before = host(lw).copy(), host(table).copy()
        out = smcsd.smc_step_tilted(dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens), G, N,
                                    K, V, cfg.temperature, cfg.alpha, dev(x.bonus_uniforms), lw,
                                    cfg.ess_threshold, dev(x.resample_uniforms), target=target,
                                    log_reward=dev(r), reward_scale=scale, table_in=table,
                                    pages_per_seq=P, num_pages=S * P, ws=ws)
        assert smcsd.check_status(ws) == 0
        o = oracle.smc_reweight_tilted(x.tgt, x.drf, x.draft_tokens, S, K, V, cfg.temperature,
                                       cfg.alpha, x.bonus_uniforms, lw_before, target_mode=target,
                                       log_reward=r, reward_scale=scale)
        L.compare("bonus_token", host(out["bonus_token"]), o["bonus_token"], o["bonus_margin"])
        rs = oracle.ess_resample(o["logw"], G, N, cfg.ess_threshold, x.resample_uniforms)
        compare_resample(L, host(out["ancestors"]), host(out["ess"]), host(out["resampled"]),
                         host(lw), rs, N)
        resampled_any |= bool(host(out["resampled"]).any())
        m = oracle.pagetable_remap(host(out["ancestors"]), host(out["resampled"]), G, N,
                                   table_before, P, num_pages=S * P)
        np.testing.assert_array_equal(host(out["table_out"]), m["table_out"])
        np.testing.assert_array_equal(host(out["refcount"]), m["refcount"])
        table = out["table_out"]
    L.finish()
    return resampled_any


@pytest.mark.parametrize("GN", [(8, 16), (3, 48)], ids=["groups_of_16", "groups_of_48"])
def test_tilted_step_teacher_forced(smcsd, GN):
    G, N = GN
    cfg = synth.SMCConfig("smc_tilted", G, N, 4, 8192, 3.0, 1.0, 0.8, 2.0, 256)
    assert run_tilted_steps(smcsd, cfg, 8, smcsd.TARGET_SEQUENCE, 0.5)


def test_tilted_step_full_size(smcsd):
    run_tilted_steps(smcsd, synth.SMC_LLAMA3, 2, smcsd.TARGET_SEQUENCE, 0.5)


def test_non_finite_reward_is_reported(smcsd):
    S, K, V = 4, 2, 4096
    c = synth.sd_case(95, S, K, V, 3.0, 1.0)
    r = np.array([0.0, np.nan, 1.0, 0.0], np.float32)
    ws = smcsd.Workspace(smcsd.OP_SMC_REWEIGHT, S, K, V)
    smcsd.smc_reweight_tilted(dev_logits(c.tgt), dev_logits(c.drf), dev(c.draft_tokens), S, K, V,
                              1.0, 2.0, dev(synth.uniforms(95, S)), torch.zeros(S, device="cuda"),
                              log_reward=dev(r), reward_scale=1.0, ws=ws)
    assert smcsd.check_status(ws) == smcsd.ERR_NONFINITE
    assert smcsd.check_status(ws) == 0  # cleared by the check
