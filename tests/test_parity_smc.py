"""GPU parity of the SMC-SD path ("Faster LLM Inference via Sequential Monte Carlo", sec. 2
steps 3-4 and sec. 3): smc_reweight, smc_ess_resample, kv_pagetable_remap and the fused
smc_step, against the float64 oracle through the C ABI, at the full workload sizes and over
32 consecutive steps."""
import numpy as np
import pytest
import torch

import oracle
from smc_reweight_resample_gb300 import synth
from gpu_util import DecisionLedger, FLOAT_ATOL, dev, dev_logits, host

pytestmark = pytest.mark.gpu


def reweight_case(smcsd, seed, S, K, V, T, alpha, sd=3.0, st=1.0, dtype="bf16"):
    c = synth.sd_case(seed, S, K, V, sd, st, T, dtype)
    u = synth.uniforms(seed, S, stream=7)
    lw0 = np.random.default_rng(seed).normal(0, 2, S).astype(np.float32)
    return c, u, lw0


def check_reweight(smcsd, c, u, lw0, T, alpha, ledger):
    S, K, V = c.S, c.K, c.V
    lw = dev(lw0.copy())
    lse_t = torch.full((S * (K + 1),), float("nan"), device="cuda")
    lse_d = torch.full((max(S * K, 1),), float("nan"), device="cuda")
    ws = smcsd.Workspace(smcsd.OP_SMC_REWEIGHT, S, K, V)
    tok = smcsd.smc_reweight(dev_logits(c.tgt), dev_logits(c.drf), dev(c.draft_tokens), S, K, V, T,
                             alpha, dev(u), lw, ws=ws, lse_tgt=lse_t, lse_drf=lse_d)
    assert smcsd.check_status(ws) == 0
    o = oracle.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, T, alpha, u, lw0,
                            threads=oracle.default_threads())
    np.testing.assert_allclose(host(lw), o["logw"], atol=FLOAT_ATOL, rtol=0)
    ledger.compare("bonus_token", host(tok), o["bonus_token"], o["bonus_margin"])
    np.testing.assert_allclose(host(lse_t), o["lse_tgt"], atol=FLOAT_ATOL, rtol=0)
    np.testing.assert_allclose(host(lse_d), o["lse_drf"], atol=FLOAT_ATOL, rtol=0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("T,alpha", [(1.0, 1.0), (0.7, 4.0), (1.3, 0.5)])
def test_reweight_small(smcsd, dtype, T, alpha):
    L = DecisionLedger()
    for seed in range(3):
        c, u, lw0 = reweight_case(smcsd, 20 + seed, 12, 3, 5003, T, alpha, dtype=dtype)
        check_reweight(smcsd, c, u, lw0, T, alpha, L)
    L.finish()


def _full_inputs(cfg, seed, step=0):
    x = synth.smc_step_inputs(cfg, seed, step)
    c = synth.SDCase(cfg.S, cfg.K, cfg.V, cfg.temperature, x.tgt, x.drf, x.draft_tokens,
                     x.bonus_uniforms)
    return c, x


@pytest.mark.parametrize("cfg", [synth.SMC_LLAMA3, synth.SMC_QWEN_POWER], ids=lambda c: c.name)
def test_reweight_full_size(smcsd, cfg):
    c, x = _full_inputs(cfg, 0)
    lw0 = np.random.default_rng(1).normal(0, 1, cfg.S).astype(np.float32)
    L = DecisionLedger()
    check_reweight(smcsd, c, x.bonus_uniforms, lw0, cfg.temperature, cfg.alpha, L)
    L.finish()


def test_identical_models_keep_weights(smcsd):
    S, K, V = 16, 4, 32000
    c = synth.sd_case(2, S, K, V, 3.0, 1.0)
    drf = c.tgt.reshape(S, K + 1, V)[:, :K].reshape(S * K, V).copy()
    lw0 = np.random.default_rng(0).normal(0, 1, S).astype(np.float32)
    lw = dev(lw0.copy())
    smcsd.smc_reweight(dev_logits(c.tgt), dev_logits(drf), dev(c.draft_tokens), S, K, V, 1.0, 1.0,
                       dev(synth.uniforms(0, S)), lw)
    np.testing.assert_allclose(host(lw), lw0, atol=1e-5, rtol=0)


# ------------------------------------------------------------------------------------------
# ESS / systematic resampling / page-table remap
# ------------------------------------------------------------------------------------------

def compare_resample(ledger, g_anc, g_ess, g_res, g_lw, o, N):
    ledger.compare("resampled", g_res, o["resampled"], o["ess_margin"])
    np.testing.assert_allclose(g_ess, o["ess"], rtol=1e-5, atol=0)
    G = g_res.size
    same = g_res == o["resampled"]
    for g in np.nonzero(same)[0]:
        sl = slice(g * N, (g + 1) * N)
        m = o["anc_margin"][sl] if o["resampled"][g] else np.ones(N)
        ledger.compare("ancestors", g_anc[sl], o["ancestors"][sl], m)
        np.testing.assert_allclose(g_lw[sl], o["logw"][sl], atol=FLOAT_ATOL, rtol=0)


@pytest.mark.parametrize("G,N", [(8, 16), (4, 64), (50, 33), (3, 1000), (1, 1)])
def test_ess_resample(smcsd, G, N):
    L = DecisionLedger()
    rng = np.random.default_rng(G * 1000 + N)
    for trial in range(4):
        lw0 = (rng.normal(0, 1.5, G * N) - 3.0 * trial).astype(np.float32)
        if trial == 3:
            lw0[rng.random(G * N) < 0.3] = -np.inf
            lw0[::N] = 0.0
        U = synth.uniforms(trial, G, stream=5)
        for thr in (0.0, N / 2.0, N + 1.0):
            lw = dev(lw0.copy())
            anc, ess, res = smcsd.smc_ess_resample(lw, G, N, thr, dev(U))
            o = oracle.ess_resample(lw0, G, N, thr, U)
            compare_resample(L, host(anc), host(ess), host(res), host(lw), o, N)
    L.finish()


@pytest.mark.parametrize("N", [5, 16, 32])
def test_ess_resample_on_decision_boundaries(smcsd, N):
    """Equal log-weights put the ESS exactly on a threshold of N and, with U = 0, every C_i on a
    point (j + U) / N of the systematic grid: groups of at most one warp then leave their float
    first attempt for the double-float path, which must still take the exact decisions."""
    G = 3
    for thr, U0 in ((float(N), 0.5), (N + 1.0, 0.0), (N + 1.0, 0.5)):
        lw0 = np.zeros(G * N, np.float32)
        U = np.full(G, U0, np.float32)
        lw = dev(lw0.copy())
        anc, ess, res = smcsd.smc_ess_resample(lw, G, N, thr, dev(U))
        o = oracle.ess_resample(lw0, G, N, thr, U)
        np.testing.assert_array_equal(host(res), o["resampled"])
        np.testing.assert_array_equal(host(anc), o["ancestors"])
        np.testing.assert_allclose(host(ess), o["ess"], rtol=1e-6, atol=0)
        np.testing.assert_allclose(host(lw), o["logw"], atol=0, rtol=0)


def test_remap(smcsd):
    G, N, P = 8, 16, 128
    rng = np.random.default_rng(4)
    table = rng.permutation(G * N * P).astype(np.int32)
    table[rng.random(table.size) < 0.05] = -1
    anc = np.sort(rng.integers(0, N, (G, N)), axis=1).astype(np.int32).reshape(-1)
    res = (rng.random(G) < 0.5).astype(np.int32)
    tout, rc = smcsd.kv_pagetable_remap(dev(anc), dev(res), G, N, dev(table), P, num_pages=G * N * P)
    o = oracle.pagetable_remap(anc, res, G, N, table, P, num_pages=G * N * P)
    np.testing.assert_array_equal(host(tout), o["table_out"])
    np.testing.assert_array_equal(host(rc), o["refcount"])
    # resampled = NULL means every group takes its ancestors
    tout, rc = smcsd.kv_pagetable_remap(dev(anc), None, G, N, dev(table), P, num_pages=G * N * P)
    o = oracle.pagetable_remap(anc, None, G, N, table, P, num_pages=G * N * P)
    np.testing.assert_array_equal(host(tout), o["table_out"])
    np.testing.assert_array_equal(host(rc), o["refcount"])


# ------------------------------------------------------------------------------------------
# fused step, 32 steps
# ------------------------------------------------------------------------------------------

def small_cfg(V=8192):
    return synth.SMCConfig("smc_small", 8, 16, 4, V, 3.0, 1.0, 1.0, 1.0, 256)


def run_steps(smcsd, cfg, steps, seed=0, teacher_forced=True):
    """Runs `steps` fused GPU steps; each step the oracle starts from the GPU's state
    (teacher-forced) and every output is compared. Also tracks a free-running oracle and
    returns the first step at which its decisions diverge (None if never)."""
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    ws = smcsd.Workspace(smcsd.OP_SMC_STEP, S, K, V)
    lw = torch.zeros(S, dtype=torch.float32, device="cuda")
    table = dev(synth.initial_page_table(S, P))
    lw_free = np.zeros(S, np.float32)
    table_free = synth.initial_page_table(S, P)
    first_div = None
    nthr = oracle.default_threads()
    L = DecisionLedger()
    for step in range(steps):
        x = synth.smc_step_inputs(cfg, seed, step)
        lw_before = host(lw).copy()
        table_before = host(table).copy()
        out = smcsd.smc_step(dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens), G, N, K, V,
                             cfg.temperature, cfg.alpha, dev(x.bonus_uniforms), lw,
                             cfg.ess_threshold, dev(x.resample_uniforms), table_in=table,
                             pages_per_seq=P, num_pages=S * P, ws=ws)
        assert smcsd.check_status(ws) == 0
        # teacher-forced oracle step from the GPU's state
        o = oracle.smc_reweight(x.tgt, x.drf, x.draft_tokens, S, K, V, cfg.temperature, cfg.alpha,
                                x.bonus_uniforms, lw_before, threads=nthr)
        L.compare("bonus_token", host(out["bonus_token"]), o["bonus_token"], o["bonus_margin"])
        r = oracle.ess_resample(o["logw"], G, N, cfg.ess_threshold, x.resample_uniforms)
        compare_resample(L, host(out["ancestors"]), host(out["ess"]), host(out["resampled"]),
                         host(lw), r, N)
        m = oracle.pagetable_remap(host(out["ancestors"]), host(out["resampled"]), G, N,
                                   table_before, P, num_pages=S * P)
        np.testing.assert_array_equal(host(out["table_out"]), m["table_out"])
        np.testing.assert_array_equal(host(out["refcount"]), m["refcount"])
        assert m["refcount"].sum() == S * P
        # free-running oracle
        of = oracle.smc_reweight(x.tgt, x.drf, x.draft_tokens, S, K, V, cfg.temperature,
                                 cfg.alpha, x.bonus_uniforms, lw_free, threads=nthr)
        rf = oracle.ess_resample(of["logw"], G, N, cfg.ess_threshold, x.resample_uniforms)
        mf = oracle.pagetable_remap(rf["ancestors"], rf["resampled"], G, N, table_free, P,
                                    num_pages=S * P)
        lw_free, table_free = rf["logw"], mf["table_out"]
        if first_div is None and not (
                np.array_equal(of["bonus_token"], host(out["bonus_token"]))
                and np.array_equal(rf["ancestors"], host(out["ancestors"]))
                and np.array_equal(rf["resampled"], host(out["resampled"]))):
            first_div = step
        table = out["table_out"]
    L.finish()
    return first_div, host(lw), lw_free


def test_smc_step_32_steps(smcsd):
    cfg = small_cfg()
    first_div, lw_gpu, lw_free = run_steps(smcsd, cfg, 32)
    assert first_div is None, f"free-running oracle diverged at step {first_div}"
    np.testing.assert_allclose(lw_gpu, lw_free, atol=FLOAT_ATOL, rtol=0)


@pytest.mark.parametrize("cfg,steps", [(synth.SMC_LLAMA3, 32), (synth.SMC_QWEN_POWER, 8)],
                         ids=["smc_llama3_32_steps", "smc_qwen_power_8_steps"])
def test_smc_step_full_size(smcsd, cfg, steps):
    """The full-size workloads run free: 32 consecutive fused steps of the 8 x 16 particle,
    K=4, V=128256 step and 8 of the 4 x 64, K=8, V=151936 power-target step, each compared
    with the oracle teacher-forced, and a free-running oracle that must take every decision the
    GPU took (tokens, resampling flags, ancestors) and end on the same log-weights."""
    first_div, lw_gpu, lw_free = run_steps(smcsd, cfg, steps)
    assert first_div is None, f"free-running oracle diverged at step {first_div}"
    np.testing.assert_allclose(lw_gpu, lw_free, atol=FLOAT_ATOL, rtol=0)


@pytest.mark.parametrize("GN", [(8, 16), (3, 48), (5, 2), (6, 5), (4, 12), (2, 24)],
                         ids=["groups_of_16", "groups_of_48", "groups_of_2", "groups_of_5", "groups_of_12",
                              "groups_of_24"])
def test_fused_step_equals_separate_calls(smcsd, GN):
    """The fused step equals reweight + resample + remap called one by one; groups of 48 take
    the fused step's path for groups larger than one warp, groups of 2..16 its thread-block
    clusters (portable sizes up to 8, the opt-in size above), groups of 24 its arrival counter."""
    G, N = GN
    cfg = synth.SMCConfig("smc_small", G, N, 4, 20000, 3.0, 1.0, 1.0, 1.0, 256)
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    x = synth.smc_step_inputs(cfg, 3, 0)
    lw0 = np.random.default_rng(3).normal(0, 2, S).astype(np.float32)
    table = dev(synth.initial_page_table(S, P))
    t, d, toks = dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens)
    ub, ur = dev(x.bonus_uniforms), dev(x.resample_uniforms)
    lw_a = dev(lw0.copy())
    a = smcsd.smc_step(t, d, toks, G, N, K, V, 1.0, 1.0, ub, lw_a, N / 2.0, ur, table_in=table,
                       pages_per_seq=P, num_pages=S * P)
    lw_b = dev(lw0.copy())
    tok_b = smcsd.smc_reweight(t, d, toks, S, K, V, 1.0, 1.0, ub, lw_b)
    anc_b, ess_b, res_b = smcsd.smc_ess_resample(lw_b, G, N, N / 2.0, ur)
    tout_b, rc_b = smcsd.kv_pagetable_remap(anc_b, res_b, G, N, table, P, num_pages=S * P)
    for ka, vb in (("bonus_token", tok_b), ("ancestors", anc_b), ("ess", ess_b),
                   ("resampled", res_b), ("table_out", tout_b), ("refcount", rc_b)):
        assert torch.equal(a[ka], vb), ka
    assert torch.equal(lw_a, lw_b)


def test_workspace_exp_table_cache_across_scales(smcsd):
    """One workspace, alternating scales alpha/T: the first call publishes its exp table in the
    workspace, calls with another scale build their own, calls with the first scale reuse it.
    Every call must match the oracle."""
    S, K, V = 16, 2, 20000
    ws = smcsd.Workspace(smcsd.OP_SMC_REWEIGHT, S, K, V)
    L = DecisionLedger()
    for i, (T, alpha) in enumerate([(1.0, 1.0), (0.7, 4.0), (1.0, 1.0), (0.7, 4.0), (1.0, 1.0)]):
        c, u, lw0 = reweight_case(smcsd, 50 + i, S, K, V, T, alpha)
        lw = dev(lw0.copy())
        tok = smcsd.smc_reweight(dev_logits(c.tgt), dev_logits(c.drf), dev(c.draft_tokens), S, K, V,
                                 T, alpha, dev(u), lw, ws=ws)
        assert smcsd.check_status(ws) == 0
        o = oracle.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, T, alpha, u, lw0)
        L.compare("bonus_token", host(tok), o["bonus_token"], o["bonus_margin"])
        np.testing.assert_allclose(host(lw), o["logw"], atol=FLOAT_ATOL, rtol=0)
    L.finish()
