"""The error bounds of "Faster LLM Inference via Sequential Monte Carlo", sec. 3 ("Theoretische
Fundierung": the squared L2 bias and the mean squared error of the importance-weighted estimate
fall as O(1/N) in the number of particles N), checked on the GPU's weights, and the robustness
claim of sec. 4 (SMC-SD's step time stays flat as the temperature rises, since every particle
emits K+1 tokens whatever is accepted).

A known target on V=8 with context-free rows (K=2): groups of N particles draw their tokens from
q, smc_reweight gives their log-weights, and each group estimates p_0 (the target's first-row
distribution, scipy's softmax) by the self-normalised weighted frequencies of its first tokens.
Over N = 4 .. 64 the log-log slope of the MSE must lie in [-1.15, -0.85] and the squared bias
must fall at least as fast. Seeds are fixed, so the test is deterministic."""
import numpy as np
import pytest
import torch

from smc_reweight_resample_gb300 import synth

pytestmark = pytest.mark.gpu

NS = (4, 8, 16, 32, 64)
TOTAL = 1 << 20  # particles per N


def estimates(smcsd, N, zt, zd, q):
    Vs, Ks = zt.shape[1], zd.shape[0]
    G = TOTAL // N
    S = G * N
    ux = synth.uniforms(12, S * Ks, stream=N).reshape(S, Ks).astype(np.float64)
    x = np.stack([np.minimum(np.searchsorted(np.cumsum(q[k]) / q[k].sum(), ux[:, k], side="right"),
                             Vs - 1) for k in range(Ks)], axis=1).astype(np.int32)
    tgt = torch.from_numpy(zt).cuda().repeat(S, 1).contiguous()
    drf = torch.from_numpy(zd).cuda().repeat(S, 1).contiguous()
    lw = torch.zeros(S, device="cuda")
    ws = smcsd.Workspace(smcsd.OP_SMC_REWEIGHT, S, Ks, Vs)
    smcsd.smc_reweight(tgt, drf, torch.from_numpy(x.reshape(-1)).cuda(), S, Ks, Vs, 1.0, 1.0,
                       torch.from_numpy(synth.uniforms(13, S, stream=N)).cuda(), lw, ws=ws)
    assert smcsd.check_status(ws) == 0
    w = np.exp(lw.cpu().numpy().astype(np.float64)).reshape(G, N)
    onehot = np.eye(Vs)[x[:, 0]].reshape(G, N, Vs)
    del tgt, drf, lw, ws
    torch.cuda.empty_cache()
    return (w[:, :, None] * onehot).sum(1) / w.sum(1)[:, None]  # [G, Vs]


def test_bias_and_mse_fall_as_one_over_n(smcsd):
    from scipy.special import softmax

    Vs, Ks = 8, 2
    rng = np.random.default_rng(11)
    zd = rng.normal(0, 1.0, (Ks + 1, Vs)).astype(np.float32)
    zt = (zd + rng.normal(0, 0.8, (Ks + 1, Vs))).astype(np.float32)
    q = softmax(zd.astype(np.float64), axis=1)
    p0 = softmax(zt[0].astype(np.float64))
    mse, bias2, floor = [], [], []
    for N in NS:
        est = estimates(smcsd, N, zt, zd[:Ks], q)
        mse.append(((est - p0) ** 2).sum(1).mean())
        bias2.append(((est.mean(0) - p0) ** 2).sum())
        floor.append(est.var(0).sum() / est.shape[0])  # sampling noise in the bias estimate
    lx = np.log(np.array(NS, np.float64))
    slope_mse = np.polyfit(lx, np.log(mse), 1)[0]
    slope_bias = np.polyfit(lx, np.log(bias2), 1)[0]
    assert -1.15 <= slope_mse <= -0.85, (slope_mse, mse)
    assert slope_bias <= slope_mse, (slope_bias, bias2)
    assert all(b > 10 * f for b, f in zip(bias2, floor)), (bias2, floor)  # bias measured, not noise


def test_step_time_flat_across_temperature(smcsd):
    """The fused step's device time at T = 0.7 and T = 2 is within 30 % of its time at T = 1
    (128 particles, K=4, V=32000 bf16; 40 graph-replayed steps per point)."""
    cfg0 = synth.SMCConfig("flat", 8, 16, 4, 32000, 3.0, 1.0, 1.0, 1.0, 256)
    S, K, V, G, N, P = cfg0.S, cfg0.K, cfg0.V, cfg0.G, cfg0.N, cfg0.pages_per_seq
    x = synth.smc_step_inputs(cfg0, 3, 0)
    from gpu_util import dev, dev_logits

    t, d, toks = dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens)
    ub, ur = dev(x.bonus_uniforms), dev(x.resample_uniforms)
    ws = smcsd.Workspace(smcsd.OP_SMC_STEP, S, K, V)
    tables = [dev(synth.initial_page_table(S, P)), torch.empty(S * P, dtype=torch.int32, device="cuda")]
    lw = torch.zeros(S, device="cuda")
    stream = torch.cuda.Stream()
    times = {}
    for T in (1.0, 0.7, 2.0):
        def step(i):
            smcsd.smc_step(t, d, toks, G, N, K, V, T, 1.0, ub, lw, N / 2.0, ur, table_in=tables[i % 2],
                           pages_per_seq=P, num_pages=S * P, ws=ws, table_out=tables[(i + 1) % 2],
                           stream=stream)
        with torch.cuda.stream(stream):
            for i in range(4):
                step(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(40):
                step(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        times[T] = e0.elapsed_time(e1) / 40
    assert smcsd.check_status(ws) == 0
    for T in (0.7, 2.0):
        assert abs(times[T] / times[1.0] - 1.0) < 0.30, times
