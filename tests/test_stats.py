"""Statistical checks of the GPU path on a small vocabulary, with fresh uniforms for every one of
about a million sequences: what the method promises in distribution, tested on the kernels'
own decisions rather than against the oracle's.

* SD ("Faster LLM Inference via Sequential Monte Carlo", sec. 1; textbook rejection sampling):
  the emitted tokens follow the target. With context-free rows p_k, q_k, the first emitted
  token (the first draft if accepted, else the correction token) is distributed as p_0, and
  the first two emitted tokens as p_0 x p_1; chi-square tests on both. The acceptance rate of
  position 0 is sum_i min(p_0(i), q_0(i)).
* SMC-SD (same page, sec. 2 step 3): with draft tokens drawn from q, the importance weights
  exp(increment) average to 1 (the target mass), and the weighted frequencies of the first
  draft token estimate p_0; both within 5 standard errors.
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax
from scipy.stats import chi2

from smc_reweight_resample_gb300 import synth
from gpu_util import dev, host

pytestmark = pytest.mark.gpu

V, K, S = 8, 2, 1 << 20
P_MIN = 1e-6  # chi-square p-value below which the test fails (fixed seeds: deterministic)


def rows(seed):
    rng = np.random.default_rng(seed)
    zd = rng.normal(0, 1.0, (K + 1, V)).astype(np.float32)
    zt = (zd + rng.normal(0, 0.8, (K + 1, V))).astype(np.float32)
    return zt, zd[:K]


def draw(prob, u):
    """Inverse-CDF draws of tokens from `prob` with uniforms u (host, test input only)."""
    c = np.cumsum(prob)
    return np.minimum(np.searchsorted(c / c[-1], u, side="right"), V - 1).astype(np.int32)


def inputs(seed):
    zt, zd = rows(seed)
    q = softmax(zd.astype(np.float64), axis=1)
    p = softmax(zt.astype(np.float64), axis=1)
    ux = synth.uniforms(seed, S * K, stream=11).reshape(S, K).astype(np.float64)
    x = np.stack([draw(q[k], ux[:, k]) for k in range(K)], axis=1).reshape(-1)
    tgt = torch.from_numpy(zt).cuda().repeat(S, 1).contiguous()  # [S*(K+1), V]
    drf = torch.from_numpy(zd).cuda().repeat(S, 1).contiguous()  # [S*K, V]
    return p, q, x, tgt, drf


def chi_square(counts, expected):
    stat = float(((counts - expected) ** 2 / expected).sum())
    return chi2.sf(stat, counts.size - 1)


def test_sd_emits_the_target_distribution(smcsd):
    p, q, x, tgt, drf = inputs(1)
    u = dev(synth.uniforms(2, S * (K + 1), stream=12))
    acc, tok = smcsd.sd_verify(tgt, drf, dev(x), S, K, V, 1.0, u)
    acc, tok, x = host(acc), host(tok), x.reshape(S, K)
    first = np.where(acc >= 1, x[:, 0], tok)
    second = np.where(acc >= 2, x[:, 1], np.where(acc == 1, tok, -1))
    # first token ~ p_0
    assert chi_square(np.bincount(first, minlength=V), S * p[0]) > P_MIN
    # acceptance rate of position 0: a_0 = sum_i min(p_0(i), q_0(i))
    a0 = np.minimum(p[0], q[0]).sum()
    # a second token is emitted iff the first draft was accepted (acc >= 1); the first token is
    # then distributed as min(p_0, q_0) / a_0 and the second, independently, as p_1
    two = acc >= 1
    pair = np.bincount(first[two] * V + second[two], minlength=V * V).astype(np.float64)
    joint = np.outer(np.minimum(p[0], q[0]) / a0, p[1]).reshape(-1)
    assert chi_square(pair, two.sum() * joint) > P_MIN
    rate = two.mean()
    assert abs(rate - a0) < 5 * np.sqrt(a0 * (1 - a0) / S)


def test_smc_weights_are_unbiased(smcsd):
    p, q, x, tgt, drf = inputs(3)
    lw = torch.zeros(S, device="cuda")
    smcsd.smc_reweight(tgt, drf, dev(x), S, K, V, 1.0, 1.0, dev(synth.uniforms(4, S, stream=13)), lw)
    w = np.exp(host(lw).astype(np.float64))
    se = w.std() / np.sqrt(S)
    assert abs(w.mean() - 1.0) < 5 * se
    x0 = x.reshape(S, K)[:, 0]
    for i in range(V):
        f = (x0 == i) * w
        assert abs(f.mean() - p[0, i]) < 5 * f.std() / np.sqrt(S) + 1e-12
