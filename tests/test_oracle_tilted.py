"""Pins of the oracle's tilted targets ("Faster LLM Inference via Sequential Monte Carlo",
sec. 3 "flexibility": power sampling and reward-weighted decoding as modified targets of the
same importance weights; sec. 5: reward optimisation and hard constraints).

Whole-sequence power target gamma(x) = prod_t p_t(x_t)^alpha, p = softmax(z/T), with draft
tokens proposed from q and the (K+1)-th token from p. Pins:
  * importance identity by enumeration: q(x) * exp(dlogw(x)) = prod_k p_k(x_k)^alpha for
    every x in V^K (bonus row one-hot, so the bonus factor is exactly 1), against scipy's
    softmax;
  * the bonus factor by enumeration over tokens: for every token b, the uniform in the middle
    of b's CDF interval draws b, and p(b) * exp(dlogw) = p(b)^alpha;
  * alpha = 1 gives the per-position target's results bit for bit;
  * normalisers at the plain scale 1/T, equal to the SD oracle's;
  * the additive log-reward: lambda * r added once, a constant reward leaves the group's
    normalised weights (ESS, ancestors) unchanged, non-finite rewards are errors.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

from smc_reweight_resample_gb300 import synth


def _enum_case(V, K, seed):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    zt[K, :] = -np.inf
    zt[K, 1] = 0.25  # one-hot bonus row: p_K(b) = 1, the bonus factor is 1
    zd = rng.normal(0, 1.5, (K, V)).astype(np.float32)
    xs = list(itertools.product(range(V), repeat=K))
    S = len(xs)
    tgt = np.tile(zt[None], (S, 1, 1)).reshape(S * (K + 1), V)
    drf = np.tile(zd[None], (S, 1, 1)).reshape(S * K, V)
    toks = np.array(xs, np.int32).reshape(S * K)
    return zt, zd, xs, tgt, drf, toks


@pytest.mark.parametrize("V,K,T,alpha", [(4, 2, 1.0, 2.0), (3, 3, 0.7, 4.0), (5, 2, 1.3, 0.5)])
def test_sequence_power_identity_by_enumeration(orc, V, K, T, alpha):
    zt, zd, xs, tgt, drf, toks = _enum_case(V, K, 23)
    S = len(xs)
    T, alpha = float(np.float32(T)), float(np.float32(alpha))
    out = orc.smc_reweight_tilted(tgt, drf, toks, S, K, V, T, alpha, synth.uniforms(3, S),
                                  np.zeros(S, np.float32), target_mode=orc.TARGET_SEQUENCE)
    assert (out["bonus_token"] == 1).all()
    p = softmax(zt[:K].astype(np.float64) / T, axis=1)
    q = softmax(zd.astype(np.float64) / T, axis=1)
    wq = np.array([np.prod([q[k, x[k]] for k in range(K)]) for x in xs])
    gamma = np.array([np.prod([p[k, x[k]] ** alpha for k in range(K)]) for x in xs])
    np.testing.assert_allclose(wq * np.exp(out["dlogw"]), gamma, rtol=1e-11)
    # E_q[w] is the target's total mass prod_k sum_i p_k(i)^alpha
    mass = np.prod((p ** alpha).sum(axis=1))
    assert (wq * np.exp(out["dlogw"])).sum() == pytest.approx(mass, rel=1e-12)


@pytest.mark.parametrize("V,T,alpha", [(6, 1.0, 3.0), (9, 0.7, 0.25)])
def test_sequence_power_bonus_factor_by_enumeration(orc, V, T, alpha):
    """K = 0: the step is the (K+1)-th token alone, drawn from p; its weight factor must make
    p(b) * w(b) the power target p(b)^alpha for every token b."""
    rng = np.random.default_rng(5)
    z = rng.normal(0, 1.5, (1, V)).astype(np.float32)
    T, alpha = float(np.float32(T)), float(np.float32(alpha))
    p = softmax(z[0].astype(np.float64) / T)
    c = np.concatenate([[0.0], np.cumsum(p)])
    u = ((c[:-1] + c[1:]) / 2).astype(np.float32)  # middle of each token's interval
    S = V
    tgt = np.tile(z, (S, 1))
    drf = np.zeros((1, V), np.float32)
    out = orc.smc_reweight_tilted(tgt, drf, np.zeros(1, np.int32), S, 0, V, T, alpha, u,
                                  np.zeros(S, np.float32), target_mode=orc.TARGET_SEQUENCE)
    np.testing.assert_array_equal(out["bonus_token"], np.arange(V))
    np.testing.assert_allclose(p * np.exp(out["dlogw"]), p ** alpha, rtol=1e-11)
    assert (p * np.exp(out["dlogw"])).sum() == pytest.approx((p ** alpha).sum(), rel=1e-12)


def test_alpha_one_equals_per_position_target(orc):
    S, K, V = 6, 3, 3000
    c = synth.sd_case(8, S, K, V, 3.0, 1.0)
    u = synth.uniforms(9, S)
    lw0 = np.random.default_rng(1).normal(0, 1, S).astype(np.float32)
    a = orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, 0.9, 1.0, u, lw0)
    b = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 0.9, 1.0, u, lw0,
                                target_mode=orc.TARGET_SEQUENCE)
    for key in ("logw", "bonus_token", "dlogw", "lse_tgt", "lse_drf", "bonus_margin"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_sequence_target_normalisers_are_plain(orc):
    """The whole-sequence target scores rows at 1/T whatever alpha is: its normalisers are the
    SD verify's, and its (K+1)-th token is the plain bonus draw from p."""
    S, K, V = 5, 2, 2500
    c = synth.sd_case(12, S, K, V, 3.0, 1.0)
    u = synth.uniforms(13, S)
    out = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 0.8, 3.0, u,
                                  np.zeros(S, np.float32), target_mode=orc.TARGET_SEQUENCE)
    plain = orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, 0.8, 1.0, u,
                             np.zeros(S, np.float32))
    np.testing.assert_array_equal(out["lse_tgt"], plain["lse_tgt"])
    np.testing.assert_array_equal(out["bonus_token"], plain["bonus_token"])


def test_reward_is_added_once(orc):
    S, K, V = 8, 2, 1500
    c = synth.sd_case(14, S, K, V, 3.0, 1.0)
    u = synth.uniforms(15, S)
    r = synth.log_rewards(16, S)
    for mode in (orc.TARGET_TOKEN, orc.TARGET_SEQUENCE):
        base = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 2.0, u,
                                       np.zeros(S, np.float32), target_mode=mode)
        zero = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 2.0, u,
                                       np.zeros(S, np.float32), target_mode=mode, log_reward=r,
                                       reward_scale=0.0)
        np.testing.assert_array_equal(zero["dlogw"], base["dlogw"])
        lam = np.float32(0.75)
        tilt = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 2.0, u,
                                       np.zeros(S, np.float32), target_mode=mode, log_reward=r,
                                       reward_scale=float(lam))
        np.testing.assert_allclose(tilt["dlogw"] - base["dlogw"], np.float64(lam) * r, atol=1e-12)
        np.testing.assert_array_equal(tilt["bonus_token"], base["bonus_token"])


def test_constant_reward_leaves_resampling_unchanged(orc):
    """A reward that is the same for every particle of a group scales all its weights alike: the
    normalised weights, ESS and ancestors do not change."""
    G, N, K, V = 2, 16, 2, 800
    S = G * N
    c = synth.sd_case(17, S, K, V, 3.0, 2.0)
    u = synth.uniforms(18, S)
    ur = synth.uniforms(19, G)
    base = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 1.0, u,
                                   np.zeros(S, np.float32))
    r = np.repeat(np.array([2.0, -3.0], np.float32), N)
    tilt = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 1.0, u,
                                   np.zeros(S, np.float32), log_reward=r, reward_scale=1.0)
    a = orc.ess_resample(base["logw"], G, N, N / 2, ur)
    b = orc.ess_resample(tilt["logw"], G, N, N / 2, ur)
    np.testing.assert_allclose(a["ess"], b["ess"], rtol=1e-5)
    np.testing.assert_array_equal(a["resampled"], b["resampled"])
    np.testing.assert_array_equal(a["ancestors"], b["ancestors"])


def test_bad_reward_and_mode(orc):
    S, K, V = 2, 1, 100
    c = synth.sd_case(20, S, K, V, 3.0, 1.0)
    u = synth.uniforms(21, S)
    lw = np.zeros(S, np.float32)
    for bad in (np.nan, np.inf, -np.inf):
        r = np.array([0.0, bad], np.float32)
        out = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 1.0, u, lw,
                                      log_reward=r, reward_scale=1.0, raise_on_error=False)
        assert out["status"] == orc.ENONFINITE
    out = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 1.0, u, lw,
                                  target_mode=2, raise_on_error=False)
    assert out["status"] == orc.EINVAL
    out = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 1.0, u, lw,
                                  log_reward=np.zeros(S, np.float32), reward_scale=float("nan"),
                                  raise_on_error=False)
    assert out["status"] == orc.EINVAL
