"""Pins of the oracle's SMC-SD steps ("Faster LLM Inference via Sequential Monte Carlo",
sec. 2 steps 3-4 and sec. 3): importance reweighting by the target/draft probability
ratio, exactly K+1 tokens per particle, effective sample size, resampling below a
threshold, the power target, and the paged-KV page-table remap.

Pins: the importance-sampling identity q(x) * exp(dlogw(x)) = pi(x) checked for every x by
enumeration against scipy's softmax; identical models leave the weights unchanged; the
bonus token's exact grid distribution equals pi at row K; ESS closed forms (uniform,
one-hot, k equal weights) and bounds; systematic resampling's offspring counts, order,
special cases and unbiasedness; remap against numpy's bincount.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

from smc_reweight_resample_gb300 import synth

GRID = 1 << 24


def _u(m):
    return (np.asarray(m, np.float64) * 2.0 ** -24).astype(np.float32)


def _enum_case(V, K, seed, dtype="fp32"):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    zd = rng.normal(0, 1.5, (K, V)).astype(np.float32)
    if dtype == "bf16":
        zt, zd = synth.bf16_bits(zt), synth.bf16_bits(zd)
    xs = list(itertools.product(range(V), repeat=K))
    S = len(xs)
    tgt = np.tile(zt[None], (S, 1, 1)).reshape(S * (K + 1), V)
    drf = np.tile(zd[None], (S, 1, 1)).reshape(S * K, V)
    toks = np.array(xs, np.int32).reshape(S * K)
    return zt, zd, xs, tgt, drf, toks


@pytest.mark.parametrize("V,K,T,alpha,dtype", [(4, 2, 1.0, 1.0, "fp32"), (3, 3, 0.7, 4.0, "fp32"),
                                               (5, 2, 1.0, 2.0, "bf16")])
def test_importance_identity_by_enumeration(orc, V, K, T, alpha, dtype):
    zt, zd, xs, tgt, drf, toks = _enum_case(V, K, 17, dtype)
    S = len(xs)
    T, alpha = float(np.float32(T)), float(np.float32(alpha))  # the oracle reads float32 parameters
    out = orc.smc_reweight(tgt, drf, toks, S, K, V, T, alpha, np.zeros(S, np.float32),
                           np.zeros(S, np.float32))
    pi = softmax(alpha * synth.widen(zt).astype(np.float64) / T, axis=1)
    q = softmax(synth.widen(zd).astype(np.float64) / T, axis=1)
    wq = np.array([np.prod([q[k, x[k]] for k in range(K)]) for x in xs])
    wp = np.array([np.prod([pi[k, x[k]] for k in range(K)]) for x in xs])
    # E_q[w] = 1 and q(x) w(x) = pi(x) for every x
    assert (wq * np.exp(out["dlogw"])).sum() == pytest.approx(1.0, abs=1e-12)
    np.testing.assert_allclose(wq * np.exp(out["dlogw"]), wp, rtol=1e-11)
    # the stored float32 weight is the double increment rounded once
    np.testing.assert_array_equal(out["logw"], out["dlogw"].astype(np.float32))


def test_identical_models_leave_weights(orc):
    S, K, V = 8, 4, 700
    c = synth.sd_case(1, S, K, V, 3.0, 1.0)
    drf = c.tgt.reshape(S, K + 1, V)[:, :K].reshape(S * K, V).copy()
    lw0 = np.random.default_rng(2).normal(0, 1, S).astype(np.float32)
    out = orc.smc_reweight(c.tgt, drf, c.draft_tokens, S, K, V, 1.0, 1.0,
                           synth.uniforms(0, S), lw0)
    assert (out["dlogw"] == 0.0).all()
    np.testing.assert_array_equal(out["logw"], lw0)
    # equal weights: ESS = N, no resampling
    r = orc.ess_resample(np.zeros(S, np.float32), 1, S, S / 2, np.array([0.3], np.float32))
    assert r["ess"][0] == S and r["resampled"][0] == 0


def test_power_target_alpha_one_and_temperature_equivalence(orc):
    S, K, V = 4, 3, 2000
    c = synth.sd_case(4, S, K, V, 3.0, 1.0)
    u = synth.uniforms(5, S)
    lw = np.zeros(S, np.float32)
    a = orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, 1.0, u, lw)
    # alpha = 1 is the plain target: its per-row lse equals the SD oracle's
    sd = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, S, K, V, 1.0, synth.uniforms(5, S * (K + 1)))
    np.testing.assert_allclose(a["lse_tgt"], sd["lse_tgt"], rtol=0, atol=1e-13)
    # target alpha*z/T with draft at T: the target part equals temperature T/alpha
    T, alpha = float(np.float32(0.7)), 4.0
    b = orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, T, alpha, u, lw)
    zt = synth.widen(c.tgt).astype(np.float64)
    zd = synth.widen(c.drf).astype(np.float64)
    for s in range(S):
        inc = 0.0
        for k in range(K):
            x = c.draft_tokens[s * K + k]
            lpi = np.log(softmax(zt[s * (K + 1) + k] / (T / alpha))[x])
            lq = np.log(softmax(zd[s * K + k] / T)[x])
            inc += lpi - lq
        assert b["dlogw"][s] == pytest.approx(inc, abs=1e-9)


def test_bonus_token_grid_distribution_is_pi(orc):
    """The (K+1)-th token: exact probabilities over the 2^24 uniform grid equal pi at row K."""
    V, K = 6, 2
    rng = np.random.default_rng(8)
    S = 1
    zt = rng.normal(0, 2, (K + 1, V)).astype(np.float32)
    zd = rng.normal(0, 2, (K, V)).astype(np.float32)
    toks = np.array([1, 4], np.int32)
    for T, alpha in ((1.0, 1.0), (float(np.float32(0.7)), 4.0)):
        bounds = [0]
        for v in range(1, V):
            lo, hi = 0, GRID
            while lo < hi:
                mid = (lo + hi) // 2
                o = orc.smc_reweight(zt, zd, toks, S, K, V, T, alpha, _u([mid]), np.zeros(1, np.float32))
                if o["bonus_token"][0] >= v:
                    hi = mid
                else:
                    lo = mid + 1
            bounds.append(lo)
        bounds.append(GRID)
        probs = np.diff(bounds) / GRID
        want = softmax(alpha * zt[K].astype(np.float64) / T)
        np.testing.assert_allclose(probs, want, atol=2e-7)


# ------------------------------------------------------------------------------------
# effective sample size and systematic resampling
# ------------------------------------------------------------------------------------

def test_ess_closed_forms(orc):
    N = 16
    lw = np.full(N, 3.25, np.float32)
    assert orc.ess_resample(lw, 1, N, 0.0, np.zeros(1, np.float32))["ess"][0] == N
    lw = np.full(N, -np.inf, np.float32)
    lw[5] = -2.0
    assert orc.ess_resample(lw, 1, N, 0.0, np.zeros(1, np.float32))["ess"][0] == 1.0
    for k in (2, 3, 7):
        lw = np.full(N, -np.inf, np.float32)
        lw[np.random.default_rng(k).choice(N, k, replace=False)] = 0.5
        assert orc.ess_resample(lw, 1, N, 0.0, np.zeros(1, np.float32))["ess"][0] == pytest.approx(k, rel=1e-12)


def test_ess_bounds_and_shift_invariance(orc):
    G, N = 50, 64
    rng = np.random.default_rng(3)
    lw = rng.normal(0, 3, G * N).astype(np.float32)
    r = orc.ess_resample(lw, G, N, 0.0, np.zeros(G, np.float32))
    assert (r["ess"] >= 1.0).all() and (r["ess"] <= N).all()
    r2 = orc.ess_resample(lw + np.float32(8.0), G, N, 0.0, np.zeros(G, np.float32))
    np.testing.assert_allclose(r2["ess"], r["ess"], rtol=1e-5)


def test_threshold_is_strict(orc):
    lw = np.array([0.0, 0.0, -np.inf, -np.inf], np.float32)  # ESS = 2 exactly
    assert orc.ess_resample(lw, 1, 4, 2.0, np.zeros(1, np.float32))["resampled"][0] == 0
    assert orc.ess_resample(lw, 1, 4, np.nextafter(np.float32(2.0), np.float32(3.0)),
                            np.zeros(1, np.float32))["resampled"][0] == 1


def test_systematic_special_cases(orc):
    N = 16
    for U in (0.0, 0.37, 1.0 - 2 ** -24):
        r = orc.ess_resample(np.zeros(N, np.float32), 1, N, N + 1.0, np.array([U], np.float32))
        assert r["resampled"][0] == 1
        np.testing.assert_array_equal(r["ancestors"], np.arange(N))
        lw = np.full(N, -np.inf, np.float32)
        lw[9] = 1.0
        r = orc.ess_resample(lw, 1, N, N + 1.0, np.array([U], np.float32))
        assert (r["ancestors"] == 9).all()
        assert (r["logw"] == 0.0).all()


def test_systematic_offspring_counts_and_unbiasedness(orc):
    G, N = 6, 16
    rng = np.random.default_rng(12)
    lw = rng.normal(0, 1.5, G * N).astype(np.float32)
    w = np.exp(lw.reshape(G, N).astype(np.float64))
    w /= w.sum(1, keepdims=True)
    M = 2048
    mean_counts = np.zeros((G, N))
    for m in range(M):
        U = np.full(G, (m + 0.5) / M, np.float32)
        r = orc.ess_resample(lw, G, N, N + 1.0, U)
        a = r["ancestors"].reshape(G, N)
        assert (np.diff(a, axis=1) >= 0).all()
        cnt = np.stack([np.bincount(a[g], minlength=N) for g in range(G)])
        assert (cnt.sum(1) == N).all()
        lo = np.floor(N * w - 1e-9)
        hi = np.ceil(N * w + 1e-9)
        assert ((cnt >= lo) & (cnt <= hi)).all()
        mean_counts += cnt
    np.testing.assert_allclose(mean_counts / M, N * w, atol=1.01 / M)


def test_no_resample_keeps_weights_bitwise(orc):
    G, N = 3, 8
    lw = np.random.default_rng(1).normal(0, 0.1, G * N).astype(np.float32)
    r = orc.ess_resample(lw, G, N, 1.0, np.full(G, 0.5, np.float32))
    assert (r["resampled"] == 0).all()
    np.testing.assert_array_equal(r["logw"], lw)
    np.testing.assert_array_equal(r["ancestors"], np.tile(np.arange(N), G))


def test_ess_nonfinite(orc):
    lw = np.zeros(4, np.float32)
    lw[2] = np.nan
    assert orc.ess_resample(lw, 1, 4, 2.0, np.zeros(1, np.float32), raise_on_error=False)["status"] == orc.ENONFINITE
    lw = np.full(4, -np.inf, np.float32)
    assert orc.ess_resample(lw, 1, 4, 2.0, np.zeros(1, np.float32), raise_on_error=False)["status"] == orc.ENONFINITE


# ------------------------------------------------------------------------------------
# page-table remap
# ------------------------------------------------------------------------------------

def test_remap_rows_and_refcount(orc):
    G, N, P = 4, 8, 16
    rng = np.random.default_rng(6)
    table = rng.permutation(G * N * P).astype(np.int32)
    table[5] = -1
    anc = np.sort(rng.integers(0, N, (G, N)), axis=1).astype(np.int32).reshape(-1)
    res = np.array([1, 0, 1, 1], np.int32)
    r = orc.pagetable_remap(anc, res, G, N, table, P, num_pages=G * N * P)
    tin = table.reshape(G, N, P)
    tout = r["table_out"].reshape(G, N, P)
    for g in range(G):
        for j in range(N):
            src = anc[g * N + j] if res[g] else j
            np.testing.assert_array_equal(tout[g, j], tin[g, src])
    valid = r["table_out"][r["table_out"] >= 0]
    np.testing.assert_array_equal(r["refcount"], np.bincount(valid, minlength=G * N * P))
    assert r["refcount"].sum() == (r["table_out"] != -1).sum()


def test_remap_identity_without_resampling(orc):
    G, N, P = 2, 4, 8
    table = np.arange(G * N * P, dtype=np.int32)
    anc = np.zeros(G * N, np.int32)  # ignored: no group resampled
    r = orc.pagetable_remap(anc, np.zeros(G, np.int32), G, N, table, P, num_pages=G * N * P)
    np.testing.assert_array_equal(r["table_out"], table)
    assert (r["refcount"] == 1).all() and r["refcount"].sum() == G * N * P


def test_remap_range_errors(orc):
    G, N, P = 1, 2, 2
    table = np.array([0, 1, 2, 9], np.int32)
    r = orc.pagetable_remap(np.array([0, 1], np.int32), None, G, N, table, P, num_pages=4,
                            raise_on_error=False)
    assert r["status"] == orc.ERANGE
    r = orc.pagetable_remap(np.array([0, 2], np.int32), None, G, N, np.arange(4, dtype=np.int32), P,
                            num_pages=4, raise_on_error=False)
    assert r["status"] == orc.ERANGE
