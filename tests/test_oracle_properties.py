"""Randomised pins of the oracle (hypothesis draws the shapes and values; each property is a
closed form or an identity of the method, checked against library routines where one applies).

* Importance identity ("Faster LLM Inference via Sequential Monte Carlo", sec. 2 step 3, and the
  power target of sec. 3): for every draft sequence x in V^K, q(x) * exp(dlogw(x)) equals the
  target's mass at x, per-position pi = softmax(alpha z / T) or whole-sequence p^alpha, for random
  V, K, T, alpha and masked tokens.
* Systematic resampling (same page, sec. 2 step 4): each particle's offspring count is floor or
  ceil of N w_i, the counts sum to N, ancestors never decrease, and the ESS lies in [1, N].
* The inverse-CDF draw: the token's interval contains u * R.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

SETTINGS = settings(max_examples=40, deadline=None)


def _logits(rng, rows, V, mask_frac):
    z = rng.normal(0, 1.5, (rows, V)).astype(np.float32)
    m = rng.random((rows, V)) < mask_frac
    m[:, 0] = False  # every row keeps some mass
    z[m] = -np.inf
    return z


@SETTINGS
@given(V=st.integers(2, 5), K=st.integers(1, 2), T=st.floats(0.4, 2.0), alpha=st.floats(0.3, 4.0),
       seq=st.booleans(), mask=st.sampled_from([0.0, 0.3]), seed=st.integers(0, 2**31 - 1))
def test_importance_identity(orc, V, K, T, alpha, seq, mask, seed):
    T, alpha = float(np.float32(T)), float(np.float32(alpha))
    rng = np.random.default_rng(seed)
    zt = _logits(rng, K + 1, V, mask)
    zt[K] = -np.inf
    zt[K, 0] = 0.5  # a one-hot last row: the (K+1)-th token is 0 and adds nothing
    zd = _logits(rng, K, V, mask)
    q = softmax(zd.astype(np.float64) / T, axis=1)
    xs = [x for x in itertools.product(range(V), repeat=K)
          if all(q[k, x[k]] > 0 for k in range(K))]  # drafts the draft can propose
    S = len(xs)
    tgt = np.tile(zt[None], (S, 1, 1)).reshape(S * (K + 1), V)
    drf = np.tile(zd[None], (S, 1, 1)).reshape(S * K, V)
    toks = np.array(xs, np.int32).reshape(S * K)
    out = orc.smc_reweight_tilted(tgt, drf, toks, S, K, V, T, alpha, np.zeros(S, np.float32),
                                  np.zeros(S, np.float32), target_mode=int(seq))
    if seq:
        gamma_rows = softmax(zt[:K].astype(np.float64) / T, axis=1) ** alpha
    else:
        gamma_rows = softmax(alpha * zt[:K].astype(np.float64) / T, axis=1)
    wq = np.array([np.prod([q[k, x[k]] for k in range(K)]) for x in xs])
    gamma = np.array([np.prod([gamma_rows[k, x[k]] for k in range(K)]) for x in xs])
    np.testing.assert_allclose(wq * np.exp(out["dlogw"]), gamma, rtol=1e-9, atol=1e-300)
    assert (out["bonus_token"] == 0).all()


@SETTINGS
@given(N=st.integers(1, 40), spread=st.floats(0.0, 6.0), U=st.floats(0.0, 0.999999),
       seed=st.integers(0, 2**31 - 1))
def test_systematic_resampling_properties(orc, N, spread, U, seed):
    lw = np.random.default_rng(seed).normal(0, spread, N).astype(np.float32)
    U = np.float32(U)
    r = orc.ess_resample(lw, 1, N, float(N + 1), np.array([U], np.float32))  # always resample
    assert r["resampled"][0] == 1
    ess = float(r["ess"][0])
    assert 1.0 - 1e-6 <= ess <= N + 1e-5
    a = r["ancestors"]
    assert (np.diff(a) >= 0).all() and a.min() >= 0 and a.max() < N
    w = np.exp(lw.astype(np.float64) - lw.max())
    w /= w.sum()
    counts = np.bincount(a, minlength=N)
    assert counts.sum() == N
    lo, hi = np.floor(N * w), np.ceil(N * w)
    ok = (counts >= lo - 1e-9) & (counts <= hi + 1e-9)
    # a count may leave [floor, ceil] only where N w_i sits within rounding of an integer
    near = np.abs(N * w - np.round(N * w)) < 1e-9
    assert (ok | near).all()
    assert (r["logw"] == 0).all()


@SETTINGS
@given(V=st.integers(1, 50), u=st.floats(0.0, 0.999999), seed=st.integers(0, 2**31 - 1))
def test_inverse_cdf_interval_contains_target(orc, V, u, seed):
    r = np.random.default_rng(seed).random(V) ** 3
    r[np.random.default_rng(seed + 1).random(V) < 0.2] = 0.0
    if r.sum() == 0:
        r[0] = 1.0
    u = float(np.float32(u))
    tok, margin = orc.sample_inverse_cdf(r, u)
    c = np.concatenate([[0.0], np.cumsum(r)])
    R = c[-1]
    assert r[tok] > 0
    assert c[tok] <= u * R + 1e-12 * R and u * R < c[tok + 1] + 1e-12 * R
    assert margin >= -1e-12
