"""Pins of the oracle's decision margins, the numbers the GPU parity tests use to excuse a
mismatched decision ("Faster LLM Inference via Sequential Monte Carlo", sec. 1: the verify's
accept tests and final token; sec. 2 steps 3-4: the (K+1)-th token, the ESS threshold and
resampling; "PACER: Blockwise Pre-verification ...", Methodik 2-3: the block mean against t).

A margin claims how far the decision's input may move before the decision changes. Each test
checks that claim on the black-box oracle: it moves the float32 input the decision reads (the
uniform, the threshold, U) one representable value at a time by bisection, finds the nearest
inputs on either side at which the decision changes, and requires the reported margin to lie
between the distances those brackets allow. A margin that is too small (which would excuse a
real mismatch) or too large fails. Hand-derived values on inputs whose probabilities are exact
in binary (tests/golden/margins_hand.json) pin the absolute numbers as well.
"""
import json
import math
import os

import numpy as np
import pytest

from smc_reweight_resample_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SLACK = 1e-12  # the oracle's own double rounding in forming a margin


# ------------------------------------------------------------------------------------------
# float32 bisection
# ------------------------------------------------------------------------------------------

def _key(x: float) -> int:
    """Integer key of a float32 that orders like the value (negative floats included)."""
    i = int(np.array([x], np.float32).view(np.int32)[0])
    return i if i >= 0 else -(i & 0x7FFFFFFF)


def _val(k: int) -> float:
    i = k if k >= 0 else (-k) | -0x80000000
    return float(np.array([i], np.int32).view(np.float32)[0])


def flip_above(decide, x, limit):
    """Smallest float32 f in (x, limit] with decide(f) != decide(x), and its predecessor (the
    largest float with the decision unchanged); None if the decision never changes up to limit.
    `decide` must be monotone in its argument."""
    d0 = decide(x)
    lo, hi = _key(x), _key(limit)
    if decide(_val(hi)) == d0:
        return None
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if decide(_val(mid)) == d0:
            lo = mid
        else:
            hi = mid
    return _val(hi), _val(lo)


def flip_below(decide, x, limit):
    """Largest float32 f in [limit, x) with decide(f) != decide(x), and its successor."""
    d0 = decide(x)
    lo, hi = _key(limit), _key(x)
    if decide(_val(lo)) == d0:
        return None
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if decide(_val(mid)) == d0:
            hi = mid
        else:
            lo = mid
    return _val(lo), _val(hi)


def bracket(x, above, below, default_above=math.inf, default_below=math.inf):
    """Interval that the distance from x to the nearer decision boundary must lie in, given the
    bisection results (a boundary lies between a changed and an unchanged neighbour)."""
    if above is None:
        up_lo = up_hi = default_above
    else:
        f, f_prev = above
        up_lo, up_hi = f_prev - x, f - x
    if below is None:
        dn_lo = dn_hi = default_below
    else:
        f, f_next = below
        dn_lo, dn_hi = x - f_next, x - f
    return min(up_lo, dn_lo), min(up_hi, dn_hi)


def assert_in(margin, lo_hi, scale=1.0):
    lo, hi = lo_hi
    assert lo * scale - SLACK <= margin <= hi * scale + SLACK, (margin, lo * scale, hi * scale)


# ------------------------------------------------------------------------------------------
# SD verify: accept tests and final token
# ------------------------------------------------------------------------------------------

def _sd_cases():
    # (seed, S, K, V, sigma_d, sigma_t, T, dtype)
    return [(3, 3, 3, 64, 2.0, 1.0, 1.0, "fp32"), (4, 3, 2, 200, 3.0, 1.0, 0.7, "bf16"),
            (5, 2, 4, 50, 1.0, 0.5, 1.3, "fp32")]


@pytest.mark.parametrize("case", _sd_cases())
def test_sd_token_margin_by_bisection(orc, case):
    seed, S, K, V, sd, st, T, dt = case
    c = synth.sd_case(seed, S, K, V, sd, st, T, dt)
    base = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, S, K, V, T, c.uniforms)
    for s in range(S):
        j = s * (K + 1) + K  # the final draw's uniform (accept tests do not read it)

        def token(u, s=s, j=j):
            uu = c.uniforms.copy()
            uu[j] = u
            o = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, S, K, V, T, uu)
            assert o["accept_len"][s] == base["accept_len"][s]
            return int(o["out_token"][s])

        u = float(c.uniforms[j])
        b = bracket(u, flip_above(token, u, 1.0 - 2.0 ** -24), flip_below(token, u, 0.0),
                    default_above=1.0 - u, default_below=u)
        assert_in(base["token_margin"][s], b)


@pytest.mark.parametrize("case", _sd_cases())
def test_sd_accept_margin_by_bisection(orc, case):
    seed, S, K, V, sd, st, T, dt = case
    c = synth.sd_case(seed, S, K, V, sd, st, T, dt)
    base = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, S, K, V, T, c.uniforms)
    tested = 0
    for s in range(S):
        for k in range(int(min(base["accept_len"][s] + 1, K))):
            j = s * (K + 1) + k

            def rejected_at_k(u, s=s, j=j, k=k):  # monotone: 0 below the ratio, 1 from it on
                uu = c.uniforms.copy()
                uu[j] = u
                return int(orc.sd_verify(c.tgt, c.drf, c.draft_tokens, S, K, V, T, uu)
                           ["accept_len"][s] == k)

            # the one boundary is the ratio min(1, p/q) itself, which may lie at 0 (a ratio that
            # underflows) or at 1: search beyond [0, 1)
            u = float(c.uniforms[j])
            b = bracket(u, flip_above(rejected_at_k, u, 2.0), flip_below(rejected_at_k, u, -1.0))
            assert_in(base["accept_margin"][s * K + k], b)
            tested += 1
    assert tested > 0


# ------------------------------------------------------------------------------------------
# SMC: bonus token, ESS threshold, systematic resampling
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("T,alpha", [(1.0, 1.0), (0.7, 4.0)])
def test_smc_bonus_margin_by_bisection(orc, T, alpha):
    S, K, V = 4, 2, 300
    c = synth.sd_case(9, S, K, V, 3.0, 1.0, T)
    u0 = synth.uniforms(9, S, stream=7)
    lw = np.zeros(S, np.float32)
    base = orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, T, alpha, u0, lw)
    for s in range(S):
        def token(u, s=s):
            uu = u0.copy()
            uu[s] = u
            return int(orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, S, K, V, T, alpha, uu, lw)
                       ["bonus_token"][s])

        u = float(u0[s])
        b = bracket(u, flip_above(token, u, 1.0 - 2.0 ** -24), flip_below(token, u, 0.0),
                    default_above=1.0 - u, default_below=u)
        assert_in(base["bonus_margin"][s], b)


def _weight_cases():
    rng = np.random.default_rng(17)
    out = []
    for N, sigma in ((8, 1.0), (16, 2.5), (33, 0.7)):
        lw = rng.normal(0.0, sigma, N).astype(np.float32)
        out.append((N, lw))
    lw = rng.normal(0.0, 1.5, 12).astype(np.float32)
    lw[[2, 3, 7]] = -np.inf  # zero weights: plateaus in the CDF
    out.append((12, lw))
    return out


@pytest.mark.parametrize("case", range(4))
def test_ess_margin_by_bisection(orc, case):
    N, lw = _weight_cases()[case]
    U = np.array([0.37], np.float32)
    ess = float(orc.ess_resample(lw, 1, N, 0.0, U)["ess"][0])
    for thr in (ess * 0.9, ess * 1.1, float(np.float32(ess)), N / 2.0):
        thr = float(np.float32(thr))
        base = orc.ess_resample(lw, 1, N, thr, U)

        def resampled(t):  # monotone: 0 up to the ESS, 1 above it
            return int(orc.ess_resample(lw, 1, N, t, U)["resampled"][0])

        b = bracket(thr, flip_above(resampled, thr, 2.0 * N), flip_below(resampled, thr, 0.0))
        assert_in(base["ess_margin"][0], b, scale=1.0 / N)


@pytest.mark.parametrize("case", range(4))
def test_ancestor_margin_by_bisection(orc, case):
    N, lw = _weight_cases()[case]
    for U in (0.0, 0.37, 0.91):
        Ua = np.array([U], np.float32)
        base = orc.ess_resample(lw, 1, N, N + 1.0, Ua)  # threshold above N: always resamples
        assert base["resampled"][0] == 1
        for j in range(N):
            def anc(x, j=j):  # monotone in U
                return int(orc.ess_resample(lw, 1, N, N + 1.0, np.array([x], np.float32))
                           ["ancestors"][j])

            u = float(Ua[0])
            v = (j + u) / N
            a = int(base["ancestors"][j])
            # with no change above, the nearest CDF point is C_{N-1} = 1 (child stays at N-1)
            b = bracket(u, flip_above(anc, u, float(N + 1)), flip_below(anc, u, float(-N - 1)),
                        default_above=(1.0 - v) * N if a == N - 1 else math.inf)
            assert_in(base["anc_margin"][j], b, scale=1.0 / N)


# ------------------------------------------------------------------------------------------
# PACER: block mean against the threshold (rho = 1, so every comparison is against t0)
# ------------------------------------------------------------------------------------------

def test_pacer_margin_by_bisection(orc):
    S, b, nb, d = 6, 4, 5, 64
    cs = synth.pacer_case(5, S=S, b=b, max_blocks=nb, d=d)
    for t0 in (0.45, 0.5, 0.55):
        t0 = float(np.float32(t0))
        base = orc.pacer_block_stop(cs.hidden, cs.w, 0.0, S, b, nb, d, t0, 1.0)
        for s in range(S):
            def shorter(t, s=s):  # monotone: the length falls as t0 rises
                return -int(orc.pacer_block_stop(cs.hidden, cs.w, 0.0, S, b, nb, d, t, 1.0)
                            ["lengths"][s])

            br = bracket(t0, flip_above(shorter, t0, 2.0), flip_below(shorter, t0, -1.0))
            assert_in(base["margin"][s], br)


# ------------------------------------------------------------------------------------------
# hand-derived values
# ------------------------------------------------------------------------------------------

def _arr(rows):
    return np.array([[-np.inf if v == "-inf" else v for v in r] for r in rows], np.float32)


@pytest.fixture(scope="module")
def hand():
    with open(os.path.join(GOLDEN, "margins_hand.json")) as f:
        return json.load(f)


def test_hand_sd_residual(orc, hand):
    g = hand["sd_residual"]
    o = orc.sd_verify(_arr(g["tgt_logits"]), _arr(g["drf_logits"]), np.array(g["draft_tokens"]),
                      1, 1, 4, 1.0, np.array(g["uniforms"], np.float32))
    assert o["accept_len"][0] == g["accept_len"] and o["out_token"][0] == g["out_token"]
    assert o["accept_margin"][0] == pytest.approx(g["accept_margin"], abs=1e-12)
    assert o["token_margin"][0] == pytest.approx(g["token_margin"], abs=1e-12)


def test_hand_sd_bonus(orc, hand):
    g = hand["sd_bonus"]
    t = _arr(g["tgt_logits"])
    o = orc.sd_verify(t, np.zeros((1, 8), np.float32), np.zeros(0, np.int32), 1, 0, 8, 1.0,
                      np.array(g["uniforms"], np.float32))
    assert o["out_token"][0] == g["out_token"]
    assert o["token_margin"][0] == pytest.approx(g["token_margin"], abs=1e-12)


def test_hand_smc_bonus(orc, hand):
    g = hand["smc_bonus"]
    t = _arr(g["tgt_logits"])
    o = orc.smc_reweight(t, np.zeros((1, 4), np.float32), np.zeros(0, np.int32), 1, 0, 4, 1.0, 1.0,
                         np.array(g["uniforms"], np.float32), np.zeros(1, np.float32))
    assert o["bonus_token"][0] == g["bonus_token"] and o["logw"][0] == 0.0
    assert o["bonus_margin"][0] == pytest.approx(g["bonus_margin"], abs=1e-12)


def test_hand_ess_resample(orc, hand):
    g = hand["ess_resample"]
    lw = np.array([-np.inf if v == "-inf" else v for v in g["logw"]], np.float32)
    o = orc.ess_resample(lw, 1, lw.size, g["threshold"], np.array([g["U"]], np.float32))
    assert o["ess"][0] == g["ess"] and o["resampled"][0] == 1
    assert o["ess_margin"][0] == pytest.approx(g["ess_margin"], abs=1e-12)
    np.testing.assert_array_equal(o["ancestors"], g["ancestors"])
    np.testing.assert_allclose(o["anc_margin"], g["anc_margin"], atol=1e-12, rtol=0)


def test_a_planted_mistake_is_caught(orc):
    """The bracket test fails for a margin measured to the wrong end of the interval: the
    distance to the far end of the drawn token's interval lies outside the bracket."""
    c = synth.sd_case(3, 3, 3, 64, 2.0, 1.0, 1.0, "fp32")
    s, K = 0, 3
    j = s * (K + 1) + K
    base = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, 3, K, 64, 1.0, c.uniforms)

    def token(u):
        uu = c.uniforms.copy()
        uu[j] = u
        return int(orc.sd_verify(c.tgt, c.drf, c.draft_tokens, 3, K, 64, 1.0, uu)["out_token"][s])

    u = float(c.uniforms[j])
    up = flip_above(token, u, 1.0 - 2.0 ** -24)
    dn = flip_below(token, u, 0.0)
    lo, hi = bracket(u, up, dn, default_above=1.0 - u, default_below=u)
    width_lo = (up[1] if up else 1.0) - (dn[1] if dn else 0.0)
    wrong = width_lo - base["token_margin"][s]  # distance to the far end
    assert not (lo - SLACK <= wrong <= hi + SLACK)
