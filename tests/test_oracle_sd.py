"""Pins of the oracle's speculative-decoding verify ("Faster LLM Inference via Sequential
Monte Carlo", sec. 1: SD verifies drafts by rejection sampling and discards the rest of
the block at the first rejection; the textbook rule is accept with min(1, p/q), draw the
correction from normalise(max(0, p - q)), and a bonus token from p when all K pass).

The strongest pin is exhaustive: for V <= 5 and K <= 3 with position-wise independent
rows, every draft sequence x in V^K is enumerated with weight prod q_k(x_k), and every
decision is integrated *exactly* over the 2^24-point uniform grid by bisection on the
black-box oracle. The emitted tokens must then follow the target: for every prefix
y_0..y_j, P(emitted prefix = y, length > j) = prod_{i<j} min(p_i, q_i)(y_i) * p_j(y_j),
with p, q taken from scipy's softmax (a library routine).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

from smc_reweight_resample_gb300 import synth

GRID = 1 << 24
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _u(m):
    return (np.asarray(m, np.float64) * 2.0 ** -24).astype(np.float32)


def _bisect_first(pred, n):
    """First grid index m in [0, GRID] with pred(m) True, per sequence (pred monotone)."""
    lo = np.zeros(n, np.int64)
    hi = np.full(n, GRID, np.int64)
    while (lo < hi).any():
        mid = (lo + hi) // 2
        p = pred(mid)
        active = lo < hi
        hi = np.where(active & p, mid, hi)
        lo = np.where(active & ~p, mid + 1, lo)
    return lo


class _Enum:
    """All draft sequences of a position-wise independent SD problem, one per sequence."""

    def __init__(self, orc, V, K, T, dtype, seed):
        rng = np.random.default_rng(seed)
        zt = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
        zd = rng.normal(0, 1.5, (max(K, 1), V)).astype(np.float32)[:K]
        if dtype == "bf16":
            zt, zd = synth.bf16_bits(zt), synth.bf16_bits(zd)
        self.orc, self.V, self.K, self.T = orc, V, K, T
        self.xs = list(itertools.product(range(V), repeat=K))
        S = self.S = len(self.xs)
        self.tgt = np.tile(zt[None], (S, 1, 1)).reshape(S * (K + 1), V)
        self.drf = np.tile(zd[None], (S, 1, 1)).reshape(S * K, V)
        self.toks = np.array(self.xs, np.int32).reshape(S * K)
        ztf = synth.widen(zt).astype(np.float64)
        zdf = synth.widen(zd).astype(np.float64)
        self.p = softmax(ztf / T, axis=1)
        self.q = softmax(zdf / T, axis=1) if K else np.zeros((0, V))

    def run(self, u):
        out = self.orc.sd_verify(self.tgt, self.drf, self.toks, self.S, self.K, self.V, self.T,
                                 u.reshape(-1))
        return out["accept_len"], out["out_token"]

    def accept_probs(self):
        """A[s, k] = exact probability that position k accepts under the uniform grid."""
        A = np.zeros((self.S, self.K))
        for k in range(self.K):
            def pred(m, k=k):
                u = np.zeros((self.S, self.K + 1), np.float32)
                u[:, k] = _u(m)
                acc, _ = self.run(u)
                return acc == k
            A[:, k] = _bisect_first(pred, self.S) / GRID
        return A

    def token_probs(self, j):
        """P[s, y] = probability of final token y given acceptance length j."""
        base = np.zeros((self.S, self.K + 1), np.float32)
        if j < self.K:
            base[:, j] = _u(GRID - 1)
        bounds = [np.zeros(self.S, np.int64)]
        for v in range(1, self.V):
            def pred(m, v=v):
                u = base.copy()
                u[:, self.K] = _u(m)
                _, tok = self.run(u)
                return tok >= v
            bounds.append(_bisect_first(pred, self.S))
        bounds.append(np.full(self.S, GRID, np.int64))
        b = np.stack(bounds, 1)
        return np.diff(b, axis=1) / GRID


@pytest.mark.parametrize("V,K,T,dtype,seed", [
    (4, 1, 1.0, "fp32", 0), (4, 2, 1.0, "fp32", 1), (3, 3, 0.7, "fp32", 2),
    (5, 2, 1.3, "bf16", 3), (2, 3, 1.0, "bf16", 4),
])
def test_exhaustive_output_distribution_is_target(orc, V, K, T, dtype, seed):
    e = _Enum(orc, V, K, T, dtype, seed)
    A = e.accept_probs()
    tokp = [e.token_probs(j) for j in range(K + 1)]
    wq = np.array([np.prod([e.q[k, x[k]] for k in range(K)]) for x in e.xs])

    # textbook acceptance probability per position: sum_x min(p_k(x), q_k(x))
    for k in range(K):
        marg = sum(wq[s] * A[s, k] for s in range(e.S))
        assert marg == pytest.approx(np.minimum(e.p[k], e.q[k]).sum(), abs=5e-6)

    # distribution of emitted sequences
    emitted = {}
    for s, x in enumerate(e.xs):
        reach = wq[s]
        for j in range(K + 1):
            pj = reach * ((1.0 - A[s, j]) if j < K else 1.0)
            for y in range(V):
                key = tuple(x[:j]) + (y,)
                emitted[key] = emitted.get(key, 0.0) + pj * tokp[j][s, y]
            if j < K:
                reach = reach * A[s, j]
    assert sum(emitted.values()) == pytest.approx(1.0, abs=1e-9)
    for j in range(K + 1):
        for y in itertools.product(range(V), repeat=j + 1):
            got = sum(pv for key, pv in emitted.items() if len(key) > j and key[:j + 1] == y)
            want = np.prod([min(e.p[i, y[i]], e.q[i, y[i]]) for i in range(j)]) * e.p[j, y[j]]
            assert got == pytest.approx(want, abs=5e-6), (j, y)


def test_identical_models_accept_everything(orc):
    """p == q: every ratio is exactly 1, so all K drafts pass for every u < 1 and the
    final token is the bonus from p at row K."""
    S, K, V = 6, 3, 50
    c = synth.sd_case(3, S, K, V, 3.0, 1.0)
    drf = c.tgt.reshape(S, K + 1, V)[:, :K].reshape(S * K, V).copy()
    u = synth.uniforms(9, S * (K + 1))
    u[: S * (K + 1): K + 1] = _u(GRID - 1)  # the largest uniform still accepts
    out = orc.sd_verify(c.tgt, drf, c.draft_tokens, S, K, V, 1.0, u)
    assert (out["accept_len"] == K).all()
    assert np.allclose(out["lse_tgt"].reshape(S, K + 1)[:, :K], out["lse_drf"].reshape(S, K), atol=0, rtol=0)
    # bonus token equals the inverse-CDF draw from row K alone
    for s in range(S):
        zK = synth.widen(c.tgt.reshape(S, K + 1, V)[s, K]).astype(np.float64)
        p = softmax(zK)
        tok, _ = orc.sample_inverse_cdf(p, u[s * (K + 1) + K])
        assert out["out_token"][s] == tok


def test_inverse_cdf_grid_histogram_and_one_hot(orc):
    rng = np.random.default_rng(11)
    p = rng.random(17)
    p[[3, 9]] = 0.0
    M = 20000
    hist = np.zeros(17)
    for i in range(M):
        t, _ = orc.sample_inverse_cdf(p, (i + 0.5) / M)
        hist[t] += 1
    assert np.abs(hist / M - p / p.sum()).max() <= 1.0 / M + 1e-12
    assert hist[3] == 0 and hist[9] == 0
    oh = np.zeros(9)
    oh[6] = 2.5
    for u in (0.0, 0.3, 1.0 - 2 ** -24):
        assert orc.sample_inverse_cdf(oh, u)[0] == 6


def test_inverse_cdf_strict_comparison(orc):
    """token = min{i : C_i > u R}: a uniform exactly on a boundary goes to the right."""
    assert orc.sample_inverse_cdf(np.array([1.0, 1.0]), 0.5)[0] == 1
    assert orc.sample_inverse_cdf(np.array([1.0, 1.0]), 0.5 - 2 ** -24)[0] == 0
    assert orc.sample_inverse_cdf(np.array([1.0, 1.0]), 0.0)[0] == 0
    assert orc.sample_inverse_cdf(np.array([0.0, 1.0]), 0.0)[0] == 1


def test_hand_worked_examples(orc):
    """Values derived by hand in tests/golden/sd_hand.json."""
    with open(os.path.join(GOLDEN, "sd_hand.json")) as f:
        g = json.load(f)
    tgt = np.array(g["tgt_logits"], np.float32)
    drf = np.array(g["drf_logits"], np.float32)
    for case in g["cases"]:
        out = orc.sd_verify(tgt, drf, np.array(case["draft_tokens"], np.int32), 1, 1, 2, 1.0,
                            np.array(case["uniforms"], np.float32))
        assert out["accept_len"][0] == case["accept_len"], case["name"]
        assert out["out_token"][0] == case["out_token"], case["name"]
        assert out["lse_tgt"][0] == pytest.approx(g["lse_tgt_row0"], abs=1e-12)
        if case.get("accept_margin") is not None:
            assert out["accept_margin"][0] == pytest.approx(case["accept_margin"], abs=1e-7)


def test_ragged_equals_fixed_per_sequence(orc):
    """A ragged call is the fixed-K verify of each sequence on its own rows."""
    lengths = np.array([3, 1, 4, 2, 0], np.int32)
    V = 300
    c = synth.ragged_sd_case(5, lengths, V, K_max=4)
    out = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, c.S, c.K, V, 1.0, c.uniforms,
                        c.tgt_offsets, c.drf_offsets)
    for s, L in enumerate(lengths):
        t0, t1 = c.tgt_offsets[s], c.tgt_offsets[s + 1]
        d0, d1 = c.drf_offsets[s], c.drf_offsets[s + 1]
        u = np.concatenate([c.uniforms[s * 5: s * 5 + L], c.uniforms[s * 5 + 4: s * 5 + 5]])
        drf = c.drf[d0:d1] if L else np.zeros((0, V), np.uint16)
        one = orc.sd_verify(c.tgt[t0:t1], drf if L else np.zeros((1, V), np.uint16),
                            c.draft_tokens[d0:d1] if L else np.zeros(1, np.int32), 1, int(L), V,
                            1.0, u)
        assert one["accept_len"][0] == out["accept_len"][s]
        assert one["out_token"][0] == out["out_token"][s]


def test_bad_inputs(orc):
    c = synth.sd_tiny(0)
    bad = c.draft_tokens.copy()
    bad[1] = c.V
    r = orc.sd_verify(c.tgt, c.drf, bad, c.S, c.K, c.V, 1.0, c.uniforms, raise_on_error=False)
    assert r["status"] == orc.ERANGE
    r = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, c.S, c.K, c.V, 0.0, c.uniforms,
                      raise_on_error=False)
    assert r["status"] == orc.EINVAL
    t = c.tgt.copy()
    t[2, 5] = np.nan
    r = orc.sd_verify(t, c.drf, c.draft_tokens, c.S, c.K, c.V, 1.0, c.uniforms,
                      raise_on_error=False)
    assert r["status"] == orc.ENONFINITE
    to = np.array([0, 3, 4, 7, 10], np.int32)  # second sequence: 1 target row but 2 draft rows
    do = np.array([0, 2, 4, 6, 8], np.int32)
    r = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, c.S, c.K, c.V, 1.0, c.uniforms, to, do,
                      raise_on_error=False)
    assert r["status"] == orc.ERANGE
