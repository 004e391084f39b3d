"""Pins of the oracle's PACER stop rule ("PACER: Blockwise Pre-verification for Speculative
Decoding with Adaptive Length", Methodik 1-3): block mean of the estimated acceptance
against a threshold that grows by rho after each block that passes; the block that stops
is kept.

Pins: a hand-derived example (tests/golden/pacer_hand.json), closed forms with a zero
head (every score is sigmoid(c)), the length range, and monotonicity in t0. With position
embeddings (Methodik 1): a hand-derived example (tests/golden/pacer_pos_hand.json), zero
embeddings give the plain rule, and on inputs whose sums h + e are exact the rule equals
the plain rule on the summed states.
"""
import json
import math
import os

import numpy as np
import pytest

from smc_reweight_resample_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_example(orc):
    with open(os.path.join(GOLDEN, "pacer_hand.json")) as f:
        g = json.load(f)
    h = synth.bf16_bits(np.array(g["hidden"], np.float32))[None]
    w = synth.bf16_bits(np.array(g["w"], np.float32))
    for case in g["cases"]:
        out = orc.pacer_block_stop(h, w, g["c"], 1, g["b"], g["max_blocks"], g["d"], case["t0"],
                                   case["rho"])
        assert out["lengths"][0] == case["length"]
        np.testing.assert_allclose(out["block_scores"], case["block_scores"], atol=1e-12)
        assert out["margin"][0] == pytest.approx(case["margin"], abs=1e-12)


def _zero_head(S, b, nb, d):
    return np.zeros((S, nb * b, d), np.uint16), np.zeros(d, np.uint16)


def test_zero_head_extremes(orc):
    h, w = _zero_head(3, 4, 5, 16)
    assert (orc.pacer_block_stop(h, w, 10.0, 3, 4, 5, 16, 0.5, 1.1)["lengths"] == 20).all()
    assert (orc.pacer_block_stop(h, w, -10.0, 3, 4, 5, 16, 0.5, 1.1)["lengths"] == 4).all()
    # score exactly 0.5 against t0 = 0.5: not below, passes; then t = 0.55 stops block 1
    assert (orc.pacer_block_stop(h, w, 0.0, 3, 4, 5, 16, 0.5, 1.1)["lengths"] == 8).all()


@pytest.mark.parametrize("c", [0.3, 0.8, 1.1, 2.0])
def test_zero_head_threshold_growth_closed_form(orc, c):
    """All block means equal m = sigmoid(c); the first stop is the smallest i with
    m < t0 rho^i, i.e. i = floor(log(m/t0)/log(rho)) + 1 for m >= t0."""
    b, nb, d, t0, rho = 2, 12, 8, 0.5, 1.1
    h, w = _zero_head(1, b, nb, d)
    m = 1.0 / (1.0 + math.exp(-c))
    i = math.floor(math.log(m / np.float32(t0)) / math.log(np.float32(rho))) + 1
    want = min(i + 1, nb) * b
    assert orc.pacer_block_stop(h, w, c, 1, b, nb, d, t0, rho)["lengths"][0] == want


def test_fixed_threshold_when_rho_is_one(orc):
    cs = synth.pacer_case(2, S=16, d=64)
    out = orc.pacer_block_stop(cs.hidden, cs.w, 0.0, cs.S, cs.b, cs.max_blocks, cs.d, 0.5, 1.0)
    bs = out["block_scores"].reshape(cs.S, cs.max_blocks)
    for s in range(cs.S):
        below = np.nonzero(bs[s][bs[s] >= 0] < 0.5)[0]
        want = (below[0] + 1) * cs.b if below.size else cs.max_blocks * cs.b
        assert out["lengths"][s] == want


def test_lengths_range_and_monotone_in_t0(orc):
    cs = synth.pacer_case(0, S=64, d=256)
    prev = None
    for t0 in (0.2, 0.35, 0.5, 0.6, 0.75):
        L = orc.pacer_block_stop(cs.hidden, cs.w, 0.0, cs.S, cs.b, cs.max_blocks, cs.d, t0, 1.1)["lengths"]
        assert ((L % cs.b) == 0).all() and (L >= cs.b).all() and (L <= cs.b * cs.max_blocks).all()
        if prev is not None:
            assert (L <= prev).all()
        prev = L


def test_scores_match_library_sigmoid(orc):
    cs = synth.pacer_case(1, S=4, d=128)
    out = orc.pacer_block_stop(cs.hidden, cs.w, 0.25, cs.S, cs.b, cs.max_blocks, cs.d, -1.0, 1.1)
    h = synth.bf16_widen(cs.hidden).astype(np.float64)
    w = synth.bf16_widen(cs.w).astype(np.float64)
    from scipy.special import expit

    m = expit(h @ w + 0.25).reshape(cs.S, cs.max_blocks, cs.b).mean(-1)
    np.testing.assert_allclose(out["block_scores"].reshape(cs.S, -1), m, atol=1e-12)
    assert (out["lengths"] == cs.b * cs.max_blocks).all()


# -------------------------------------------------------------------------------------------
# position embeddings (Methodik 1: hidden states together with position embeddings)
# -------------------------------------------------------------------------------------------


def test_pos_emb_hand_worked_example(orc):
    with open(os.path.join(GOLDEN, "pacer_pos_hand.json")) as f:
        g = json.load(f)
    h = synth.bf16_bits(np.array(g["hidden"], np.float32))
    w = synth.bf16_bits(np.array(g["w"], np.float32))
    e = synth.bf16_bits(np.array(g["pos_emb"], np.float32))
    out = orc.pacer_block_stop(h, w, g["c"], 2, g["b"], g["max_blocks"], g["d"], g["t0"], g["rho"],
                               pos_emb=e)
    np.testing.assert_array_equal(out["lengths"], g["lengths"])
    np.testing.assert_allclose(out["block_scores"], np.ravel(g["block_scores"]), atol=1e-12)


def test_zero_pos_emb_is_the_plain_rule(orc):
    cs = synth.pacer_case(3, S=8, d=128)
    e = np.zeros((cs.max_blocks * cs.b, cs.d), np.uint16)
    a = orc.pacer_block_stop(cs.hidden, cs.w, 0.1, cs.S, cs.b, cs.max_blocks, cs.d, 0.5, 1.1)
    b = orc.pacer_block_stop(cs.hidden, cs.w, 0.1, cs.S, cs.b, cs.max_blocks, cs.d, 0.5, 1.1,
                             pos_emb=e)
    for k in ("lengths", "block_scores", "margin"):
        np.testing.assert_array_equal(a[k], b[k])


def test_pos_emb_equals_plain_rule_on_summed_states(orc):
    """h and e on a grid of eighths in [-1/2, 1/2], so that every h + e is exact in bf16: the rule
    with embeddings equals the plain rule on hidden states h + e, position by position."""
    S, b, nb, d = 6, 4, 5, 32
    rng = np.random.default_rng(7)
    hf = rng.integers(-4, 5, (S, nb * b, d)).astype(np.float32) / 8
    ef = rng.integers(-4, 5, (nb * b, d)).astype(np.float32) / 8
    w = synth.bf16_bits(rng.normal(0, 0.5, d).astype(np.float32))
    a = orc.pacer_block_stop(synth.bf16_bits(hf), w, 0.05, S, b, nb, d, 0.45, 1.1,
                             pos_emb=synth.bf16_bits(ef))
    summed = synth.bf16_bits(hf + ef[None])
    assert np.array_equal(synth.bf16_widen(summed), hf + ef[None])  # the sums are exact
    p = orc.pacer_block_stop(summed, w, 0.05, S, b, nb, d, 0.45, 1.1)
    for k in ("lengths", "block_scores"):
        np.testing.assert_array_equal(a[k], p[k])
    assert len(set(a["lengths"].tolist())) > 1  # the case exercises several stop points
