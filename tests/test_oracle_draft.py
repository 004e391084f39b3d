"""Pins of the oracle's draft-token sampler ("Faster LLM Inference via Sequential Monte Carlo",
sec. 2 step 1: the draft model proposes K tokens per particle, drawn from its tempered
distribution q = softmax(z/T)).

Pins: on a grid of uniforms the drawn tokens' histogram is q (scipy softmax) within 1/M; each
token's log q equals scipy's log_softmax at it and its normaliser numpy's logaddexp.reduce; a
row with one unmasked token always draws it; drafts drawn this way are accepted in full by an
SD verify whose target equals the draft; masked tokens are never drawn; bad inputs."""
import numpy as np
import pytest
from scipy.special import log_softmax, softmax

from smc_reweight_resample_gb300 import synth


def test_grid_histogram_is_q(orc):
    V, M, T = 37, 1 << 14, 0.8
    z = np.random.default_rng(1).normal(0, 2, V).astype(np.float32)
    u = ((np.arange(M) + 0.5) / M).astype(np.float32)
    out = orc.draft_sample(np.tile(z, (M, 1)), M, V, T, u)
    q = softmax(z.astype(np.float64) / np.float32(T))
    h = np.bincount(out["tokens"], minlength=V) / M
    assert np.abs(h - q).max() <= 1.0 / M + 1e-12
    np.testing.assert_allclose(out["logq"], log_softmax(z.astype(np.float64) / np.float32(T))[out["tokens"]],
                               atol=1e-12)
    np.testing.assert_allclose(out["lse"], np.logaddexp.reduce(z.astype(np.float64) / np.float32(T)),
                               atol=1e-12)


def test_one_unmasked_token_and_masks(orc):
    V, R = 50, 8
    z = np.full((R, V), -np.inf, np.float32)
    z[np.arange(R), np.arange(R) * 3] = np.arange(R, dtype=np.float32)
    out = orc.draft_sample(z, R, V, 1.0, synth.uniforms(0, R))
    np.testing.assert_array_equal(out["tokens"], np.arange(R) * 3)
    np.testing.assert_array_equal(out["logq"], 0.0)
    # half the vocabulary masked: never drawn
    z2 = np.random.default_rng(2).normal(0, 1, (64, V)).astype(np.float32)
    z2[:, ::2] = -np.inf
    out2 = orc.draft_sample(z2, 64, V, 1.0, synth.uniforms(1, 64))
    assert (out2["tokens"] % 2 == 1).all()


def test_drafts_accepted_by_an_identical_target(orc):
    S, K, V = 6, 3, 900
    c = synth.sd_case(5, S, K, V, 3.0, 1.0)
    d = orc.draft_sample(c.drf, S * K, V, 1.0, synth.uniforms(9, S * K))
    tgt = c.tgt.reshape(S, K + 1, V).copy()
    tgt[:, :K] = c.drf.reshape(S, K, V)
    o = orc.sd_verify(tgt.reshape(S * (K + 1), V), c.drf, d["tokens"], S, K, V, 1.0, c.uniforms)
    np.testing.assert_array_equal(o["accept_len"], K)


def test_bad_inputs(orc):
    z = np.zeros((2, 4), np.float32)
    u = np.zeros(2, np.float32)
    assert orc.draft_sample(z, 2, 4, 0.0, u, raise_on_error=False)["status"] == orc.EINVAL
    z[1] = np.nan
    assert orc.draft_sample(z, 2, 4, 1.0, u, raise_on_error=False)["status"] == orc.ENONFINITE
