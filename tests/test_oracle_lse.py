"""Pins of the oracle's scaled log-softmax normaliser (the target/draft probabilities that
"Faster LLM Inference via Sequential Monte Carlo", sec. 2 step 3, weighs particles by).

Closed forms and a library routine, none of which repeats the oracle's own loop:
constant rows give z/T + log V, a single unmasked token gives z/T, random rows agree with
numpy's pairwise ``logaddexp.reduce``, and the power target alpha*z/T equals temperature
T/alpha.
"""
import math

import numpy as np
import pytest

from smc_reweight_resample_gb300 import synth


@pytest.mark.parametrize("V", [1, 7, 1000, 32000])
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_constant_row_closed_form(orc, V, T):
    z = np.full((1, V), 1.75, np.float32)
    L = orc.row_lse(z, 0, V, 1.0 / T)
    assert abs(L - (1.75 / T + math.log(V))) < 1e-12 * max(1.0, abs(L))


def test_one_unmasked_token(orc):
    V = 513
    z = np.full((1, V), -np.inf, np.float32)
    z[0, 200] = 3.5
    for T in (1.0, 0.25):
        assert orc.row_lse(z, 0, V, 1.0 / T) == pytest.approx(3.5 / T, abs=1e-13)


def test_bf16_widening_exact(orc):
    # bf16 0x3FC0 = 1.5, 0xC000 = -2.0: lse of [1.5, -2.0] = 1.5 + log(1 + e^-3.5)
    z = np.array([[0x3FC0, 0xC000]], np.uint16)
    assert orc.row_lse(z, 0, 2, 1.0) == pytest.approx(1.5 + math.log1p(math.exp(-3.5)), abs=1e-14)


@pytest.mark.parametrize("seed", range(4))
def test_random_rows_match_library(orc, seed):
    V = 4099
    rng = np.random.default_rng(seed)
    z = synth.bf16_bits(rng.normal(0, 3, (3, V)).astype(np.float32))
    zf = synth.bf16_widen(z).astype(np.float64)
    for row in range(3):
        for T in (1.0, 0.7):
            ref = np.logaddexp.reduce(zf[row] / T)
            assert orc.row_lse(z, row, V, 1.0 / T) == pytest.approx(ref, abs=1e-10)


def test_masked_tokens_ignored(orc):
    V = 64
    rng = np.random.default_rng(5)
    z = rng.normal(0, 2, (1, V)).astype(np.float32)
    zm = z.copy()
    zm[0, ::3] = -np.inf
    ref = np.logaddexp.reduce(z[0, np.isfinite(zm[0])].astype(np.float64))
    assert orc.row_lse(zm, 0, V, 1.0) == pytest.approx(ref, abs=1e-12)


def test_power_target_is_temperature_T_over_alpha(orc):
    V = 3000
    rng = np.random.default_rng(7)
    z = synth.bf16_bits(rng.normal(0, 3, (1, V)).astype(np.float32))
    T, alpha = 0.7, 4.0
    a = orc.row_lse(z, 0, V, alpha / T)
    b = orc.row_lse(z, 0, V, 1.0 / (T / alpha))
    assert a == pytest.approx(b, rel=1e-13)


def test_nonfinite_rows_rejected(orc):
    V = 8
    for bad in (np.nan, np.inf):
        z = np.zeros((1, V), np.float32)
        z[0, 3] = bad
        with pytest.raises(orc.OracleError) as e:
            orc.row_lse(z, 0, V, 1.0)
        assert e.value.code == orc.ENONFINITE
    z = np.full((1, V), -np.inf, np.float32)
    with pytest.raises(orc.OracleError) as e:
        orc.row_lse(z, 0, V, 1.0)
    assert e.value.code == orc.ENONFINITE
