"""GPU parity of pacer_block_stop and pacer_block_stop_pos ("PACER: Blockwise Pre-verification
for Speculative Decoding with Adaptive Length", Methodik 1-3; position embeddings from
Methodik 1) and of the ragged verify that follows it, against the float64 oracle through the
C ABI."""
import numpy as np
import pytest
import torch

import oracle
from smc_reweight_resample_gb300 import synth
from gpu_util import DecisionLedger, dev, dev_logits, host
from test_parity_sd import run_sd

pytestmark = pytest.mark.gpu


def run_pacer(smcsd, cs, ledger):
    h = dev_logits(cs.hidden)
    w = dev_logits(cs.w)
    L, bs, to, do = smcsd.pacer_block_stop(h, w, cs.c, cs.S, cs.b, cs.max_blocks, cs.d, cs.t0, cs.rho)
    o = oracle.pacer_block_stop(cs.hidden, cs.w, cs.c, cs.S, cs.b, cs.max_blocks, cs.d, cs.t0, cs.rho)
    ledger.compare("length", host(L), o["lengths"], o["margin"])
    same = host(L) == o["lengths"]
    np.testing.assert_allclose(host(bs).reshape(cs.S, -1)[same], o["block_scores"].reshape(cs.S, -1)[same],
                               atol=1e-6, rtol=0)
    Lh = host(L)
    np.testing.assert_array_equal(host(do), np.concatenate([[0], np.cumsum(Lh)]))
    np.testing.assert_array_equal(host(to), np.concatenate([[0], np.cumsum(Lh + 1)]))
    return Lh


@pytest.mark.parametrize("seed", range(3))
def test_pacer_default_workload(smcsd, seed):
    L = DecisionLedger()
    run_pacer(smcsd, synth.pacer_case(seed), L)
    L.finish()


@pytest.mark.parametrize("t0,rho,c", [(0.3, 1.1, 0.0), (0.5, 1.0, 0.0), (0.45, 1.3, 0.2), (0.9, 1.1, 0.0)])
def test_pacer_thresholds(smcsd, t0, rho, c):
    cs = synth.pacer_case(7, t0=t0, rho=rho, c=c)
    L = DecisionLedger()
    run_pacer(smcsd, cs, L)
    L.finish()


def test_pacer_odd_dimension_scalar_path(smcsd):
    cs = synth.pacer_case(3, S=9, b=3, max_blocks=4, d=77)
    L = DecisionLedger()
    run_pacer(smcsd, cs, L)
    L.finish()


def test_pacer_then_ragged_verify(smcsd):
    """The whole PACER-style flow: stop rule -> lengths -> ragged verify over 32256 logits."""
    cs = synth.pacer_case(0)
    L = DecisionLedger()
    lengths = run_pacer(smcsd, cs, L)
    c = synth.ragged_sd_case(5, lengths, cs.V, K_max=cs.b * cs.max_blocks)
    run_sd(smcsd, c, L)
    L.finish()


def run_pacer_pos(smcsd, cs, pos_emb, ledger):
    L, bs, to, do = smcsd.pacer_block_stop_pos(dev_logits(cs.hidden), dev_logits(cs.w),
                                               dev_logits(pos_emb), cs.c, cs.S, cs.b, cs.max_blocks,
                                               cs.d, cs.t0, cs.rho)
    o = oracle.pacer_block_stop(cs.hidden, cs.w, cs.c, cs.S, cs.b, cs.max_blocks, cs.d, cs.t0,
                                cs.rho, pos_emb=pos_emb)
    ledger.compare("length", host(L), o["lengths"], o["margin"])
    same = host(L) == o["lengths"]
    np.testing.assert_allclose(host(bs).reshape(cs.S, -1)[same],
                               o["block_scores"].reshape(cs.S, -1)[same], atol=1e-6, rtol=0)
    Lh = host(L)
    np.testing.assert_array_equal(host(do), np.concatenate([[0], np.cumsum(Lh)]))
    np.testing.assert_array_equal(host(to), np.concatenate([[0], np.cumsum(Lh + 1)]))
    return Lh


@pytest.mark.parametrize("seed", range(3))
def test_pacer_pos_emb_default_workload(smcsd, seed):
    """Methodik 1: hidden states together with position embeddings (64 sequences, b=4, up to 5
    blocks, d=2048)."""
    cs = synth.pacer_case(seed)
    pe = synth.pacer_pos_emb(seed, cs.max_blocks, cs.b, cs.d)
    L = DecisionLedger()
    lengths = run_pacer_pos(smcsd, cs, pe, L)
    L.finish()
    assert len(set(lengths.tolist())) > 1


def test_pacer_pos_emb_scalar_path_and_ragged_verify(smcsd):
    """An odd dimension takes the scalar loads; the lengths then drive a ragged verify."""
    cs = synth.pacer_case(4, S=9, b=3, max_blocks=4, d=77)
    pe = synth.pacer_pos_emb(4, cs.max_blocks, cs.b, cs.d)
    L = DecisionLedger()
    lengths = run_pacer_pos(smcsd, cs, pe, L)
    c = synth.ragged_sd_case(6, lengths, cs.V, K_max=cs.b * cs.max_blocks)
    run_sd(smcsd, c, L)
    L.finish()
