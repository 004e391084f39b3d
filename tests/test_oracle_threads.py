"""The oracle's thread split (contiguous blocks of sequences, particles or rows, each a call of
the same C function) gives the same bits as one call over everything: every sequence and
particle is computed on its own, and this checks that the block offsets are right."""
import numpy as np
import pytest

from smc_reweight_resample_gb300 import synth


def _same(a, b):
    for k in a:
        if k == "status":
            assert a[k] == b[k]
            continue
        np.testing.assert_array_equal(np.asarray(a[k]), np.asarray(b[k]), err_msg=k)


@pytest.mark.parametrize("threads", [2, 3, 8])
def test_sd_verify_fixed_and_ragged(orc, threads):
    c = synth.sd_case(5, 11, 3, 700, 3.0, 1.0, 0.9, "bf16")
    one = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, c.S, c.K, c.V, 0.9, c.uniforms)
    many = orc.sd_verify(c.tgt, c.drf, c.draft_tokens, c.S, c.K, c.V, 0.9, c.uniforms,
                         threads=threads)
    _same(one, many)
    r = synth.ragged_sd_case(6, np.array([4, 0, 8, 12, 4, 20, 16]), 333, K_max=20)
    one = orc.sd_verify(r.tgt, r.drf, r.draft_tokens, r.S, r.K, r.V, 1.0, r.uniforms,
                        tgt_offsets=r.tgt_offsets, drf_offsets=r.drf_offsets)
    many = orc.sd_verify(r.tgt, r.drf, r.draft_tokens, r.S, r.K, r.V, 1.0, r.uniforms,
                         tgt_offsets=r.tgt_offsets, drf_offsets=r.drf_offsets, threads=threads)
    _same(one, many)


@pytest.mark.parametrize("threads", [2, 5])
def test_smc_reweight_and_tilted(orc, threads):
    c = synth.sd_case(7, 13, 4, 900, 3.0, 1.0, 0.7, "bf16")
    u = synth.uniforms(7, 13, stream=3)
    lw0 = np.random.default_rng(7).normal(0, 1, 13).astype(np.float32)
    one = orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, 13, 4, 900, 0.7, 4.0, u, lw0)
    many = orc.smc_reweight(c.tgt, c.drf, c.draft_tokens, 13, 4, 900, 0.7, 4.0, u, lw0,
                            threads=threads)
    _same(one, many)
    rw = synth.log_rewards(7, 13)
    one = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, 13, 4, 900, 0.7, 2.0, u, lw0,
                                  target_mode=orc.TARGET_SEQUENCE, log_reward=rw, reward_scale=0.5)
    many = orc.smc_reweight_tilted(c.tgt, c.drf, c.draft_tokens, 13, 4, 900, 0.7, 2.0, u, lw0,
                                   target_mode=orc.TARGET_SEQUENCE, log_reward=rw,
                                   reward_scale=0.5, threads=threads)
    _same(one, many)


def test_draft_sample(orc):
    c = synth.sd_case(8, 6, 3, 500, 3.0, 1.0)
    u = synth.uniforms(8, 18, stream=4)
    one = orc.draft_sample(c.drf, 18, 500, 1.0, u)
    many = orc.draft_sample(c.drf, 18, 500, 1.0, u, threads=4)
    _same(one, many)


def test_error_status_is_the_single_call_status(orc):
    c = synth.sd_case(9, 8, 2, 300, 3.0, 1.0)
    toks = c.draft_tokens.copy()
    toks[11] = 300  # out of range in particle 5
    u = synth.uniforms(9, 8)
    one = orc.smc_reweight(c.tgt, c.drf, toks, 8, 2, 300, 1.0, 1.0, u, np.zeros(8, np.float32),
                           raise_on_error=False)
    many = orc.smc_reweight(c.tgt, c.drf, toks, 8, 2, 300, 1.0, 1.0, u, np.zeros(8, np.float32),
                            raise_on_error=False, threads=4)
    assert one["status"] == many["status"] == orc.ERANGE
