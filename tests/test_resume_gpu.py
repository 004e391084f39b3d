"""Checkpoint / resume and run-to-run determinism of the fused SMC-SD step on the GPU.

The state an SMC-SD run carries from step to step ("Faster LLM Inference via Sequential Monte
Carlo", sec. 2-3) is the particles' log-weights and their page-table rows; the workspace is
scratch. So 16 steps, a copy of that state to the host, fresh device buffers and a fresh
workspace filled from the copy, and 16 more steps must give, bit for bit, what 32 steps in one
run give. A second run of the 32 steps must repeat the first exactly: every reduction runs in a
fixed order, whichever warp or block computes it."""
import numpy as np
import pytest
import torch

from smc_reweight_resample_gb300 import synth
from gpu_util import dev, dev_logits, host

pytestmark = pytest.mark.gpu

CFG = synth.SMCConfig("resume", 8, 16, 4, 8192, 3.0, 1.0, 1.0, 1.0, 256)
KEYS = ("bonus_token", "ancestors", "ess", "resampled", "table_out", "refcount")


def run(smcsd, steps, lw, table, first_step=0, ws=None):
    cfg = CFG
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    ws = ws or smcsd.Workspace(smcsd.OP_SMC_STEP, S, K, V)
    outs = []
    for step in range(first_step, first_step + steps):
        x = synth.smc_step_inputs(cfg, 5, step)
        o = smcsd.smc_step(dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens), G, N, K, V,
                           cfg.temperature, cfg.alpha, dev(x.bonus_uniforms), lw,
                           cfg.ess_threshold, dev(x.resample_uniforms), table_in=table,
                           pages_per_seq=P, num_pages=S * P, ws=ws)
        assert smcsd.check_status(ws) == 0
        outs.append({k: host(o[k]).copy() for k in KEYS})
        table = o["table_out"]
    return outs, lw, table


def fresh_state():
    return (torch.zeros(CFG.S, dtype=torch.float32, device="cuda"),
            dev(synth.initial_page_table(CFG.S, CFG.pages_per_seq)))


def test_resume_from_host_checkpoint_equals_one_run(smcsd):
    lw, table = fresh_state()
    straight, lw_a, table_a = run(smcsd, 32, lw, table)
    assert any(o["resampled"].any() for o in straight)  # the run exercises resampling

    lw, table = fresh_state()
    first, lw_mid, table_mid = run(smcsd, 16, lw, table)
    ckpt = (host(lw_mid).copy(), host(table_mid).copy())  # the whole state, on the host
    del lw_mid, table_mid
    torch.cuda.synchronize()
    lw_r, table_r = dev(ckpt[0].copy()), dev(ckpt[1].copy())
    second, lw_b, table_b = run(smcsd, 16, lw_r, table_r, first_step=16)
    for i, (a, b) in enumerate(zip(straight, first + second)):
        for k in KEYS:
            assert np.array_equal(a[k], b[k]), (i, k)
    assert torch.equal(lw_a, lw_b)
    assert torch.equal(table_a, table_b)


def test_two_runs_are_bit_identical(smcsd):
    lw, table = fresh_state()
    a, lw_a, _ = run(smcsd, 8, lw, table)
    lw, table = fresh_state()
    b, lw_b, _ = run(smcsd, 8, lw, table)
    for i, (x, y) in enumerate(zip(a, b)):
        for k in KEYS:
            assert np.array_equal(x[k], y[k]), (i, k)
    assert torch.equal(lw_a, lw_b)
