"""smc_step_static (the fused step on the library's own scratch area, no workspace argument)
against smc_step with a caller workspace, through the C ABI: identical results on consecutive
calls, including a change of shape between calls, the device-side status of a failing call
delivered to `status` with the next call clean again, and a shape too large for the area
rejected before any device work. Kept in the last file collected, so that it also runs after
every other test in the same process."""
import numpy as np
import pytest
import torch

from smc_reweight_resample_gb300 import synth
from gpu_util import dev, dev_logits

pytestmark = pytest.mark.gpu

OUTPUTS = ("bonus_token", "ancestors", "ess", "resampled", "table_out", "refcount")


def cfg_of(G, N, K, V, ctx):
    return synth.SMCConfig("no_alloc", G, N, K, V, 3.0, 1.0, 1.0, 1.0, ctx)


def step_pair(smcsd, cfg, seed, step, lw_ws, lw_st, ws):
    """One step through both entry points from equal log-weights; returns both output sets."""
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    x = synth.smc_step_inputs(cfg, seed, step)
    t, d, toks = dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens)
    ub, ur = dev(x.bonus_uniforms), dev(x.resample_uniforms)
    table = dev(synth.initial_page_table(S, P))
    a = smcsd.smc_step(t, d, toks, G, N, K, V, 1.0, 1.0, ub, lw_ws, N / 2.0, ur, table_in=table,
                       pages_per_seq=P, num_pages=S * P, ws=ws)
    assert smcsd.check_status(ws) == 0
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    b = smcsd.smc_step_static(t, d, toks, G, N, K, V, 1.0, 1.0, ub, lw_st, N / 2.0, ur,
                              table_in=table, pages_per_seq=P, num_pages=S * P, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return a, b


def assert_same(a, b, lw_ws, lw_st):
    for k in OUTPUTS:
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(lw_ws, lw_st)


def test_static_matches_workspace_on_consecutive_calls(smcsd):
    cfg = cfg_of(4, 16, 4, 20000, 256)
    ws = smcsd.Workspace(smcsd.OP_SMC_STEP, cfg.S, cfg.K, cfg.V)
    lw0 = np.random.default_rng(11).normal(0, 2, cfg.S).astype(np.float32)
    lw_ws, lw_st = dev(lw0.copy()), dev(lw0.copy())
    for step in range(2):
        a, b = step_pair(smcsd, cfg, 11, step, lw_ws, lw_st, ws)
        assert_same(a, b, lw_ws, lw_st)


def test_static_across_a_change_of_shape(smcsd):
    """Two shapes in turn: the scratch's layout (and the cached exp table's place in it) moves."""
    for cfg, seed in ((cfg_of(2, 16, 3, 30000, 128), 21), (cfg_of(4, 8, 5, 12000, 64), 22),
                      (cfg_of(2, 16, 3, 30000, 128), 23)):
        ws = smcsd.Workspace(smcsd.OP_SMC_STEP, cfg.S, cfg.K, cfg.V)
        lw0 = np.random.default_rng(seed).normal(0, 2, cfg.S).astype(np.float32)
        lw_ws, lw_st = dev(lw0.copy()), dev(lw0.copy())
        for step in range(2):
            a, b = step_pair(smcsd, cfg, seed, step, lw_ws, lw_st, ws)
            assert_same(a, b, lw_ws, lw_st)


def test_static_reports_device_status_and_recovers(smcsd):
    cfg = cfg_of(2, 16, 2, 8192, 64)
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    x = synth.smc_step_inputs(cfg, 31, 0)
    bad = x.tgt.copy()
    bad[3, 100] = 0x7FC0  # a bf16 NaN logit in one target row
    ub, ur = dev(x.bonus_uniforms), dev(x.resample_uniforms)
    table = dev(synth.initial_page_table(S, P))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lw = torch.zeros(S, device="cuda")
    smcsd.smc_step_static(dev_logits(bad), dev_logits(x.drf), dev(x.draft_tokens), G, N, K, V, 1.0,
                          1.0, ub, lw, N / 2.0, ur, table_in=table, pages_per_seq=P,
                          num_pages=S * P, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == smcsd.ERR_NONFINITE
    # the next call starts from a cleared scratch and matches the workspace path
    ws = smcsd.Workspace(smcsd.OP_SMC_STEP, S, K, V)
    lw_ws, lw_st = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
    a, b = step_pair(smcsd, cfg, 31, 1, lw_ws, lw_st, ws)
    assert_same(a, b, lw_ws, lw_st)


def test_static_rejects_a_shape_larger_than_its_area(smcsd):
    G, N, K, V = 4, 64, 8, 151936  # needs about 63 MiB of scratch
    assert smcsd.workspace_size(smcsd.OP_SMC_STEP, G * N, K, V) > smcsd.STATIC_SCRATCH_BYTES
    tiny = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(16, dtype=torch.int32, device="cuda")
    f32 = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(smcsd.SMCSDError) as e:
        smcsd.smc_step_static(tiny, tiny, i32, G, N, K, V, 1.0, 1.0, f32, f32, N / 2.0, f32,
                              bonus_token=i32, ancestors=i32, ess=f32, resampled=i32)
    assert e.value.code == smcsd.ERR_WORKSPACE
