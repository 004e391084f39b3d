"""smc_step_static (the fused step on the library's own scratch area, no workspace argument)
against smc_step with a caller workspace, through the C ABI: identical results on consecutive
calls, including a change of shape between calls, a call recorded in a CUDA graph and replayed
after calls of another shape, the device-side status of a failing call delivered to `status`
with the next call clean again, and a shape too large for the area rejected before any device
work. Kept in the last file collected, so that it also runs after every other test in the same
process."""
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


def test_static_replayed_after_calls_of_another_shape(smcsd):
    """A recorded call replayed after calls of a larger shape, whose sections cover where the
    recorded shape's sections lie, must still match the workspace path: the cached exp table
    the replay copies may not have been overwritten by the calls in between."""
    a_cfg, b_cfg = cfg_of(2, 16, 3, 30000, 128), cfg_of(8, 16, 5, 40000, 64)
    S, K, V, G, N, P = a_cfg.S, a_cfg.K, a_cfg.V, a_cfg.G, a_cfg.N, a_cfg.pages_per_seq
    x = synth.smc_step_inputs(a_cfg, 41, 0)
    t, d, toks = dev_logits(x.tgt), dev_logits(x.drf), dev(x.draft_tokens)
    ub, ur = dev(x.bonus_uniforms), dev(x.resample_uniforms)
    table = dev(synth.initial_page_table(S, P))
    lw0 = np.random.default_rng(41).normal(0, 2, S).astype(np.float32)
    # reference: the workspace path from the same log-weights
    ws = smcsd.Workspace(smcsd.OP_SMC_STEP, S, K, V)
    lw_ws = dev(lw0.copy())
    want = smcsd.smc_step(t, d, toks, G, N, K, V, 1.0, 1.0, ub, lw_ws, N / 2.0, ur, table_in=table,
                          pages_per_seq=P, num_pages=S * P, ws=ws)
    assert smcsd.check_status(ws) == 0
    # eager call of shape A (publishes its table), then the same call recorded in a graph
    lw_st = dev(lw0.copy())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = dict(bonus_token=torch.empty(S, dtype=torch.int32, device="cuda"),
                ancestors=torch.empty(S, dtype=torch.int32, device="cuda"),
                ess=torch.empty(G, device="cuda"), resampled=torch.empty(G, dtype=torch.int32, device="cuda"),
                table_out=torch.empty_like(table), refcount=torch.empty(S * P, dtype=torch.int32, device="cuda"))

    def call_a(stream=None):
        return smcsd.smc_step_static(t, d, toks, G, N, K, V, 1.0, 1.0, ub, lw_st, N / 2.0, ur,
                                     table_in=table, pages_per_seq=P, num_pages=S * P,
                                     status=status, stream=stream, **outs)

    call_a()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call_a(stream)
    torch.cuda.synchronize()
    # eager calls of shape B in between
    for step in range(2):
        y = synth.smc_step_inputs(b_cfg, 42, step)
        sb = torch.zeros(1, dtype=torch.int32, device="cuda")
        smcsd.smc_step_static(dev_logits(y.tgt), dev_logits(y.drf), dev(y.draft_tokens), b_cfg.G,
                              b_cfg.N, b_cfg.K, b_cfg.V, 1.0, 1.0, dev(y.bonus_uniforms),
                              torch.zeros(b_cfg.S, device="cuda"), b_cfg.N / 2.0,
                              dev(y.resample_uniforms),
                              table_in=dev(synth.initial_page_table(b_cfg.S, b_cfg.pages_per_seq)),
                              pages_per_seq=b_cfg.pages_per_seq,
                              num_pages=b_cfg.S * b_cfg.pages_per_seq, status=sb)
        torch.cuda.synchronize()
        assert int(sb.item()) == 0
    # replay A from the reference's starting log-weights
    lw_st.copy_(dev(lw0.copy()))
    status.fill_(12345)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_same(want, outs, lw_ws, lw_st)


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
