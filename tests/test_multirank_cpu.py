"""The multi-GPU path on CPU ranks (gloo, world size 2): prompt groups split into blocks of
whole groups per rank give the same step as one process over all groups (groups are independent:
"Faster LLM Inference via Sequential Monte Carlo", sec. 2-3), and the bench's timing reduction
takes the slowest rank's time on every rank. The float64 oracle stands in for each rank's GPU."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from smc_reweight_resample_gb300 import shard, synth

CFG = synth.SMCConfig("multirank", 5, 8, 2, 600, 3.0, 1.5, 0.9, 1.0, 64)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def run_block(cfg, x, table, lw, s0, s1):
    """One rank's step over particles [s0, s1) (whole groups) with the oracle."""
    import oracle

    K, V, N, P = cfg.K, cfg.V, cfg.N, cfg.pages_per_seq
    S, G = s1 - s0, (s1 - s0) // N
    o = oracle.smc_reweight(x.tgt[s0 * (K + 1):s1 * (K + 1)], x.drf[s0 * K:s1 * K],
                            x.draft_tokens[s0 * K:s1 * K], S, K, V, cfg.temperature, cfg.alpha,
                            x.bonus_uniforms[s0:s1], lw[s0:s1])
    r = oracle.ess_resample(o["logw"], G, N, cfg.ess_threshold,
                            x.resample_uniforms[s0 // N:s1 // N])
    m = oracle.pagetable_remap(r["ancestors"], r["resampled"], G, N, table[s0 * P:s1 * P], P,
                               num_pages=cfg.S * P)
    return dict(bonus=o["bonus_token"], logw=r["logw"], anc=r["ancestors"],
                res=r["resampled"], table=m["table_out"], refcount=m["refcount"])


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        # timing: every rank gets the slowest rank's time
        got = bench.max_over_ranks(1.0 + 0.5 * rank, "cpu")
        # data: this rank's block of whole groups
        x = synth.smc_step_inputs(CFG, 3, 0)
        table = synth.initial_page_table(CFG.S, CFG.pages_per_seq)
        lw = np.random.default_rng(4).normal(0, 1, CFG.S).astype(np.float32)
        s0, s1 = shard.particle_range(CFG.G, CFG.N, world, rank)
        mine = run_block(CFG, x, table, lw, s0, s1)
        parts = [None] * world
        dist.all_gather_object(parts, (rank, s0, s1, mine))
        if rank == 0:
            out.put((got, parts))
        else:
            out.put((got, None))
    finally:
        dist.destroy_process_group()


def test_group_range_covers_every_group_once():
    for G in range(0, 13):
        for world in range(1, 6):
            seen = []
            for r in range(world):
                g0, g1 = shard.group_range(G, world, r)
                assert g1 - g0 in (G // world, G // world + 1)
                seen.extend(range(g0, g1))
            assert seen == list(range(G))
    with pytest.raises(ValueError):
        shard.group_range(4, 2, 2)


def test_two_ranks_equal_one_process(orc):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(abs(got - 1.5) == 0 for got, _ in results)  # max of 1.0 and 1.5 on both ranks
    parts = next(parts for _, parts in results if parts is not None)
    # one process over all groups
    x = synth.smc_step_inputs(CFG, 3, 0)
    table = synth.initial_page_table(CFG.S, CFG.pages_per_seq)
    lw = np.random.default_rng(4).normal(0, 1, CFG.S).astype(np.float32)
    full = run_block(CFG, x, table, lw, 0, CFG.S)
    P = CFG.pages_per_seq
    refcount = np.zeros_like(full["refcount"])
    for rank, s0, s1, mine in sorted(parts, key=lambda t: t[0]):
        g0, g1 = s0 // CFG.N, s1 // CFG.N
        np.testing.assert_array_equal(mine["bonus"], full["bonus"][s0:s1])
        np.testing.assert_array_equal(mine["logw"], full["logw"][s0:s1])
        np.testing.assert_array_equal(mine["anc"], full["anc"][s0:s1])
        np.testing.assert_array_equal(mine["res"], full["res"][g0:g1])
        np.testing.assert_array_equal(mine["table"], full["table"][s0 * P:s1 * P])
        refcount += mine["refcount"]
    np.testing.assert_array_equal(refcount, full["refcount"])
    assert full["res"].any()  # the case resamples at least one group
