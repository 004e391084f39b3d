"""The benchmark's host-side arithmetic (no GPU): workload shapes, algorithmic bytes, positions,
the whole-job rate over ranks, and the recorded ncu traffic's tie to the CUDA sources."""
import os

import pytest

import bench


def test_headline_workload_bytes_and_positions():
    cfg, config, kind = bench.workload_config(bench.DEFAULT_WORKLOAD)
    assert kind == "smc" and (cfg.G, cfg.N, cfg.K, cfg.V) == (8, 16, 4, 128256)
    # every target and draft logit once: 128 particles x 9 rows x 128256 bf16 logits
    assert bench.logit_bytes(cfg) == 128 * 9 * 128256 * 2 == 295_501_824
    assert bench.algorithmic_bytes(cfg) == 295_702_624  # plus tokens, uniforms, weights, tables
    assert config["positions_per_step"] == bench.positions_per_step(cfg) == 128 * 5
    assert "larger than L2" in config["l2"]


def test_other_workloads():
    cfg, config, kind = bench.workload_config("smc_sd_step_4x64_k8_v151936_bf16_power")
    assert bench.logit_bytes(cfg) == 256 * 17 * 151936 * 2 == 1_322_450_944
    cfg, config, kind = bench.workload_config("draft_sample_512_v128256_bf16")
    assert kind == "draft" and config["positions_per_step"] == 512
    assert bench.algorithmic_bytes(cfg, kind) == 512 * 128256 * 2 + 512 * 12
    cfg, config, kind = bench.workload_config("sd_verify_16_k4_v32000_bf16")
    assert kind == "sd" and "L2 flushed" in config["l2"]


def test_aggregate_rate_and_single_process_max():
    assert bench.aggregate_rate(4, 640, 100, 2.0) == 4 * 640 * 100 / 2.0
    assert bench.max_over_ranks(1.25, "cpu") == 1.25  # no process group: the value itself


def test_recorded_traffic_follows_the_sources():
    name = bench.DEFAULT_WORKLOAD
    path = os.path.join(bench.ROOT, "profiles", f"traffic_{name}.txt")
    assert os.path.exists(path)
    kv = dict(line.split(":", 1) for line in open(path) if ":" in line and not line.startswith("#"))
    recorded = float(kv["traffic_bytes_per_step"])
    if bench.recorded_traffic(name) is None:
        pytest.skip("the CUDA sources changed since the counters were taken: bench reports null")
    assert bench.recorded_traffic(name) == recorded
    # DRAM traffic is the logits read once plus a little: no re-reads
    assert 1.0 <= recorded / bench.algorithmic_bytes(bench.workload_config(name)[0]) < 1.03


def test_pacer_workload_config():
    cfg, config, kind = bench.workload_config("pacer_ragged_verify_64_v32256_bf16")
    assert kind == "pacer" and config["S"] == 64 and config["V"] == 32256
    assert config["b"] * config["max_blocks"] == cfg.K == 20
