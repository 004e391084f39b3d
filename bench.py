"""Benchmark: one SMC-SD step per iteration on the Llama-3-vocabulary workload.

Workload (synthetic): 8 prompts x 16 particles, K=4 draft tokens, V=128256, bf16 logits
(draft ~ N(0,3), target = draft + N(0,1)), T=1, ESS threshold N/2, systematic resampling and
the page-table remap of a 2048-token context in 16-token pages. One step = smc_step: every
target and draft logit read once (logsumexp of 1152 rows), the log-weight update, the
(K+1)-th token of every particle, per-group ESS, resampling and page-table remap.

Timing: W warm-up steps, then exactly K steps on the device, bracketed by a barrier and a
synchronize, timed with CUDA events on the launching stream. Steps are replayed from a CUDA
graph that cycles through 4 logit sets of 295.5 MB each (the working set exceeds the 129 MB
L2, so no step is served from cache). Metric: verified positions/s = S*(K+1) per step.

`--impl reference` times the float64 CPU oracle (single thread) on a bounded sample of the
same workload and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified positions/s at V=128256 bf16; achieved HBM GB/s as % of GB300 peak"
UNIT = "positions/s"
NSETS = 4


DEFAULT_WORKLOAD = "smc_sd_step_8x16_k4_v128256_bf16"
# name -> (kind, config); "smc": one smc_step per step, "smc_logq": one smc_step_logq per step
# (the draft given as the sampler's log q), "sd": one sd_verify per step, "draft": one
# draft_sample over the S*K draft rows per step
WORKLOADS = {
    DEFAULT_WORKLOAD: ("smc", "SMC_LLAMA3"),
    "smc_sd_step_4x64_k8_v151936_bf16_power": ("smc", "SMC_QWEN_POWER"),
    "smc_sd_step_logq_8x16_k4_v128256_bf16": ("smc_logq", "SMC_LLAMA3"),
    "sd_verify_128_k4_v128256_bf16": ("sd", "SMC_LLAMA3"),
    "sd_verify_16_k4_v32000_bf16": ("sd", None),
    "draft_sample_512_v128256_bf16": ("draft", "SMC_LLAMA3"),
    "pacer_ragged_verify_64_v32256_bf16": ("pacer", None),
}


def workload_config(name: str = DEFAULT_WORKLOAD):
    from smc_reweight_resample_gb300 import synth

    kind, cname = WORKLOADS[name]
    if kind == "pacer":  # 64 sequences, blocks of 4 up to 5, d=2048, then the ragged verify
        cfg = synth.SMCConfig("pacer_ragged_64_v32256", 1, 64, 20, 32256, 3.0, 1.0, 1.0, 1.0, 256)
        config = {"workload": name, "S": 64, "b": 4, "max_blocks": 5, "d": 2048, "t0": 0.5,
                  "rho": 1.1, "V": 32256, "temperature": 1.0,
                  "positions": "verified positions = target rows of the ragged verify, sum(L+1)"}
        return cfg, config, kind
    if cname is None:  # the Mistral-vocabulary SD verify: 16 sequences, K=4, V=32000
        cfg = synth.SMCConfig("sd_mistral_16_k4_v32000", 1, 16, 4, 32000, 3.0, 1.0, 1.0, 1.0, 256)
    else:
        cfg = getattr(synth, cname)
    lb = logit_bytes(cfg, kind)
    big = NSETS * lb > 129e6
    config = {
        "workload": name, "K": cfg.K, "V": cfg.V, "temperature": cfg.temperature,
        "positions_per_step": positions_per_step(cfg, kind),
        "l2": (f"inputs larger than L2: {NSETS} rotating logit sets of {lb / 1e6:.1f} MB"
               if big else
               f"{NSETS} rotating logit sets of {lb / 1e6:.1f} MB; L2 flushed (256 MB "
               f"write) before every timed graph replay of {NSETS} calls"),
    }
    if kind in ("smc", "smc_logq"):
        config.update({"G": cfg.G, "N": cfg.N, "alpha": cfg.alpha,
                       "ess_threshold": cfg.ess_threshold, "ctx": cfg.ctx, "page": cfg.page})
        if kind == "smc_logq":
            config["draft"] = ("tokens and log q from draft_sample on the draft logits (before the "
                               "timed region, as the draft tokens of the logits workload); the step "
                               "reads the target logits only")
    elif kind == "draft":
        config.update({"rows": cfg.S * cfg.K, "positions": "drafted tokens (one per draft row)"})
    else:
        config.update({"S": cfg.S})
    return cfg, config, kind


def logit_bytes(cfg, kind: str = "smc") -> int:
    if kind == "draft":  # the draft rows only
        return cfg.S * cfg.K * cfg.V * 2
    if kind == "smc_logq":  # the target rows only
        return cfg.S * (cfg.K + 1) * cfg.V * 2
    return cfg.S * (2 * cfg.K + 1) * cfg.V * 2


def positions_per_step(cfg, kind: str = "smc") -> int:
    """Verified positions (target rows) per step; for the draft sampler, drafted tokens."""
    return cfg.S * cfg.K if kind == "draft" else cfg.S * (cfg.K + 1)


def algorithmic_bytes(cfg, kind: str = "smc") -> int:
    """Bytes one step must move: every logit once, plus tokens, uniforms, weights and tables."""
    if kind == "sd":  # draft tokens, uniforms, accept lengths and tokens out
        return logit_bytes(cfg) + cfg.S * cfg.K * 4 + cfg.S * (cfg.K + 1) * 4 + cfg.S * 8
    if kind == "draft":  # uniforms in, tokens and log q out
        return logit_bytes(cfg, kind) + cfg.S * cfg.K * 12
    small = (cfg.S * cfg.K * 4 + cfg.S * 4 + cfg.G * 4 + cfg.S * 4 * 2 + cfg.S * 4 + cfg.G * 8
             + 2 * cfg.S * cfg.pages_per_seq * 4 + cfg.S * cfg.pages_per_seq * 4)
    if kind == "smc_logq":  # plus the given log q of every draft token
        return logit_bytes(cfg, kind) + small + cfg.S * cfg.K * 4
    return logit_bytes(cfg) + small


KERNELS_PER_STEP = 2  # stream pass (which also zeroes the refcounts) and finishing pass;
# groups of more than 32 particles add the stand-alone resampling and page-table kernels
SD_KERNELS_PER_CALL = 6  # stream, epilogue, rows stream and epilogue, residual stream and draw
KERNEL_NOTE = {
    "smc": "one smc_step call: stream_tma_kernel and finish_kernel (kernel shares in "
           "profiles/launches_<workload>.md); achieved = algorithmic bytes per step / device time "
           "per step",
    "sd": "one sd_verify call: the stream over every row, the SD epilogue, the final-token rows "
          "and residual passes with their epilogues; achieved = algorithmic bytes per call / "
          "device time per call",
    "smc_logq": "one smc_step_logq call: stream_tma_kernel over the target rows and finish_kernel; "
                "achieved = algorithmic bytes per step / device time per step",
    "draft": "one draft_sample call: stream_tma_kernel (precise partials of every row) and "
             "finish_kernel (one inverse-CDF draw per row); achieved = algorithmic bytes per call "
             "/ device time per call",
}


def _code_only(text: str) -> bytes:
    """C/C++ source without its comments and with whitespace runs collapsed: what compiles."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split()).encode()


def _source_sha256() -> str:
    """Hash of the code (comments and layout aside) of the CUDA sources and the ABI header, as
    recorded beside the ncu counters."""
    import hashlib

    h = hashlib.sha256()
    d = os.path.join(ROOT, "smc_reweight_resample_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        h.update(f.encode())
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()))
    with open(os.path.join(ROOT, "include", "smcsd.h"), encoding="utf-8") as fh:
        h.update(_code_only(fh.read()))
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per step from the committed ncu summary, or None once the kernels have changed
    since those counters were taken (or if there is no summary for this workload)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != _source_sha256():
        return None
    return float(kv["traffic_bytes_per_step"])


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if len(inside) < 2:  # a short timed region: take the samples around it
            inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0]
            window = "timed region +-1 s (region shorter than the 100 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in inside for i in range(4) if p[5 + i].lower() == "active"})
        pw = [num(p[3]) for _, p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(inside), "window": window}


# --------------------------------------------------------------------------------------------
# oracle CPU baseline
# --------------------------------------------------------------------------------------------

_GROUP_CACHE = {}


def _group_inputs(cfg, seed: int):
    """One prompt group's inputs (N particles), generated once and reused by the timing loop."""
    key = (cfg.name, seed)
    if key not in _GROUP_CACHE:
        from smc_reweight_resample_gb300 import synth

        x = synth.smc_step_inputs(
            synth.SMCConfig(cfg.name, 1, cfg.N, cfg.K, cfg.V, cfg.sigma_d, cfg.sigma_t,
                            cfg.temperature, cfg.alpha, cfg.ctx, cfg.page), seed, 0)
        _GROUP_CACHE[key] = x
    return _GROUP_CACHE[key]


def cpu_model() -> str:
    """The host CPU's model name (or the Arm part numbers) from /proc/cpuinfo."""
    names, parts = [], set()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k in ("model name", "Model Name", "cpu model") and v:
                    names.append(v)
                elif k == "CPU part":
                    parts.add(v)
    except OSError:
        return "unknown"
    if names:
        return names[0]
    import platform

    known = {"0xd4f": "Arm Neoverse V2"}  # MIDR part number of the Neoverse V2 core
    desc = ", ".join(known.get(p.lower(), f"CPU part {p}") for p in sorted(parts)) or "unknown"
    return f"{platform.machine()} ({desc})"


def oracle_positions(cfg, seconds: float, seed: int = 0, threads: int = 1):
    """Runs the float64 oracle on whole particles (and their group's ESS, resampling and
    page-table remap) of the workload for about `seconds` of oracle time, cycling through one
    pre-generated group of N particles. threads == 1: one particle per call; threads > 1: the
    group's N particles per call, split over `threads` host threads. Returns (positions/s,
    positions, particles, seconds)."""
    import numpy as np

    import oracle
    from smc_reweight_resample_gb300 import synth

    oracle.build()
    x = _group_inputs(cfg, seed)
    K, V, N = cfg.K, cfg.V, cfg.N
    table = synth.initial_page_table(N, cfg.pages_per_seq)
    t_oracle = 0.0
    positions = 0
    particles = 0
    lw = np.zeros(N, np.float32)
    per_call = 1 if threads <= 1 else N
    while t_oracle < seconds or particles == 0:
        j = particles % N
        n = min(per_call, N - j)
        tgt = x.tgt[j * (K + 1):(j + n) * (K + 1)]
        drf = x.drf[j * K:(j + n) * K]
        toks = x.draft_tokens[j * K:(j + n) * K]
        t0 = time.perf_counter()
        o = oracle.smc_reweight(tgt, drf, toks, n, K, V, cfg.temperature, cfg.alpha,
                                x.bonus_uniforms[j:j + n], lw[j:j + n], threads=threads)
        lw[j:j + n] = o["logw"]
        if j + n == N:
            r = oracle.ess_resample(lw, 1, N, cfg.ess_threshold, x.resample_uniforms[:1])
            oracle.pagetable_remap(r["ancestors"], r["resampled"], 1, N, table, cfg.pages_per_seq,
                                   num_pages=N * cfg.pages_per_seq)
            lw = r["logw"]
        t_oracle += time.perf_counter() - t0
        positions += n * (K + 1)
        particles += n
    return positions / t_oracle, positions, particles, t_oracle


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(cfg, seconds=12.0):
    """Two legs of the oracle on the host: every core (the particles of a group split over
    threads; the line's value) and one thread."""
    cores = host_cores()
    model = cpu_model()
    rate1, pos1, parts1, secs1 = oracle_positions(cfg, seconds / 2)
    rate, pos, parts, secs = oracle_positions(cfg, seconds / 2, threads=cores)
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu": model,
            "sample": f"{parts} particles ({pos} positions, {parts * (2 * cfg.K + 1)} rows of "
                      f"{cfg.V} bf16 logits) cycling through one group of {cfg.N} particles of the "
                      f"same workload, the group's particles split over {cores} threads, with the "
                      f"group's ESS, resampling and remap; {secs:.1f} s of float64 oracle time",
            "single_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                              "sample": f"{parts1} particles ({pos1} positions) one per call, "
                                        f"{secs1:.1f} s"}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cfg, config, kind = workload_config(args.workload)
    if kind != "smc":
        print(json.dumps({"impl": "reference", "unavailable": "the timed oracle leg covers the "
                          "SMC workloads only"}), flush=True)
        return 0
    config["parallelism"] = parallelism(kind, args.gpus)
    cores = host_cores()
    budget = 120.0
    per_step = max(0.02, budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_positions(cfg, per_step, threads=cores)
    pos_total = 0
    t_all = 0.0
    for _ in range(args.steps):
        rate, pos, parts, secs = oracle_positions(cfg, per_step, threads=cores)
        pos_total += pos
        t_all += secs
    value = pos_total / t_all
    rate1, pos1, _, secs1 = oracle_positions(cfg, min(10.0, budget / 4))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * t_all / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"each step: whole particles of the workload for about "
                                   f"{per_step:.2f} s of float64 oracle time, a group's particles "
                                   f"split over {cores} threads ({pos_total} positions in total)",
                         "single_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                                           "sample": f"{pos1} positions, {secs1:.1f} s"}},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def parallelism(kind: str, world: int) -> str:
    unit_name = {"smc": "prompt groups", "smc_logq": "prompt groups", "sd": "sequences",
                 "draft": "draft rows"}.get(kind, "units")
    return f"replicas x{world} (independent {unit_name} per GPU, no collective)"


# --------------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------------

def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (all ranks get it). One process: x itself."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, units_per_step: int, steps: int, seconds: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return world * units_per_step * steps / seconds


def gpu_numa_cpus(gpu_index):
    """(NUMA node, its CPUs) of the GPU's PCI device, or (None, None) if unknown."""
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        dom, rest = bus.split(":", 1)
        sysfs = f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest.lower()}/numa_node"
        with open(sysfs) as f:
            node = int(f.read().strip())
        if node < 0:
            return None, None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            if not part:
                continue
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return node, (cpus or None)
    except Exception:
        return None, None


def h2d_link(dev, nbytes: int, gpu_index) -> dict:
    """GB/s of a plain host-to-device copy of nbytes from pinned memory (best of 5), with the
    pinned buffer placed by the default policy, and allocated while the process runs on the
    CPUs of the GPU's NUMA node (so that its pages land on that node)."""
    import torch

    def measure():
        h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        h.fill_(1)
        d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        best = float("inf")
        for _ in range(5):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            d.copy_(h, non_blocking=True)
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        del h, d
        return nbytes / best / 1e9

    out = {"bytes": nbytes, "default": measure()}
    node, cpus = gpu_numa_cpus(gpu_index)
    out["gpu_numa_node"] = node
    if cpus:
        all_cpus = os.sched_getaffinity(0)
        os.sched_setaffinity(0, cpus)
        try:
            out["gpu_local_node"] = measure()
        finally:
            os.sched_setaffinity(0, all_cpus)
        out["use_local"] = out["gpu_local_node"] > 1.05 * out["default"]
        out["local_cpus"], out["all_cpus"] = sorted(cpus), sorted(all_cpus)
    return out


def run_pacer(args):
    """PACER's blockwise stop followed by the ragged verify of the lengths it chose, as one step:
    pacer_block_stop (which writes the ragged row offsets on the device) then sd_verify over the
    packed rows. Four input sets (hidden states and the packed logits for the lengths their stop
    rule yields) rotate through a graph of four steps."""
    import numpy as np
    import torch

    from smc_reweight_resample_gb300 import _binding as B
    from smc_reweight_resample_gb300 import build as _build
    from smc_reweight_resample_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and rank != 0:
        return 0  # replicas of this extra workload are not timed
    cfg, config, kind = workload_config(args.workload)
    torch.cuda.set_device(local)
    _build.build()
    B.load()
    dev = torch.device("cuda", local)
    S, b, nb, d, V, T = 64, 4, 5, 2048, cfg.V, 1.0
    Kmax = b * nb
    sets, pos, alg = [], [], []
    for i in range(NSETS):
        cs = synth.pacer_case(200 + i, S=S, b=b, max_blocks=nb, d=d)
        h = torch.from_numpy(cs.hidden.view(np.int16)).view(torch.bfloat16).to(dev)
        w = torch.from_numpy(cs.w.view(np.int16)).view(torch.bfloat16).to(dev)
        L, _, _, _ = B.pacer_block_stop(h, w, cs.c, S, b, nb, d, cs.t0, cs.rho)
        lengths = L.cpu().numpy().astype(np.int64)
        tgt_full, drf_full = synth.torch_logits_pair(300 + i, S, Kmax, V, cfg.sigma_d, cfg.sigma_t, dev)
        it = np.concatenate([s * (Kmax + 1) + np.arange(lengths[s] + 1) for s in range(S)])
        idr = np.concatenate([s * Kmax + np.arange(lengths[s]) for s in range(S)])
        tgt = tgt_full[torch.from_numpy(it).to(dev)].contiguous()
        drf = drf_full[torch.from_numpy(idr).to(dev)].contiguous()
        del tgt_full, drf_full
        toks = synth.torch_gumbel_draft_tokens(400 + i, drf, T)
        u = torch.from_numpy(synth.uniforms(rank, S * (Kmax + 1), stream=500 + i)).to(dev)
        outs = (torch.empty(S, dtype=torch.int32, device=dev), torch.empty(S * nb, device=dev),
                torch.empty(S + 1, dtype=torch.int32, device=dev),
                torch.empty(S + 1, dtype=torch.int32, device=dev))
        sets.append((h, w, cs, tgt, drf, toks, u, outs))
        pos.append(int((lengths + 1).sum()))
        # hidden states up to the stop, the head, every packed logit once, tokens, uniforms, outputs
        alg.append(int(lengths.sum()) * d * 2 + d * 2 + (tgt.numel() + drf.numel()) * 2
                   + int(lengths.sum()) * 4 + S * (Kmax + 1) * 4 + S * 4 * 4 + 2 * (S + 1) * 4)
    torch.cuda.synchronize()
    ws_p = B.Workspace(B.OP_PACER_BLOCK_STOP, S, 0, 1, dev)
    ws_v = B.Workspace(B.OP_SD_VERIFY, S, Kmax, V, dev)
    acc = torch.empty(S, dtype=torch.int32, device=dev)
    tok = torch.empty(S, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        h, w, cs, tgt, drf, toks, u, (L, bs, to, do) = sets[i % NSETS]
        lib = B.load()
        wp, n = ws_p.args
        rc = lib.pacer_block_stop(B._ptr(h), B._ptr(w), float(cs.c), S, b, nb, d, float(cs.t0),
                                  float(cs.rho), B._ptr(L), B._ptr(bs), B._ptr(to), B._ptr(do),
                                  wp, n, B._stream(stream))
        B._check(rc, "pacer_block_stop")
        B.sd_verify(tgt, drf, toks, S, Kmax, V, T, u, tgt_offsets=to, drf_offsets=do, ws=ws_v,
                    accept_len=acc, out_token=tok, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, NSETS)):
            step(i)
    stream.synchronize()
    assert B.check_status(ws_p, stream) == 0 and B.check_status(ws_v, stream) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(NSETS):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    total = sum(x[3].numel() * 2 + x[4].numel() * 2 + x[0].numel() * 2 for x in sets)
    small_set = total <= 129e6
    flush = torch.empty((256 << 20) if small_set else 0, dtype=torch.uint8, device=dev)
    reps = max(1, args.steps // NSETS)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(vis.split(",")[local] if vis else local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ms = 0.0
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if small_set:
            for r in range(reps):
                flush.fill_(r & 255)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                e1.synchronize()
                ms += e0.elapsed_time(e1)
        else:
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    time.sleep(0.3)
    clocks.stop()
    assert B.check_status(ws_p, stream) == 0 and B.check_status(ws_v, stream) == 0
    steps = reps * NSETS
    ms_per_step = ms / steps
    positions = sum(pos) / NSETS
    alg_bytes = sum(alg) / NSETS
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (ms_per_step / 1000.0) / 1e9
    config.update({"l2": (f"{NSETS} rotating input sets of {total / NSETS / 1e6:.1f} MB on average"
                          + ("; L2 flushed (256 MB write) before every timed graph replay"
                             if small_set else ", larger than L2 together")),
                   "mean_length": positions / S - 1, "positions_per_step": positions})
    line = {
        "metric": METRIC, "value": positions / (ms_per_step / 1000.0), "unit": UNIT, "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "one pacer_block_stop and one ragged sd_verify; achieved = "
                               "algorithmic bytes per step / device time per step",
                     "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": steps * (1 + SD_KERNELS_PER_CALL),
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfg, config, kind = workload_config(args.workload)
    config["parallelism"] = parallelism(kind, world)

    base = None
    if rank == 0 and not args.no_cpu_baseline and kind == "smc":
        base = cpu_baseline(cfg, args.cpu_seconds)  # before any GPU work

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from smc_reweight_resample_gb300 import _binding as B
    from smc_reweight_resample_gb300 import build as _build
    from smc_reweight_resample_gb300 import synth

    _build.build()
    B.load()
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    dev = torch.device("cuda", local)
    sets = []
    for i in range(NSETS):
        tgt, drf = synth.torch_logits_pair(1000 * rank + i, S, K, V, cfg.sigma_d, cfg.sigma_t, dev)
        toks = synth.torch_gumbel_draft_tokens(77 + 1000 * rank + i, drf, cfg.temperature)
        ub = torch.from_numpy(synth.uniforms(rank, S, stream=100 + 2 * i)).to(dev)
        ur = torch.from_numpy(synth.uniforms(rank, G, stream=101 + 2 * i)).to(dev)
        if kind == "smc_logq":  # the draft sampler's tokens and log q stand in for the draft rows
            ud = torch.from_numpy(synth.uniforms(rank, S * K, stream=700 + i)).to(dev)
            toks, logq = B.draft_sample(drf, S * K, V, cfg.temperature, ud)
            drf = logq
        sets.append((tgt, drf, toks, ub, ur))
    torch.cuda.synchronize()
    ws = (B.Workspace(B.OP_DRAFT_SAMPLE, S * K, 0, V, dev) if kind == "draft" else
          B.Workspace(B.OP_SMC_STEP if kind in ("smc", "smc_logq") else B.OP_SD_VERIFY, S, K, V, dev))
    draft_out = (torch.empty(S * K, dtype=torch.int32, device=dev),
                 torch.empty(S * K, dtype=torch.float32, device=dev))
    usd = [torch.from_numpy(synth.uniforms(rank, S * (K + 1), stream=300 + i)).to(dev)
           for i in range(NSETS)]
    sd_out = (torch.empty(S, dtype=torch.int32, device=dev), torch.empty(S, dtype=torch.int32, device=dev))
    small_set = NSETS * logit_bytes(cfg, kind) <= 129e6
    flush = torch.empty((256 << 20) if small_set else 0, dtype=torch.uint8, device=dev)
    logw = torch.zeros(S, dtype=torch.float32, device=dev)
    tables = [torch.from_numpy(synth.initial_page_table(S, P)).to(dev),
              torch.empty(S * P, dtype=torch.int32, device=dev)]
    outs = dict(bonus_token=torch.empty(S, dtype=torch.int32, device=dev),
                ancestors=torch.empty(S, dtype=torch.int32, device=dev),
                ess=torch.empty(G, dtype=torch.float32, device=dev),
                resampled=torch.empty(G, dtype=torch.int32, device=dev),
                refcount=torch.empty(S * P, dtype=torch.int32, device=dev))

    def step(i, stream):
        tgt, drf, toks, ub, ur = sets[i % NSETS]
        if kind == "sd":
            B.sd_verify(tgt, drf, toks, S, K, V, cfg.temperature, usd[i % NSETS], ws=ws,
                        accept_len=sd_out[0], out_token=sd_out[1], stream=stream)
            return
        if kind == "draft":
            B.draft_sample(drf, S * K, V, cfg.temperature, usd[i % NSETS][:S * K], ws=ws,
                           tokens=draft_out[0], logq=draft_out[1], stream=stream)
            return
        if kind == "smc_logq":  # (drf holds log q here)
            B.smc_step_logq(tgt, toks, drf, G, N, K, V, cfg.temperature, cfg.alpha, ub, logw,
                            cfg.ess_threshold, ur, table_in=tables[i % 2], pages_per_seq=P,
                            num_pages=S * P, ws=ws, table_out=tables[(i + 1) % 2], stream=stream,
                            **outs)
            return
        B.smc_step(tgt, drf, toks, G, N, K, V, cfg.temperature, cfg.alpha, ub, logw,
                   cfg.ess_threshold, ur, table_in=tables[i % 2], pages_per_seq=P,
                   num_pages=S * P, ws=ws, table_out=tables[(i + 1) % 2], stream=stream, **outs)

    stream = torch.cuda.Stream(device=dev)
    # warm-up, eager
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i, stream)
    stream.synchronize()
    assert B.check_status(ws, stream) == 0
    # The timed steps are replayed from one CUDA graph of gsteps consecutive steps (a multiple
    # of NSETS, so that consecutive steps always read different logit sets and the page-table
    # double buffer stays aligned; up to 256 steps, so that a short run is one replay and not a
    # string of replays with a launch gap between each); steps beyond a whole number of replays
    # run eagerly. A second graph of NSETS steps serves the L2-flushed timing of small working
    # sets and the spread below.
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i, stream)
        torch.cuda.synchronize()
        return g

    graph = capture(NSETS)
    gsteps = NSETS * max(1, min(256, args.steps) // NSETS)
    big_graph = graph if gsteps == NSETS or small_set else capture(gsteps)
    for _ in range(2):
        graph.replay()
        if big_graph is not graph:
            big_graph.replay()
    torch.cuda.synchronize()

    reps, tail = divmod(args.steps, gsteps if big_graph is not graph else NSETS)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(vis.split(",")[local] if vis else local)
    clocks.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ms_flushed = None
    with torch.cuda.stream(stream):
        if small_set:  # working set inside L2: time each graph replay after an L2 flush
            ms_flushed = 0.0
            for r in range(reps):
                flush.fill_(r & 255)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                e1.synchronize()
                ms_flushed += e0.elapsed_time(e1)
            ev0.record(stream)
            ev1.record(stream)
        else:
            ev0.record(stream)
            for _ in range(reps):
                big_graph.replay()
            for i in range(tail):
                step(i, stream)
            ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    time.sleep(0.3)
    clocks.stop()
    ms = ev0.elapsed_time(ev1)
    if ms_flushed is not None:
        ms = ms_flushed
        args.steps = reps * NSETS
    ms = max_over_ranks(ms, dev)
    # spread of the step time, after the timed region: 200 graph replays, each between its own
    # events (with the L2 flush before each when the inputs fit in L2)
    per_step = []
    with torch.cuda.stream(stream):
        for r in range(200):
            if small_set:
                flush.fill_(r & 255)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            per_step.append(e0.elapsed_time(e1) / NSETS)
    per_step.sort()
    spread = {"p10": per_step[20], "median": per_step[100], "p90": per_step[180],
              "unit": "ms per step", "replays": 200,
              "note": f"each a graph replay of {NSETS} steps between two events, after the timed region"}
    assert B.check_status(ws, stream) == 0
    ms_per_step = ms / args.steps
    positions = positions_per_step(cfg, kind)
    value = aggregate_rate(world, positions, args.steps, ms / 1000.0)

    # e2e: inputs from pinned host memory, results back to the host, every step
    e2e = None
    if not args.no_e2e and kind == "smc":
        e_steps = min(args.steps, args.e2e_steps)
        # the host link: a plain pinned copy of one step's input bytes, with the pinned buffer
        # placed by the default policy and placed on the GPU's own NUMA node; the faster
        # placement then holds the e2e host buffers
        link = h2d_link(dev, logit_bytes(cfg), vis.split(",")[local] if vis else local)
        if link.get("use_local"):
            os.sched_setaffinity(0, link["local_cpus"])
        host_sets = []
        for i in range(2):
            tgt, drf, toks, ub, ur = sets[i]
            host_sets.append([x.cpu().pin_memory() for x in (tgt, drf, toks, ub, ur)])
        dsets = [[torch.empty_like(x) for x in sets[0]] for _ in range(2)]
        hout = [torch.empty(S, dtype=torch.int32).pin_memory(), torch.empty(S, dtype=torch.int32).pin_memory(),
                torch.empty(G, dtype=torch.float32).pin_memory(), torch.empty(G, dtype=torch.int32).pin_memory(),
                torch.empty(S, dtype=torch.float32).pin_memory()]
        h2d = sum(x.numel() * x.element_size() for x in host_sets[0])
        d2h = sum(x.numel() * x.element_size() for x in hout)
        # double-buffered: the copies of step i+1 run on their own stream while step i computes;
        # a device set is refilled only after the step that read it has finished
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]

        def issue_copy(i):
            b = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(used[b])
                for h, d in zip(host_sets[i % 2], dsets[b]):
                    d.copy_(h, non_blocking=True)
                copied[b].record(copy_stream)

        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for b in range(2):
            used[b].record(stream)
        issue_copy(0)
        for i in range(e_steps):
            if i + 1 < e_steps:
                issue_copy(i + 1)
            b = i % 2
            with torch.cuda.stream(stream):
                stream.wait_event(copied[b])
                tgt, drf, toks, ub, ur = dsets[b]
                B.smc_step(tgt, drf, toks, G, N, K, V, cfg.temperature, cfg.alpha, ub, logw,
                           cfg.ess_threshold, ur, table_in=tables[i % 2], pages_per_seq=P,
                           num_pages=S * P, ws=ws, table_out=tables[(i + 1) % 2], stream=stream,
                           **outs)
                used[b].record(stream)
                for h, d in zip(hout, (outs["bonus_token"], outs["ancestors"], outs["ess"],
                                        outs["resampled"], logw)):
                    h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        et = max_over_ranks(t1 - t0, dev)
        e2e = {"value": aggregate_rate(world, positions, e_steps, et), "unit": UNIT,
               "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e_steps,
               "note": "pinned host inputs copied to the device, smc_step through the C ABI, "
                       "results copied back, every step; the copies of step i+1 (own stream) "
                       "overlap the compute of step i",
               "h2d_copy_GBps": {k: v for k, v in link.items() if k not in ("local_cpus", "all_cpus")}}
        if link.get("use_local"):
            os.sched_setaffinity(0, link["all_cpus"])

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    peak, peak_kind = measured_peaks()
    alg = algorithmic_bytes(cfg, kind)
    achieved = alg / (ms_per_step / 1000.0) / 1e9
    traffic = args.ncu_traffic if args.ncu_traffic is not None else recorded_traffic(config["workload"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": KERNEL_NOTE[kind],
                     "traffic_source": "profiles/traffic_<workload>.txt (ncu dram bytes of one step)",
                     "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": alg,
                     "frac_of_8TBps_spec": achieved / 8000.0},
        "step_ms_spread": spread, "cpu_baseline": base, "e2e": e2e,
        "gpu_launches": args.steps * (SD_KERNELS_PER_CALL if kind == "sd" else
                                      KERNELS_PER_STEP if kind == "draft" else
                                      KERNELS_PER_STEP + (2 if cfg.N > 32 else 0)),
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------------------------
# sweeps (measurement only, not the bench line)
# --------------------------------------------------------------------------------------------

SWEEP_TEMPERATURES = (0.5, 0.7, 1.0, 1.4, 2.0)
SWEEP_PARTICLES = (2, 4, 8, 16, 32, 64, 128)


def _graph_ms(step, n_steps, stream):
    """Device ms per call of step(i) replayed from a CUDA graph of NSETS calls."""
    import torch

    with torch.cuda.stream(stream):
        for i in range(NSETS):
            step(i)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(NSETS):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    reps = max(1, n_steps // NSETS)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / (reps * NSETS)


def sweep_temperature(args):
    """SD against SMC-SD as the sampling temperature rises ("Faster LLM Inference via Sequential
    Monte Carlo", sec. 4 "robustness": SD's throughput falls with its acceptance rate while
    SMC-SD emits K+1 tokens per particle whatever the temperature). On the 8 x 16 particle,
    K=4, V=128256 bf16 shape: per temperature, SD verify of the 128 sequences (acceptance length,
    emitted tokens, device time per call) and the fused SMC-SD step (ESS, resampling rate, device
    time per step), both through the C ABI on the synthetic logits of the workload."""
    import numpy as np
    import torch

    from smc_reweight_resample_gb300 import _binding as B
    from smc_reweight_resample_gb300 import synth

    B.load()
    cfg = synth.SMC_LLAMA3
    S, K, V, G, N, P = cfg.S, cfg.K, cfg.V, cfg.G, cfg.N, cfg.pages_per_seq
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    rows = []
    for T in SWEEP_TEMPERATURES:
        sets = []
        for i in range(NSETS):
            tgt, drf = synth.torch_logits_pair(500 + i, S, K, V, cfg.sigma_d, cfg.sigma_t, dev)
            toks = synth.torch_gumbel_draft_tokens(600 + i, drf, T)
            sets.append((tgt, drf, toks))
        usd = [torch.from_numpy(synth.uniforms(7, S * (K + 1), stream=700 + i)).to(dev)
               for i in range(NSETS)]
        wsd = B.Workspace(B.OP_SD_VERIFY, S, K, V, dev)
        acc = [torch.empty(S, dtype=torch.int32, device=dev) for _ in range(NSETS)]
        tok = torch.empty(S, dtype=torch.int32, device=dev)

        def sd_step(i):
            t, d, x = sets[i % NSETS]
            B.sd_verify(t, d, x, S, K, V, T, usd[i % NSETS], ws=wsd, accept_len=acc[i % NSETS],
                        out_token=tok, stream=stream)

        sd_ms = _graph_ms(sd_step, args.sweep_steps, stream)
        assert B.check_status(wsd, stream) == 0
        a = np.concatenate([acc[i].cpu().numpy() for i in range(NSETS)]).astype(np.float64)
        sd_tokens = float((a + 1).mean())  # accepted drafts + the residual or bonus token

        ws = B.Workspace(B.OP_SMC_STEP, S, K, V, dev)
        logw = torch.zeros(S, dtype=torch.float32, device=dev)
        tables = [torch.from_numpy(synth.initial_page_table(S, P)).to(dev),
                  torch.empty(S * P, dtype=torch.int32, device=dev)]
        ub = [torch.from_numpy(synth.uniforms(8, S, stream=800 + i)).to(dev) for i in range(NSETS)]
        ur = [torch.from_numpy(synth.uniforms(8, G, stream=900 + i)).to(dev) for i in range(NSETS)]
        outs = [dict(bonus_token=torch.empty(S, dtype=torch.int32, device=dev),
                     ancestors=torch.empty(S, dtype=torch.int32, device=dev),
                     ess=torch.empty(G, dtype=torch.float32, device=dev),
                     resampled=torch.empty(G, dtype=torch.int32, device=dev),
                     refcount=torch.empty(S * P, dtype=torch.int32, device=dev))
                for _ in range(NSETS)]

        def smc_step(i):
            t, d, x = sets[i % NSETS]
            B.smc_step(t, d, x, G, N, K, V, T, cfg.alpha, ub[i % NSETS], logw, cfg.ess_threshold,
                       ur[i % NSETS], table_in=tables[i % 2], pages_per_seq=P, num_pages=S * P,
                       ws=ws, table_out=tables[(i + 1) % 2], stream=stream, **outs[i % NSETS])

        smc_ms = _graph_ms(smc_step, args.sweep_steps, stream)
        assert B.check_status(ws, stream) == 0
        ess = np.concatenate([o["ess"].cpu().numpy() for o in outs]) / N
        res = np.concatenate([o["resampled"].cpu().numpy() for o in outs])
        rows.append({
            "temperature": T,
            "sd": {"mean_accept_len": float(a.mean()), "tokens_per_seq_per_call": sd_tokens,
                   "ms_per_call": sd_ms, "tokens_per_s": S * sd_tokens / (sd_ms / 1e3)},
            "smc": {"tokens_per_particle_per_step": K + 1, "ms_per_step": smc_ms,
                    "tokens_per_s": S * (K + 1) / (smc_ms / 1e3),
                    "mean_ess_over_n": float(ess.mean()), "resample_rate": float(res.mean())},
        })
        del sets, wsd, ws
        torch.cuda.empty_cache()
    return {"sweep": "temperature", "workload": "8 prompts x 16 particles, K=4, V=128256 bf16",
            "data": "synthetic: draft ~ N(0,3), target = draft + N(0,1); draft tokens by Gumbel-max "
                    "at each temperature", "steps_per_point": args.sweep_steps, "rows": rows}


def sweep_particles(args):
    """Error of the importance-weighted estimate against the number of particles ("Faster LLM
    Inference via Sequential Monte Carlo", sec. 3: L2 bias and MSE fall as O(1/N), L1 bias as
    O(1/sqrt(N))). A known target on V=8 (context-free rows p_k, q_k, K=2): G groups of N
    particles each draw their K tokens from q, smc_reweight gives the weights, and each group
    estimates p_0 by the self-normalised weighted frequencies of its first tokens. Reported per
    N: the squared bias |E est - p_0|^2 (L2 bias), the mean squared error and the L1 bias."""
    import numpy as np
    import torch
    from scipy.special import softmax

    from smc_reweight_resample_gb300 import _binding as B
    from smc_reweight_resample_gb300 import synth

    B.load()
    Vs, Ks = 8, 2
    rng = np.random.default_rng(11)
    zd = rng.normal(0, 1.0, (Ks + 1, Vs)).astype(np.float32)
    zt = (zd + rng.normal(0, 0.8, (Ks + 1, Vs))).astype(np.float32)
    q = softmax(zd.astype(np.float64), axis=1)
    p0 = softmax(zt[0].astype(np.float64))
    rows = []
    total = 1 << 21  # particles per N
    for N in SWEEP_PARTICLES:
        G = total // N
        S = G * N
        ux = synth.uniforms(12, S * Ks, stream=N).reshape(S, Ks).astype(np.float64)
        x = np.stack([np.minimum(np.searchsorted(np.cumsum(q[k]) / q[k].sum(), ux[:, k],
                                                 side="right"), Vs - 1)
                      for k in range(Ks)], axis=1).astype(np.int32)
        tgt = torch.from_numpy(zt).cuda().repeat(S, 1).contiguous()
        drf = torch.from_numpy(zd[:Ks]).cuda().repeat(S, 1).contiguous()
        lw = torch.zeros(S, device="cuda")
        B.smc_reweight(tgt, drf, torch.from_numpy(x.reshape(-1)).cuda(), S, Ks, Vs, 1.0, 1.0,
                       torch.from_numpy(synth.uniforms(13, S, stream=N)).cuda(), lw)
        w = np.exp(lw.cpu().numpy().astype(np.float64)).reshape(G, N)
        onehot = np.eye(Vs)[x[:, 0]].reshape(G, N, Vs)
        est = (w[:, :, None] * onehot).sum(1) / w.sum(1)[:, None]  # [G, Vs]
        bias = est.mean(0) - p0
        rows.append({"N": N, "groups": G, "l2_bias_sq": float((bias ** 2).sum()),
                     "mse": float(((est - p0) ** 2).sum(1).mean()),
                     "l1_bias": float(np.abs(bias).sum()),
                     # what sampling noise alone adds to l2_bias_sq (sum of Var(est) / G)
                     "l2_bias_sq_noise_floor": float(est.var(0).sum() / G)})
        del tgt, drf, lw
        torch.cuda.empty_cache()
    return {"sweep": "particles", "target": "V=8, K=2, context-free rows; estimate of p_0",
            "particles_per_point": total, "rows": rows}


def run_sweep(args):
    import torch

    torch.cuda.set_device(0)
    out = sweep_temperature(args) if args.sweep == "temperature" else sweep_particles(args)
    print(json.dumps(out), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS),
                    help="the default is the headline workload; the others are extra measurements")
    ap.add_argument("--ncu-traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture")
    ap.add_argument("--sweep", choices=["temperature", "particles"], default=None,
                    help="print a measurement sweep instead of the bench line")
    ap.add_argument("--sweep-steps", type=int, default=400)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep:
        return run_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    if WORKLOADS[args.workload][0] == "pacer":
        return run_pacer(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
