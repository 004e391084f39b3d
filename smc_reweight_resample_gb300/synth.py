"""Seeded synthetic inputs for the verify / reweight / resample path.

This module is shared by the tests, the benchmark and the oracle side. It holds no
arithmetic of the method itself: it only draws random numbers and lays them out.

* Logits: a draft row is N(0, sigma_d); the matching target row is that draft row plus
  independent N(0, sigma_t) noise (the second parameter is a standard deviation). Values
  are drawn in float32 and rounded to bf16 (round to nearest even) for the bf16 cases.
  Each sequence has K+1 target rows and K draft rows; target row K (the bonus position)
  is built the same way from a draft row that is never stored.
* Uniforms: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014), counter based: output i of stream (seed, stream) is
  mix64(seed_state + (i+1) * 0x9E3779B97F4A7C15); the top 24 bits times 2^-24 give a
  float32 in [0, 1). Independent of numpy and torch versions.
* Draft tokens: each draft token is drawn from its own draft row at temperature T by the
  Gumbel-max trick (argmax of z/T plus Gumbel noise). This stands in for the draft model's
  sampler, which precedes the verify step and is not part of it.
* Hidden states for the stop rule: N(0,1) rounded to bf16; head weights N(0, 1/d); position
  embeddings N(0,1) rounded to bf16.
* Log-rewards of a reward-tilted target: N(0,1) float32 per particle.

The logit distributions and vocabulary sizes follow the synthetic workloads stated for
the path (Mistral-size V=32000, Llama-3 V=128256, Qwen2.5 V=151936, DeepSeek-Coder
V=32256). No benchmark data is used.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM = np.uint64(0xD1B54A32D192ED03)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniforms(seed: int, n: int, stream: int = 0, offset: int = 0) -> np.ndarray:
    """``n`` float32 uniforms in [0,1) from SplitMix64 stream (seed, stream), outputs
    ``offset .. offset+n-1``."""
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (np.uint64(stream & 0xFFFFFFFF) * _STREAM)
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = _mix64(state + i * _GAMMA)
    return ((z >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)).astype(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even; NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    r = ((b >> 16) & 1) + 0x7FFF
    out = ((b + r) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed & 0xFFFFFFFF, stream])


def logits_pair(seed: int, S: int, K: int, V: int, sigma_d: float, sigma_t: float,
                dtype: str = "bf16"):
    """Target [S*(K+1), V] and draft [S*K, V] logits (uint16 bf16 bits or float32)."""
    rng = _rng(seed, 11)
    tgt = np.empty((S, K + 1, V), np.uint16 if dtype == "bf16" else np.float32)
    drf = np.empty((S, max(K, 0), V), tgt.dtype)
    for s in range(S):
        d = rng.normal(0.0, sigma_d, (K + 1, V)).astype(np.float32)
        t = (d + rng.normal(0.0, sigma_t, (K + 1, V)).astype(np.float32)).astype(np.float32)
        if dtype == "bf16":
            tgt[s] = bf16_bits(t)
            drf[s] = bf16_bits(d[:K])
        else:
            tgt[s] = t
            drf[s] = d[:K]
    return tgt.reshape(S * (K + 1), V), drf.reshape(S * K, V)


def widen(logits: np.ndarray) -> np.ndarray:
    return bf16_widen(logits) if logits.dtype == np.uint16 else logits


def gumbel_draft_tokens(seed: int, drf: np.ndarray, V: int, temperature: float) -> np.ndarray:
    """One token per draft row, drawn from that row at temperature T by Gumbel-max."""
    rows = drf.shape[0] if drf.ndim == 2 else drf.size // V
    rng = _rng(seed, 23)
    out = np.empty(rows, np.int32)
    z = widen(drf.reshape(rows, V))
    for r in range(rows):
        g = -np.log(-np.log(rng.random(V) * (1.0 - 2e-16) + 1e-16))
        out[r] = int(np.argmax(z[r].astype(np.float64) / temperature + g))
    return out


# ------------------------------------------------------------------------------------
# named workloads
# ------------------------------------------------------------------------------------

@dataclass
class SDCase:
    S: int
    K: int
    V: int
    temperature: float
    tgt: np.ndarray
    drf: np.ndarray
    draft_tokens: np.ndarray
    uniforms: np.ndarray
    tgt_offsets: np.ndarray | None = None
    drf_offsets: np.ndarray | None = None

    @property
    def dtype_code(self) -> int:
        return 1 if self.tgt.dtype == np.uint16 else 0


def sd_case(seed: int, S: int, K: int, V: int, sigma_d: float, sigma_t: float,
            temperature: float = 1.0, dtype: str = "bf16") -> SDCase:
    tgt, drf = logits_pair(seed, S, K, V, sigma_d, sigma_t, dtype)
    toks = gumbel_draft_tokens(seed + 1, drf, V, temperature) if K > 0 else np.zeros(0, np.int32)
    u = uniforms(seed, S * (K + 1), stream=1)
    return SDCase(S, K, V, temperature, tgt, drf, toks, u)


def sd_tiny(seed: int = 0) -> SDCase:
    """Tiny SD verify: 4 sequences, K=2, V=1000, fp32, draft N(0,2), target + N(0,0.5)."""
    return sd_case(seed, 4, 2, 1000, 2.0, 0.5, 1.0, "fp32")


def sd_mistral(seed: int = 0, K: int = 4) -> SDCase:
    """SD verify at the Mistral vocabulary: 16 sequences, K in {2,4,6}, V=32000, bf16."""
    return sd_case(seed, 16, K, 32000, 3.0, 1.0, 1.0, "bf16")


@dataclass
class SMCConfig:
    name: str
    G: int
    N: int
    K: int
    V: int
    sigma_d: float
    sigma_t: float
    temperature: float
    alpha: float
    ctx: int
    page: int = 16
    steps: int = 32

    @property
    def S(self) -> int:
        return self.G * self.N

    @property
    def pages_per_seq(self) -> int:
        return self.ctx // self.page

    @property
    def ess_threshold(self) -> float:
        return self.N / 2.0


SMC_LLAMA3 = SMCConfig("smc_llama3_8x16_k4_v128256", 8, 16, 4, 128256, 3.0, 1.0, 1.0, 1.0, 2048)
SMC_QWEN_POWER = SMCConfig("smc_qwen25_power_4x64_k8_v151936", 4, 64, 8, 151936, 3.0, 1.5, 0.7, 4.0,
                           4096)


@dataclass
class SMCStepInputs:
    tgt: np.ndarray
    drf: np.ndarray
    draft_tokens: np.ndarray
    bonus_uniforms: np.ndarray
    resample_uniforms: np.ndarray


def smc_step_inputs(cfg: SMCConfig, seed: int, step: int) -> SMCStepInputs:
    s = seed * 1000003 + step
    tgt, drf = logits_pair(s, cfg.S, cfg.K, cfg.V, cfg.sigma_d, cfg.sigma_t, "bf16")
    toks = gumbel_draft_tokens(s + 1, drf, cfg.V, cfg.temperature)
    ub = uniforms(seed, cfg.S, stream=100 + 2 * step)
    ur = uniforms(seed, cfg.G, stream=101 + 2 * step)
    return SMCStepInputs(tgt, drf, toks, ub, ur)


def initial_page_table(cfg_S: int, pages_per_seq: int) -> np.ndarray:
    """Particle s owns pages s*P .. s*P+P-1 (distinct physical pages)."""
    return np.arange(cfg_S * pages_per_seq, dtype=np.int32)


@dataclass
class PacerCase:
    S: int
    b: int
    max_blocks: int
    d: int
    c: float
    t0: float
    rho: float
    hidden: np.ndarray
    w: np.ndarray
    V: int = 32256
    sigma_d: float = 3.0
    sigma_t: float = 1.0


def pacer_case(seed: int = 0, S: int = 64, b: int = 4, max_blocks: int = 5, d: int = 2048,
               t0: float = 0.5, rho: float = 1.1, c: float = 0.0) -> PacerCase:
    """Stop-rule inputs: hidden N(0,1) bf16 [S, max_blocks*b, d], head w ~ N(0, 1/d)."""
    rng = _rng(seed, 31)
    h = bf16_bits(rng.normal(0.0, 1.0, (S, max_blocks * b, d)).astype(np.float32))
    w = bf16_bits(rng.normal(0.0, 1.0 / np.sqrt(d), d).astype(np.float32))
    return PacerCase(S, b, max_blocks, d, c, t0, rho, h, w)


def pacer_pos_emb(seed: int, max_blocks: int, b: int, d: int, sigma: float = 1.0) -> np.ndarray:
    """Position embeddings for the stop rule's head: N(0, sigma) bf16 [max_blocks*b, d], one
    row per draft position, shared by all sequences."""
    rng = _rng(seed, 37)
    return bf16_bits(rng.normal(0.0, sigma, (max_blocks * b, d)).astype(np.float32))


def log_rewards(seed: int, S: int, sigma: float = 1.0) -> np.ndarray:
    """Per-particle log-rewards for a reward-tilted target: N(0, sigma) float32 [S]."""
    rng = _rng(seed, 41)
    return rng.normal(0.0, sigma, S).astype(np.float32)


def ragged_sd_case(seed: int, lengths: np.ndarray, V: int, sigma_d: float = 3.0,
                   sigma_t: float = 1.0, temperature: float = 1.0, K_max: int | None = None) -> SDCase:
    """Packed ragged verify inputs: sequence s has lengths[s] draft rows and lengths[s]+1
    target rows; offsets are row offsets into the packed buffers."""
    lengths = np.asarray(lengths, dtype=np.int32)
    S = lengths.size
    K = int(lengths.max()) if K_max is None else int(K_max)
    rng = _rng(seed, 41)
    tgt_rows, drf_rows = [], []
    for s in range(S):
        L = int(lengths[s])
        d = rng.normal(0.0, sigma_d, (L + 1, V)).astype(np.float32)
        t = (d + rng.normal(0.0, sigma_t, (L + 1, V)).astype(np.float32)).astype(np.float32)
        tgt_rows.append(bf16_bits(t))
        drf_rows.append(bf16_bits(d[:L]))
    tgt = np.concatenate(tgt_rows, 0)
    drf = np.concatenate(drf_rows, 0) if lengths.sum() > 0 else np.zeros((0, V), np.uint16)
    to = np.zeros(S + 1, np.int32)
    do = np.zeros(S + 1, np.int32)
    to[1:] = np.cumsum(lengths + 1)
    do[1:] = np.cumsum(lengths)
    toks = gumbel_draft_tokens(seed + 1, drf, V, temperature) if drf.shape[0] else np.zeros(0, np.int32)
    u = uniforms(seed, S * (K + 1), stream=1)
    return SDCase(S, K, V, temperature, tgt, drf, toks, u, to, do)


# ------------------------------------------------------------------------------------
# device-side generation for large benchmark inputs (torch is used only as an RNG and
# for device memory here)
# ------------------------------------------------------------------------------------

def torch_logits_pair(seed: int, S: int, K: int, V: int, sigma_d: float, sigma_t: float,
                      device: str = "cuda"):
    """Same recipe as ``logits_pair`` drawn with torch's device RNG (bf16 tensors)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    d = torch.randn((S, K + 1, V), generator=g, device=device, dtype=torch.float32) * sigma_d
    t = d + torch.randn((S, K + 1, V), generator=g, device=device, dtype=torch.float32) * sigma_t
    tgt = t.to(torch.bfloat16).reshape(S * (K + 1), V).contiguous()
    drf = d[:, :K].to(torch.bfloat16).reshape(S * K, V).contiguous()
    del d, t
    return tgt, drf


def torch_gumbel_draft_tokens(seed: int, drf, temperature: float):
    """Gumbel-max draw of one token per draft row, on the device."""
    import torch

    g = torch.Generator(device=drf.device)
    g.manual_seed(seed)
    out = torch.empty(drf.shape[0], dtype=torch.int32, device=drf.device)
    for r0 in range(0, drf.shape[0], 64):
        z = drf[r0:r0 + 64].float() / temperature
        u = torch.rand(z.shape, generator=g, device=drf.device, dtype=torch.float32)
        u = u.clamp_(1e-12, 1.0 - 1e-7)
        out[r0:r0 + 64] = torch.argmax(z - torch.log(-torch.log(u)), dim=1).to(torch.int32)
    return out
