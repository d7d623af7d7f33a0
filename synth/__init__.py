"""Seeded synthetic inputs for the NVFP4 MoE layer (shared by the GPU path and the oracle).

This module is data plumbing only: it draws the layer's *inputs* (BF16 activations, FP32 router
logits, BF16 expert weights) and holds none of the layer's arithmetic (no quantisation, routing,
GEMM or combine).  Both sides of every parity test receive the identical bytes it produces.

Generator (counter based, so any slice of any tensor can be drawn on its own, on CPU or GPU):
  * SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number generators", OOPSLA
    2014): the element counter c of a stream with key K yields mix64(K + (c + 1) * golden).
  * key = mix64(seed << 32 | config_id << 16 | tensor_id).
  * uniform u = ((bits >> 11) + 0.5) * 2^-53, strictly inside (0, 1).
  * normal via Box-Muller in float64: element 2m is r*cos(theta), 2m+1 is r*sin(theta),
    with r = sqrt(-2 ln u(2m)) and theta = 2*pi*u(2m+1); then * sigma, cast to float32, and
    (for BF16 tensors) rounded to BF16 by PyTorch's round-to-nearest-even cast.

The workloads follow the five configurations of the fused NVFP4 MoE problem statement (tiny,
decode, prefill, large with a shared expert, Zipf-skewed routing).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_MASK64 = (1 << 64) - 1


def _i64(v: int) -> int:
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


_GOLDEN = _i64(0x9E3779B97F4A7C15)
_C1 = _i64(0xBF58476D1CE4E5B9)
_C2 = _i64(0x94D049BB133111EB)


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def mix64(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 finaliser on int64 tensors (two's-complement wrap-around arithmetic)."""
    z = (z ^ _srl(z, 30)) * _C1
    z = (z ^ _srl(z, 27)) * _C2
    return z ^ _srl(z, 31)


def mix64_int(z: int) -> int:
    """Python-int SplitMix64 finaliser, the reference the tensor version is tested against."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, config_id: int, tensor_id: int) -> int:
    base = ((seed & 0xFFFFFFFF) << 32) | ((config_id & 0xFFFF) << 16) | (tensor_id & 0xFFFF)
    return _i64(mix64_int(base))


def raw_bits(key: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """64-bit draws for counters [start, start + count) as int64 bit patterns."""
    c = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    return mix64(c * _GOLDEN + key)


def uniform(key: int, start: int, count: int, device="cpu") -> torch.Tensor:
    bits = _srl(raw_bits(key, start, count, device), 11)
    return (bits.to(torch.float64) + 0.5) * (2.0 ** -53)


def normal(key: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """float64 N(0,1) draws for element indices [start, start + count)."""
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    pair = idx >> 1
    c1 = pair * 2 + 1
    u1 = (_srl(mix64(c1 * _GOLDEN + key), 11).to(torch.float64) + 0.5) * (2.0 ** -53)
    u2 = (_srl(mix64((c1 + 1) * _GOLDEN + key), 11).to(torch.float64) + 0.5) * (2.0 ** -53)
    r = torch.sqrt(-2.0 * torch.log(u1))
    th = (2.0 * math.pi) * u2
    return torch.where((idx & 1) == 0, r * torch.cos(th), r * torch.sin(th))


# tensor ids inside one configuration's stream family
T_X, T_LOGITS, T_GATE, T_UP, T_DOWN, T_SGATE, T_SUP, T_SDOWN, T_ZIPF_RANK, T_SHARE_POOL = range(10)


@dataclass(frozen=True)
class MoeConfig:
    """One synthetic MoE workload (shapes, value distributions, routing structure)."""
    config_id: int
    name: str
    tokens: tuple           # token counts this configuration is run at
    hidden: int
    experts: int
    top_k: int
    inter: int
    w_sigma: float = 0.02
    shared_inter: int = 0   # 0: no shared expert
    zipf_s: float = 0.0     # 0: iid N(0,1) logits ("uniform routing")
    zipf_beta: float = 0.0  # logit bias scale for the Zipf popularity
    seed: int = 0
    description: str = field(default="", compare=False)

    @property
    def has_shared(self) -> int:
        return 1 if self.shared_inter else 0


# Zipf-skewed routing: logits = N(0,1) + beta * ln p_e with p_e proportional to rank_e^-1.2.
# beta was chosen by tests/golden/calibrate_zipf_beta.py (which routes with the oracle) so that
# the most popular expert receives about 4000 of the 16384*4 assignments; observed loads with
# seed 0 run from 532 to 4002 tokens per expert.
ZIPF_BETA = 0.2373

CONFIGS = {
    "tiny": MoeConfig(0, "tiny", (16,), 256, 8, 2, 512, 0.02,
                      description="T=16 H=256 E=8 top-2 I=512 SwiGLU"),
    "decode": MoeConfig(1, "decode", (1, 8, 32, 64), 2048, 128, 8, 768, 0.02,
                        description="decode: T in {1,8,32,64}, H=2048, E=128, top-8, I=768"),
    "prefill": MoeConfig(2, "prefill", (8192,), 2048, 256, 8, 512, 0.02,
                         description="prefill: T=8192, H=2048, E=256, top-8, I=512"),
    "large": MoeConfig(3, "large", (4096,), 7168, 256, 8, 2048, 0.015, shared_inter=2048,
                       description="large: T=4096, H=7168, E=256 (+1 shared), top-8, I=2048"),
    "skewed": MoeConfig(4, "skewed", (16384,), 4096, 64, 4, 1536, 0.02, zipf_s=1.2,
                        zipf_beta=ZIPF_BETA,
                        description="Zipf(1.2)-skewed routing: T=16384, H=4096, E=64, top-4, I=1536"),
}


def _key(cfg: MoeConfig, tensor_id: int) -> int:
    return stream_key(cfg.seed, cfg.config_id, tensor_id)


def gen_x(cfg: MoeConfig, T: int, device="cpu", row0: int = 0) -> torch.Tensor:
    """Activations x [T, H] BF16 ~ N(0,1); rows row0..row0+T-1 of the configuration's stream."""
    n = normal(_key(cfg, T_X), row0 * cfg.hidden, T * cfg.hidden, device)
    return n.to(torch.float32).to(torch.bfloat16).reshape(T, cfg.hidden)


def zipf_bias(cfg: MoeConfig, device="cpu") -> torch.Tensor:
    """Per-expert logit bias beta * ln p_e (float64), p_e ~ rank_e^-s over a seeded rank order."""
    u = uniform(_key(cfg, T_ZIPF_RANK), 0, cfg.experts, "cpu")
    order = torch.argsort(u)                       # expert order[i] gets rank i+1
    rank = torch.empty(cfg.experts, dtype=torch.float64)
    rank[order] = torch.arange(1, cfg.experts + 1, dtype=torch.float64)
    logp = -cfg.zipf_s * torch.log(rank)
    logp = logp - torch.logsumexp(logp, 0)
    return (cfg.zipf_beta * logp).to(device)


def gen_logits(cfg: MoeConfig, T: int, device="cpu", row0: int = 0, beta=None) -> torch.Tensor:
    """Router logits [T, E] FP32: N(0,1), plus the Zipf bias for the skewed configuration."""
    n = normal(_key(cfg, T_LOGITS), row0 * cfg.experts, T * cfg.experts, device)
    n = n.reshape(T, cfg.experts)
    if cfg.zipf_s:
        b = zipf_bias(cfg, device) if beta is None else (
            zipf_bias(MoeConfig(**{**cfg.__dict__, "zipf_beta": beta}), device))
        n = n + b[None, :]
    return n.to(torch.float32)


def sharing_unique_experts(T: int, k: int, share: int, E: int) -> int:
    """Distinct experts of a T-token batch at `share` percent expert sharing: the T*k
    assignments reuse share% of them across the batch, never below the k experts of one token
    (share 100 is that floor)."""
    return min(E, max(k, round(T * k * (100 - share) / 100)))


def sharing_routing(cfg: MoeConfig, T: int, share: int) -> torch.Tensor:
    """Expert ids [T, k] of the expert-sharing decode workload shared_<share>: a pool of
    U = sharing_unique_experts(...) experts drawn by a seeded permutation, token t's slot j taking
    pool[(t*k + j) mod U] - every pool expert used, no expert twice within one token."""
    k, E = cfg.top_k, cfg.experts
    U = sharing_unique_experts(T, k, share, E)
    u = uniform(_key(cfg, T_SHARE_POOL), share * E, E, "cpu")
    pool = torch.argsort(u)[:U]
    idx = (torch.arange(T)[:, None] * k + torch.arange(k)[None, :]) % U
    return pool[idx]


def gen_sharing_logits(cfg: MoeConfig, T: int, share: int, device="cpu") -> torch.Tensor:
    """Router logits [T, E] that route the batch as sharing_routing(cfg, T, share): the N(0,1)
    logits with each token's planted experts raised to 8 - j/4 (slot j), far above the rest."""
    lg = gen_logits(cfg, T, "cpu")
    ids = sharing_routing(cfg, T, share)
    planted = 8.0 - 0.25 * torch.arange(cfg.top_k, dtype=torch.float32)
    lg.scatter_(1, ids, planted.expand(T, -1).contiguous())
    return lg.to(device)


def gen_expert(cfg: MoeConfig, e: int, device="cpu"):
    """BF16 weights of routed expert e: gate [I,H], up [I,H], down [H,I] ~ N(0, w_sigma)."""
    n_gu = cfg.inter * cfg.hidden
    out = []
    for tid, shape in ((T_GATE, (cfg.inter, cfg.hidden)), (T_UP, (cfg.inter, cfg.hidden)),
                       (T_DOWN, (cfg.hidden, cfg.inter))):
        v = normal(_key(cfg, tid), e * n_gu, n_gu, device) * cfg.w_sigma
        out.append(v.to(torch.float32).to(torch.bfloat16).reshape(shape))
    return tuple(out)


def gen_shared(cfg: MoeConfig, device="cpu"):
    """BF16 weights of the always-on shared expert, or None."""
    if not cfg.shared_inter:
        return None
    n = cfg.shared_inter * cfg.hidden
    out = []
    for tid, shape in ((T_SGATE, (cfg.shared_inter, cfg.hidden)), (T_SUP, (cfg.shared_inter, cfg.hidden)),
                       (T_SDOWN, (cfg.hidden, cfg.shared_inter))):
        v = normal(_key(cfg, tid), 0, n, device) * cfg.w_sigma
        out.append(v.to(torch.float32).to(torch.bfloat16).reshape(shape))
    return tuple(out)


def gen_all_experts(cfg: MoeConfig, device="cpu", chunk: int = 16):
    """All routed experts stacked: gate [E,I,H], up [E,I,H], down [E,H,I] (BF16)."""
    E, I, H = cfg.experts, cfg.inter, cfg.hidden
    g = torch.empty(E, I, H, dtype=torch.bfloat16, device=device)
    u = torch.empty_like(g)
    d = torch.empty(E, H, I, dtype=torch.bfloat16, device=device)
    n_gu = I * H
    for tid, dst in ((T_GATE, g), (T_UP, u), (T_DOWN, d)):
        for e0 in range(0, E, chunk):
            e1 = min(E, e0 + chunk)
            v = normal(_key(cfg, tid), e0 * n_gu, (e1 - e0) * n_gu, device) * cfg.w_sigma
            dst[e0:e1] = v.to(torch.float32).to(torch.bfloat16).reshape(dst[e0:e1].shape)
            del v
    return g, u, d


def custom_config(name: str, T: int, H: int, E: int, k: int, I: int, config_id: int = 100,
                  shared_inter: int = 0, w_sigma: float = 0.02, seed: int = 0) -> MoeConfig:
    """A small ad-hoc workload (edge cases: ragged experts, k=1, k=E, shared expert ...)."""
    return MoeConfig(config_id, name, (T,), H, E, k, I, w_sigma, shared_inter=shared_inter, seed=seed)
