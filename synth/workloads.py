"""The five synthetic MoE-layer workloads and their seeded input recipes.

Shapes follow the pages' regimes: the 384-expert / top-6 layer of "763B MoE in
two 96 GB cards" (section "Where the VRAM gap comes from": 40 layers x 384
routed experts, 4,608 of 15,360 in host memory), and the many-expert cached
decode of "Running a 24k-expert MoE on a single 32 GB card" (sections 2-3:
~70% of experts in an HBM cache, skewed popularity).

Everything here is an input: shapes, random draws, and which experts the
caller places in host memory.  No quantisation, routing or FFN arithmetic.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import (TAG_BIAS, TAG_DRIFT, TAG_NOISE, TAG_ROUTER, TAG_WEIGHT, TAG_X, key, normal_bf16,
               normal_f32, zipf_bias)
from .popularity import calibrated_rank_bias

SC_F32, SC_BF16, SC_F16 = 0, 1, 2
GATE, UP, DOWN = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    experts: int
    hidden: int
    inter: int
    top_k: int
    tokens: tuple
    bits: int
    group: int
    scale_dtype: int
    router: str                 # "plain": Wr ~ N(0, 0.05), no bias; "zipf": see router()
    zipf_s: float = 0.0
    host_total: int = 0         # static placement: experts in pinned host memory (whole stack)
    cache_frac: float = 0.0     # >0: LFU cache of floor(frac * L * E) HBM slots, all experts in host
    steps: int = 1
    drift: float = 0.0          # per-step random walk of the router bias (cached decode)
    w_sigma: float = 0.02
    seed: int = 0
    desc: str = field(default="", compare=False)

    @property
    def total_experts(self) -> int:
        return self.layers * self.experts

    @property
    def cache_slots(self) -> int:
        return int(math.floor(self.cache_frac * self.total_experts)) if self.cache_frac > 0 else 0

    def matrix_shape(self, m: int) -> tuple[int, int]:
        return (self.inter, self.hidden) if m in (GATE, UP) else (self.hidden, self.inter)

    def codes_bytes(self, m: int) -> int:
        r, c = self.matrix_shape(m)
        return r * c * self.bits // 8

    def scales_bytes(self, m: int) -> int:
        r, c = self.matrix_shape(m)
        return r * (c // self.group) * (4 if self.scale_dtype == SC_F32 else 2)

    @property
    def expert_bytes(self) -> int:
        """Algorithmic bytes of one expert: codes + scales of gate, up, down."""
        return sum(self.codes_bytes(m) + self.scales_bytes(m) for m in range(3))

    @property
    def router_bytes(self) -> int:
        return self.experts * self.hidden * 2

    def host_count(self, layer: int) -> int:
        """Experts of `layer` in host memory: the stack total spread as evenly as
        integers allow, floor((l+1) N / L) - floor(l N / L)."""
        n, L = self.host_total, self.layers
        return (layer + 1) * n // L - layer * n // L


WORKLOADS = {
    "tiny": Workload(
        "tiny", 1, 16, 256, 128, 2, (8,), 4, 32, SC_F32, "plain",
        desc="tiny layer: H=256, I=128, E=16, top-2, T=8, int4 G32 fp32 scales, all HBM"),
    "decode": Workload(
        "decode", 1, 384, 4096, 1024, 6, (1, 4, 6), 3, 128, SC_BF16, "zipf", 1.0, host_total=115,
        desc="decode layer: H=4096, I=1024, E=384, top-6, T in {1,4,6}, int3 G128 bf16 scales, "
             "Zipf(1.0), 115 least-popular experts in pinned host memory (UVA), 269 in HBM"),
    "stack40": Workload(
        "stack40", 40, 384, 4096, 1024, 6, (1, 4), 3, 128, SC_BF16, "zipf", 1.0, host_total=4608,
        desc="40-layer stack of the decode layer: 15,360 experts, 4,608 in host memory, "
             "T in {1,4}, each layer fed bf16(previous output + N(0,1) noise)"),
    "prefill": Workload(
        "prefill", 1, 384, 4096, 1024, 6, (8192,), 4, 128, SC_BF16, "zipf", 1.0,
        desc="prefill layer: T=8192, H=4096, I=1024, E=384, top-6, int4 G128 bf16 scales, "
             "Zipf(1.0), all experts in HBM"),
    "cached": Workload(
        "cached", 48, 512, 2048, 512, 8, (1,), 2, 64, SC_F16, "zipf", 1.2, cache_frac=0.7,
        steps=2048, drift=0.01,
        desc="cached decode: 48 layers x 512 experts, H=2048, I=512, top-8, int2 G64 fp16 scales, "
             "Zipf(1.2) with per-step bias drift, all experts pinned in host memory, LFU cache "
             "of 17,203 HBM slots, T=1, 2048 steps"),
}


def expert_master(wl: Workload, layer: int, expert: int, m: int) -> np.ndarray:
    """fp32 master weights of one matrix, ~N(0, w_sigma), row-major [rows][cols]."""
    r, c = wl.matrix_shape(m)
    return normal_f32(key(wl.seed, TAG_WEIGHT, layer, expert, m), r * c, wl.w_sigma).reshape(r, c)


def router_noise_sd() -> float:
    """Standard deviation of the noise term x . Wr[e] of the "zipf" router for
    x ~ N(0, 1): that of a standard Gumbel variable, pi / sqrt(6)."""
    return math.pi / math.sqrt(6.0)


def router(wl: Workload, layer: int):
    """(wr bf16 bits [E][H], bias fp32 [E] or None, popularity rank [E] or None).

    "plain": Wr ~ N(0, 0.05) rounded to bf16, no bias.
    "zipf":  Wr ~ N(0, sd / sqrt H) with sd = pi / sqrt 6, so that x . Wr[e] for
             x ~ N(0,1) is close to independent N(0, sd^2) noise per expert;
             expert e gets a seeded popularity rank and the bias of that rank
             from synth.popularity.calibrated_rank_bias, for which top-k of
             (bias + noise) includes every rank with its Plackett-Luce Zipf(s)
             probability (k draws without replacement, p_r proportional to
             (r+1)^-s)."""
    E, H = wl.experts, wl.hidden
    if wl.router == "plain":
        wr = normal_bf16(key(wl.seed, TAG_ROUTER, layer), E * H, 0.05).reshape(E, H)
        return wr, None, None
    sd = router_noise_sd()
    wr = normal_bf16(key(wl.seed, TAG_ROUTER, layer), E * H, sd / math.sqrt(H)).reshape(E, H)
    _, rank = zipf_bias(key(wl.seed, TAG_BIAS, layer), E, wl.zipf_s)
    by_rank, _ = calibrated_rank_bias(E, wl.top_k, float(wl.zipf_s), sd)
    bias = np.asarray(by_rank, dtype=np.float32)[rank]
    return wr, bias, rank


def host_experts(wl: Workload, layer: int, rank: np.ndarray | None) -> np.ndarray:
    """Experts of `layer` the caller places in host memory: the least popular ones."""
    n = wl.host_count(layer) if wl.host_total else 0
    if n == 0 or rank is None:
        return np.zeros(0, dtype=np.int32)
    return np.sort(np.nonzero(rank >= wl.experts - n)[0]).astype(np.int32)


def tokens(wl: Workload, step: int, layer: int, T: int) -> np.ndarray:
    """Layer input x ~ N(0,1) as bf16 bits [T][H] (a fresh draw per step)."""
    return normal_bf16(key(wl.seed, TAG_X, step, layer), T * wl.hidden, 1.0).reshape(T, wl.hidden)


def residual_noise(wl: Workload, step: int, layer: int, T: int) -> np.ndarray:
    """N(0,1) fp32 [T][H] added to a layer's output to form the next layer's input."""
    return normal_f32(key(wl.seed, TAG_NOISE, step, layer), T * wl.hidden, 1.0).reshape(T, wl.hidden)


def bias_drift(wl: Workload, step: int, layer: int) -> np.ndarray:
    """Per-step random-walk increment of the router bias: drift * N(0,1) [E]."""
    return normal_f32(key(wl.seed, TAG_DRIFT, step, layer), wl.experts, 1.0) * np.float32(wl.drift)
