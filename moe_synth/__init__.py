"""Seeded synthetic inputs for the fused MoE layer forward.

This module is shared by the oracle side (tests) and the CUDA side (tests,
bench).  It holds no arithmetic of the method: it only draws random tensors.

Recipe (the workloads' shapes and distributions):
  x        ~ N(0, 1)          [T, H]
  w_router ~ N(0, 1/H)        [H, E]
  W1       ~ N(0, 1/H)        [E, H, F]    (gated experts: [E, H, 2F] = [gate | up])
  W2       ~ N(0, 1/F)        [E, F, H]
  bias     optional fp32 [E] (the skewed workload puts +4.0 on expert 0)
Every tensor, and every expert's slice of W1 and W2, has its own stream:
numpy's PCG64 bit generator seeded by SeedSequence((seed, tensor id,
expert)).  Normal values come from the Box-Muller transform in float64 --
pairs (u1, u2) of uniform doubles give sqrt(-2 ln(1 - u1)) cos(2 pi u2) and
then the matching sines -- scaled by the std, rounded to fp32 and then to
bf16 (round-to-nearest-even each time).  The bits are the same on any
machine: the stream is integer arithmetic, and a one-ulp difference between
two platforms' float64 log or cos changes a bf16 value with probability
about 2^-44 per draw (a vectorised fp32 generator, as torch's randn, gives
different bits on different CPU architectures).  One expert's weights can
be regenerated alone and the slices are drawn in parallel threads; the bits
do not depend on the thread count.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np
import torch

_TENSOR_ID = {"x": 1, "w_router": 2, "w1": 3, "w2": 4}


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    F: int  # 0 for router-only workloads
    E: int
    k: int
    seed: int = 0
    capacity_factor: float | None = None
    bias0: float | None = None  # router bias on expert 0 (others 0)
    act: str = "gelu"  # "gelu": W1 [E,H,F]; "swiglu": W1 [E,H,2F] = [gate | up]
    notes: str = ""

    @property
    def has_ffn(self) -> bool:
        return self.F > 0

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# The five seeded workloads.
TINY = MoEConfig("tiny", T=64, H=128, F=256, E=8, k=2, seed=0)
PREFILL = MoEConfig("prefill", T=4096, H=4096, F=14336, E=8, k=2, seed=0)
ROUTER = {kk: MoEConfig(f"router_k{kk}", T=2048, H=4096, F=0, E=128, k=kk, seed=0)
          for kk in (1, 2, 4, 8)}
SKEWED = MoEConfig("skewed", T=8192, H=2048, F=1408, E=64, k=4, seed=0, bias0=4.0)
SKEWED_CF = SKEWED.with_(name="skewed_cf1.2", capacity_factor=1.2)
DECODE = MoEConfig("decode", T=32, H=4096, F=14336, E=8, k=2, seed=7)

# Gated (SwiGLU) experts at the same shapes: 3 matrices per expert, so the
# decode workload streams 2.82 GB of weights.
PREFILL_SWIGLU = PREFILL.with_(name="prefill_swiglu", act="swiglu")
# One expert per token (top-1 routing, as in Switch-style layers): the
# combine is a single scaled row, written by the second GEMM itself.
PREFILL_K1 = PREFILL.with_(name="prefill_k1", k=1)
DECODE_SWIGLU = DECODE.with_(name="decode_swiglu", act="swiglu")

ALL = {c.name: c for c in [TINY, PREFILL, *ROUTER.values(), SKEWED, SKEWED_CF, DECODE,
                           PREFILL_SWIGLU, DECODE_SWIGLU, PREFILL_K1]}


_CHUNK = 1 << 22  # draws per Box-Muller block (bounds the float64 temporaries)


def _stream(seed: int, tensor: str, part: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence((seed, _TENSOR_ID[tensor],
                                                                        part))))


def _box_muller(rng: np.random.Generator, n: int) -> np.ndarray:
    """n standard normal float64 values: for m = ceil(n / 2) uniform pairs
    (u1, u2), r = sqrt(-2 ln(1 - u1)) (1 - u1 in (0, 1]), then r cos(2 pi u2)
    for the m pairs followed by r sin(2 pi u2), truncated to n."""
    m = (n + 1) // 2
    u1 = rng.random(m)
    u2 = rng.random(m)
    np.subtract(1.0, u1, out=u1)
    np.log(u1, out=u1)
    u1 *= -2.0
    np.sqrt(u1, out=u1)
    u2 *= 2.0 * math.pi
    z = np.empty(2 * m)
    np.cos(u2, out=z[:m])
    np.sin(u2, out=z[m:])
    z[:m] *= u1
    z[m:] *= u1
    return z[:n]


def _normal_bf16(shape, std: float, rng: np.random.Generator) -> torch.Tensor:
    n = math.prod(shape)
    out = np.empty(n, dtype=np.float32)
    for i in range(0, n, _CHUNK):
        k = min(_CHUNK, n - i)
        z = _box_muller(rng, k)
        if std != 1.0:
            z *= std
        out[i:i + k] = z  # float64 -> fp32, round to nearest even
    return torch.from_numpy(out).reshape(shape).to(torch.bfloat16)


def make_x(cfg: MoEConfig) -> torch.Tensor:
    return _normal_bf16((cfg.T, cfg.H), 1.0, _stream(cfg.seed, "x"))


def make_w_router(cfg: MoEConfig) -> torch.Tensor:
    return _normal_bf16((cfg.H, cfg.E), 1.0 / math.sqrt(cfg.H), _stream(cfg.seed, "w_router"))


def make_bias(cfg: MoEConfig) -> torch.Tensor | None:
    if cfg.bias0 is None:
        return None
    b = torch.zeros(cfg.E, dtype=torch.float32)
    b[0] = cfg.bias0
    return b


def w1_cols(cfg: MoEConfig) -> int:
    return 2 * cfg.F if cfg.act == "swiglu" else cfg.F


def make_w1_expert(cfg: MoEConfig, e: int) -> torch.Tensor:
    return _normal_bf16((cfg.H, w1_cols(cfg)), 1.0 / math.sqrt(cfg.H), _stream(cfg.seed, "w1", e))


def make_w2_expert(cfg: MoEConfig, e: int) -> torch.Tensor:
    return _normal_bf16((cfg.F, cfg.H), 1.0 / math.sqrt(cfg.F), _stream(cfg.seed, "w2", e))


def _stack_experts(cfg: MoEConfig, fn, shape, threads: int) -> torch.Tensor:
    out = torch.empty((cfg.E, *shape), dtype=torch.bfloat16)

    def one(e):
        out[e].copy_(fn(cfg, e))

    if threads <= 1 or cfg.E == 1:
        for e in range(cfg.E):
            one(e)
    else:
        with ThreadPoolExecutor(max_workers=min(threads, cfg.E)) as ex:
            list(ex.map(one, range(cfg.E)))
    return out


def make_inputs(cfg: MoEConfig, with_ffn: bool = True, threads: int = 8) -> dict:
    """All inputs of ``cfg`` as CPU tensors (bf16, bias fp32 or None)."""
    d = dict(x=make_x(cfg), w_router=make_w_router(cfg), bias=make_bias(cfg))
    if with_ffn and cfg.has_ffn:
        d["w1"] = _stack_experts(cfg, make_w1_expert, (cfg.H, w1_cols(cfg)), threads)
        d["w2"] = _stack_experts(cfg, make_w2_expert, (cfg.F, cfg.H), threads)
    return d


def sampled_rows(T: int, stride: int) -> list[int]:
    """Every ``stride``-th token (0, stride, 2*stride, ...)."""
    return list(range(0, T, stride))
