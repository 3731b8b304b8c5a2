"""Seeded synthetic inputs for the fused MoE layer forward.

This module is shared by the oracle side (tests) and the CUDA side (tests,
bench).  It holds no arithmetic of the method: it only draws random tensors.

Recipe (the workloads' shapes and distributions):
  x        ~ N(0, 1)          [T, H]
  w_router ~ N(0, 1/H)        [H, E]
  W1       ~ N(0, 1/H)        [E, H, F]    (gated experts: [E, H, 2F] = [gate | up])
  W2       ~ N(0, 1/F)        [E, F, H]
  bias     optional fp32 [E] (the skewed workload puts +4.0 on expert 0)
Each value is drawn as fp32 from torch's CPU generator and rounded to bf16
(round-to-nearest-even).  Every tensor, and every expert's slice of W1 and
W2, has its own generator seeded from (seed, tensor id, expert), so one
expert's weights can be regenerated alone and all slices can be drawn in
parallel threads; the bits do not depend on the thread count or the device.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

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


def _gen(seed: int, tensor: str, part: int = 0) -> torch.Generator:
    s = ((seed * 1000003 + _TENSOR_ID[tensor]) * 1000003 + part) % (2**63 - 1)
    return torch.Generator().manual_seed(s)


def _normal_bf16(shape, std: float, gen: torch.Generator) -> torch.Tensor:
    a = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        a.mul_(std)
    return a.to(torch.bfloat16)


def make_x(cfg: MoEConfig) -> torch.Tensor:
    return _normal_bf16((cfg.T, cfg.H), 1.0, _gen(cfg.seed, "x"))


def make_w_router(cfg: MoEConfig) -> torch.Tensor:
    return _normal_bf16((cfg.H, cfg.E), 1.0 / math.sqrt(cfg.H), _gen(cfg.seed, "w_router"))


def make_bias(cfg: MoEConfig) -> torch.Tensor | None:
    if cfg.bias0 is None:
        return None
    b = torch.zeros(cfg.E, dtype=torch.float32)
    b[0] = cfg.bias0
    return b


def w1_cols(cfg: MoEConfig) -> int:
    return 2 * cfg.F if cfg.act == "swiglu" else cfg.F


def make_w1_expert(cfg: MoEConfig, e: int) -> torch.Tensor:
    return _normal_bf16((cfg.H, w1_cols(cfg)), 1.0 / math.sqrt(cfg.H), _gen(cfg.seed, "w1", e))


def make_w2_expert(cfg: MoEConfig, e: int) -> torch.Tensor:
    return _normal_bf16((cfg.F, cfg.H), 1.0 / math.sqrt(cfg.F), _gen(cfg.seed, "w2", e))


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
