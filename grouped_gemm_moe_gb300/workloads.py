"""Seeded synthetic workloads for one MoE layer.

This module only draws inputs: shapes, seeds and value distributions. It holds
none of the layer's arithmetic (no routing, no sorting, no GEMM), so both the
CUDA path and the CPU oracle can be fed from it without sharing any code of the
method itself.

The five shapes follow the workloads the source pages train on:

* ``tiny``      a small layer the oracle finishes in milliseconds;
* ``qwen3``     Qwen3-30B-A3B-shaped layer (PithTrain PR "MoE parallel folding",
                validated-mesh table: qwen3-30b-a3b at seq 2048);
* ``dsv2lite``  DeepSeek-V2-Lite-shaped layer with two always-on shared experts
                (same table: deepseek-v2-lite at seq 4096; shared experts as in
                SpecForge PR "expert parallelism for MoE drafters", "What this adds");
* ``skew``      the Qwen3 shape with Zipf-biased logits, standing in for the
                real-routing load imbalance reported in the PithTrain PR review;
* ``drafter``   a DeepSeek-V4-Flash drafter-shaped layer at EP4, 16 of 64
                experts per rank (SpecForge PR, "What this adds", recipe bullet).

No dataset, tokenizer or trained weight is involved: N(0,1) router logits and
activations, N(0, 0.02) expert weights, all drawn from a CPU
``torch.Generator`` so that every consumer sees identical bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens in the layer's batch
    d: int            # hidden size
    E: int            # routed experts
    K: int            # experts per token (top-k)
    I: int            # routed expert intermediate size
    R: int            # simulated expert-parallel ranks
    shared_I: int = 0  # total intermediate size of the always-on shared experts (0 = none)
    backward: bool = True
    skew: bool = False
    seed: int = 0
    renorm: int = 1   # top-k weights renormalised over the K selected experts

    @property
    def TK(self) -> int:
        return self.T * self.K

    @property
    def El(self) -> int:
        return self.E // self.R


CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=256, d=128, E=8, K=2, I=256, R=2, backward=False),
    "qwen3": MoEConfig("qwen3", T=8192, d=2048, E=128, K=8, I=768, R=8),
    "dsv2lite": MoEConfig("dsv2lite", T=16384, d=2048, E=64, K=6, I=1408, R=8,
                          shared_I=2 * 1408),
    "skew": MoEConfig("skew", T=8192, d=2048, E=128, K=8, I=768, R=8, skew=True),
    "drafter": MoEConfig("drafter", T=32768, d=4096, E=64, K=8, I=2048, R=4),
}

# The configuration the throughput metric is quoted on: the largest workload
# that runs forward and backward on one GPU.
BENCH_CONFIG = "drafter"
# The other forward + backward workloads, reported beside it.
SIDE_CONFIGS = ("qwen3", "dsv2lite", "skew")


def zipf_bias(E: int) -> torch.Tensor:
    """Per-expert logit bias 1.5*ln(1/rank^1.2) with the Zipf rank of expert e
    taken as e+1 (identity ranking), i.e. -1.8*ln(e+1), in fp32."""
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    return (1.5 * torch.log(1.0 / ranks.pow(1.2))).to(torch.float32)


def make_inputs(cfg: MoEConfig, T: Optional[int] = None, seed: Optional[int] = None,
                with_backward: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Draw one layer's inputs on the CPU.

    Draw order (fixed, so that a prefix of draws never depends on later ones):
    logits [T,E] fp32 N(0,1) (+ Zipf bias for the skew workload); x [T,d] N(0,1)
    -> bf16; w_gate [E,d,I], w_up [E,d,I], w_down [E,I,d] N(0,0.02) -> bf16;
    shared w_gate/w_up [d,Is], w_down [Is,d] N(0,0.02) -> bf16 when present;
    dout [T,d] N(0,1) -> bf16 when the backward pass is wanted.

    ``T`` may override the token count (a bounded sample of the workload for
    timing the CPU oracle); the weights keep the workload's full shapes.
    """
    T = cfg.T if T is None else T
    seed = cfg.seed if seed is None else seed
    bwd = cfg.backward if with_backward is None else with_backward
    g = torch.Generator().manual_seed(seed)
    out: Dict[str, torch.Tensor] = {}
    logits = torch.randn(T, cfg.E, generator=g, dtype=torch.float32)
    if cfg.skew:
        logits = logits + zipf_bias(cfg.E)[None, :]
    out["logits"] = logits.contiguous()
    out["x"] = torch.randn(T, cfg.d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    out["w_gate"] = (torch.randn(cfg.E, cfg.d, cfg.I, generator=g) * 0.02).to(torch.bfloat16)
    out["w_up"] = (torch.randn(cfg.E, cfg.d, cfg.I, generator=g) * 0.02).to(torch.bfloat16)
    out["w_down"] = (torch.randn(cfg.E, cfg.I, cfg.d, generator=g) * 0.02).to(torch.bfloat16)
    if cfg.shared_I:
        out["ws_gate"] = (torch.randn(cfg.d, cfg.shared_I, generator=g) * 0.02).to(torch.bfloat16)
        out["ws_up"] = (torch.randn(cfg.d, cfg.shared_I, generator=g) * 0.02).to(torch.bfloat16)
        out["ws_down"] = (torch.randn(cfg.shared_I, cfg.d, generator=g) * 0.02).to(torch.bfloat16)
    if bwd:
        out["dout"] = torch.randn(T, cfg.d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def small_config(name: str = "small", T: int = 64, d: int = 128, E: int = 8, K: int = 2,
                 I: int = 128, R: int = 2, shared_I: int = 0, skew: bool = False,
                 seed: int = 0, renorm: int = 1) -> MoEConfig:
    """A freely-shaped configuration for tests."""
    return MoEConfig(name, T=T, d=d, E=E, K=K, I=I, R=R, shared_I=shared_I,
                     backward=True, skew=skew, seed=seed, renorm=renorm)


def to_f64(t: torch.Tensor):
    """Exact float64 numpy copy of a bf16/fp32 CPU tensor (bf16 -> f64 is exact)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def flops_per_assignment_fwd(cfg: MoEConfig) -> int:
    """Dense-contraction flops of the routed SwiGLU FFN per (token, expert)
    assignment: gate and up projections (2*d*I each) plus down (2*I*d)."""
    return 6 * cfg.d * cfg.I


def describe(cfg: MoEConfig) -> str:
    s = (f"T={cfg.T} d={cfg.d} E={cfg.E} K={cfg.K} I={cfg.I} R={cfg.R}")
    if cfg.shared_I:
        s += f" shared_I={cfg.shared_I}"
    if cfg.skew:
        s += " zipf-skew"
    return s


__all__ = ["MoEConfig", "CONFIGS", "BENCH_CONFIG", "SIDE_CONFIGS", "make_inputs", "small_config",
           "zipf_bias", "to_f64", "describe", "flops_per_assignment_fwd"]
