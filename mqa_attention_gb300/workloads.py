"""The benchmark workloads: shapes, RoPE base and pass set of each, and the
FLOP / byte counts the throughput and roofline figures are computed from.

Shapes come from the model families the source pages train: Llama-3-8B
attention (32 query heads over 8 KV heads, head_dim 128, rope_theta 500000;
"深度学习系统设计llama3-from-scratch：并行计算架构", §模型配置参数解析), PaLM-style
multi-query attention (8 heads of 64 over one K/V head; "ColossalAI 中的 PaLM
教学实现…", §2.5, §2.6), a SmolLM-1.7B micro-batch (batch 4, sequence 1024;
"Picotron模型实现解析Llama架构与Flash Attention集成", §配置与使用指南) and a 32K
sequence ("Megatron-DeepSpeed序列并行技术深度解析支持32K长序列训练的完整方案"), run
here on one GPU without sequence parallelism.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

__all__ = ["Workload", "WORKLOADS", "by_index", "by_name"]


@dataclass(frozen=True)
class Workload:
    index: int  # also the seed base: seed = 1000 * index + tensor id
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    theta: float
    backward: bool
    causal: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def pairs(self) -> int:
        """(query, key) score pairs computed per pass: causal counts j <= i."""
        per_head = self.S * (self.S + 1) // 2 if self.causal else self.S * self.S
        return self.B * self.Hq * per_head

    @property
    def fwd_flops(self) -> int:
        return 4 * self.D * self.pairs  # Q.Kᵀ and P.V, 2 flops per multiply-add

    @property
    def bwd_flops(self) -> int:
        return 10 * self.D * self.pairs  # recomputed Q.Kᵀ, dO.Vᵀ, Pᵀ.dO, dSᵀ.Q, dS.K

    @property
    def flops(self) -> int:
        return self.fwd_flops + (self.bwd_flops if self.backward else 0)

    def shapes(self):
        q = (self.B, self.Hq, self.S, self.D)
        kv = (self.B, self.Hkv, self.S, self.D)
        return {"q": q, "k": kv, "v": kv, "dout": q}

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} Hq={self.Hq} Hkv={self.Hkv} S={self.S} D={self.D} "
                f"theta={self.theta:g} {'fwd+bwd' if self.backward else 'fwd'}"
                f"{' causal' if self.causal else ''}")


WORKLOADS = (
    Workload(1, "tiny_mqa_fwd", 1, 4, 1, 128, 64, 10000.0, backward=False),
    Workload(2, "llama3_8b_gqa_s4096", 1, 32, 8, 4096, 128, 500000.0, backward=True),
    Workload(3, "palm_mqa_s2048", 8, 8, 1, 2048, 64, 10000.0, backward=True),
    Workload(4, "smollm_mha_s1024", 4, 32, 32, 1024, 64, 10000.0, backward=True),
    Workload(5, "long_gqa_s32768", 1, 32, 8, 32768, 128, 500000.0, backward=True),
)


def by_index(i: int) -> Workload:
    return next(w for w in WORKLOADS if w.index == i)


def by_name(name: str) -> Workload:
    return next(w for w in WORKLOADS if w.name == name)
