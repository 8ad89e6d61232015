"""Named synthetic workloads for the CRISP sparse-prefill path.

Each workload is one attention layer of causal prefill with the model shapes the CRISP
analysis page ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with
Structural-Mass-Motivated Routing", paper.rainbus.top, section "Reproduction
assessment") evaluates on: Llama-3.1-8B (32 query heads, 8 KV heads, d=128) and
Qwen2.5-7B (28 query heads, 4 KV heads, d=128), at the lengths of its latency table
(128k and 512k tokens) plus a tiny 4k case and a 32k case.

The real-model activations of the page's benchmarks are not available; the planted
generator in ``workloads.planted`` stands in for them (recipe in its module docstring).
The method's hyper-parameters are the page's defaults (section "Method step details"):
tau_proxy=0.2, gamma=0.95, alpha in {1.0, 1.25}, B=b=128, w_sink=w_local=128,
k_min=1024 tokens.

This module holds no arithmetic of the method; it only names shapes and seeds.
"""
from dataclasses import dataclass, field, replace
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    n: int                      # tokens
    hq: int                     # query heads
    hkv: int                    # key/value heads
    d: int = 128
    batch: int = 1
    seed: int = 0
    sink_scale: float = 4.0     # u-scale s: sink logit gain is s*s
    needles: Tuple = ("fixed", 6)   # ("fixed", k) or ("uniform", lo, hi) per VS head
    pe_heads: Tuple = ()        # explicit list of diffuse (PE-planted) query heads
    # method parameters
    B: int = 128
    b: int = 128
    w_sink: int = 128
    w_local: int = 128
    k_min_tokens: int = 1024
    tau_proxy: float = 0.2
    alpha: float = 1.0
    gamma: float = 0.95
    vs_floor: str = "mean"      # "mean" (the page's rule) or "median" (variant)
    vs_rule: str = "floor"      # "floor" (alpha * mu) or "gamma" (cumulative coverage variant)

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def n_blocks(self) -> int:
        return self.n // self.B

    def with_params(self, **kw) -> "Workload":
        return replace(self, **kw)


def _one_pe_per_group(hq: int, hkv: int) -> Tuple:
    g = hq // hkv
    return tuple(grp * g + (g - 1) for grp in range(hkv))


WORKLOADS = {
    # 2 heads, no GQA: head 0 VS-planted, head 1 diffuse.
    "tiny_n4k": Workload("tiny_n4k", n=4096, hq=2, hkv=2, seed=1000, sink_scale=4.0,
                         needles=("fixed", 6), pe_heads=(1,)),
    # Llama-3-8B layer shape, 25% diffuse heads (one per KV group).
    "llama8b_n32k": Workload("llama8b_n32k", n=32768, hq=32, hkv=8, seed=1001,
                             sink_scale=4.0, needles=("uniform", 2, 16),
                             pe_heads=_one_pe_per_group(32, 8)),
    "llama8b_n128k_a1": Workload("llama8b_n128k_a1", n=131072, hq=32, hkv=8, seed=1002,
                                 sink_scale=4.0, needles=("uniform", 2, 16),
                                 pe_heads=_one_pe_per_group(32, 8), alpha=1.0),
    "llama8b_n128k_a125": Workload("llama8b_n128k_a125", n=131072, hq=32, hkv=8, seed=1002,
                                   sink_scale=4.0, needles=("uniform", 2, 16),
                                   pe_heads=_one_pe_per_group(32, 8), alpha=1.25),
    # Qwen2-7B layer shape, stronger sink (s=5), one diffuse head per KV group (4/28).
    "qwen7b_n128k": Workload("qwen7b_n128k", n=131072, hq=28, hkv=4, seed=1003,
                             sink_scale=5.0, needles=("uniform", 2, 16),
                             pe_heads=_one_pe_per_group(28, 4)),
    # Llama-3-8B layer shape at the other lengths of the latency sweep (8k .. 256k).
    **{f"llama8b_n{n // 1024}k": Workload(f"llama8b_n{n // 1024}k", n=n, hq=32, hkv=8, seed=1100 + i,
                                          sink_scale=4.0, needles=("uniform", 2, 16),
                                          pe_heads=_one_pe_per_group(32, 8))
       for i, n in enumerate((8192, 16384, 65536, 262144))},
    # Llama-3-8B layer shape at 512k tokens, 16 needle blocks per VS head.
    "llama8b_n512k": Workload("llama8b_n512k", n=524288, hq=32, hkv=8, seed=1004,
                              sink_scale=4.0, needles=("fixed", 16),
                              pe_heads=_one_pe_per_group(32, 8)),
    # The first two KV groups of llama8b_n512k (the same heads, bit for bit: every head has
    # its own seed stream): the 512k layer's per-KV-head attention launches on a case that
    # holds ~3.5 GB on the device, for counter captures.
    "llama8b_n512k_kv2": Workload("llama8b_n512k_kv2", n=524288, hq=8, hkv=2, seed=1004,
                                  sink_scale=4.0, needles=("fixed", 16),
                                  pe_heads=_one_pe_per_group(8, 2)),
}


# The latency sweep over sequence length (Llama-3-8B layer shape): the page's latency
# table spans 64k-512k and its limitations section places the sparse/dense crossover
# between 8k and 64k.
SWEEP = ("llama8b_n8k", "llama8b_n16k", "llama8b_n32k", "llama8b_n64k", "llama8b_n128k_a1",
         "llama8b_n256k", "llama8b_n512k")


def get(name: str) -> Workload:
    return WORKLOADS[name]
