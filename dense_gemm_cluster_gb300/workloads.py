"""The synthetic workloads the library is measured and checked on.

Each entry names a GEMM (or the batched score form) with its sizes, input
distributions, layouts and the operand-sharing mode it runs in. Inputs come
from ``inputs`` with seed 0 (A / Q on stream 0, B / K on stream 1, C_in on
stream 2). Layouts the workload text leaves open are row-major.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    batch: int = 1
    dist: str = "normal"            # "normal" (N(0,1)) or "uniform" (U(-1,1))
    scale: float = 1.0              # multiplies A and B draws before rounding
    layout_a: str = "row"
    layout_b: str = "row"
    layout_c: str = "row"
    out: str = "bf16"
    alpha: float = 1.0
    beta: float = 0.0
    c_dist: str = "normal"
    options: dict = field(default_factory=dict)
    description: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K * self.batch

    def min_hbm_bytes(self) -> int:
        """Each input read once, C written once (and read once when beta != 0)."""
        esc = 4 if self.out == "f32" else 2
        b = (self.M * self.K + self.K * self.N) * 2 * self.batch + self.M * self.N * esc * self.batch
        if self.beta != 0.0:
            b += self.M * self.N * esc * self.batch
        return b


WORKLOADS = {
    "gemm256_f32_mcastB": Workload(
        "gemm256_f32_mcastB", 256, 256, 256, dist="normal", out="f32",
        options=dict(mode="mcast", mcast_b=1, cluster_m=2, cluster_n=1),
        description="GEMM 256^3, N(0,1), fp32 out, row-major, 2-CTA cluster multicasting B"),
    "gemm4096_bf16_cluster2x1": Workload(
        "gemm4096_bf16_cluster2x1", 4096, 4096, 4096, dist="uniform", layout_a="row", layout_b="col",
        options=dict(mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=1),
        description="GEMM 4096^3, U(-1,1), A row-major, B column-major, bf16 out, 2x1 cluster "
                    "multicasting A and B (A's multicast extent is 1)"),
    "gemm4096_bf16_cluster2x2": Workload(
        "gemm4096_bf16_cluster2x2", 4096, 4096, 4096, dist="uniform", layout_a="row", layout_b="col",
        options=dict(mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2),
        description="GEMM 4096^3 as above with a 2x2 cluster multicasting both A and B"),
    "gemm4096_bf16_pair2x1": Workload(
        "gemm4096_bf16_pair2x1", 4096, 4096, 4096, dist="uniform", layout_a="row", layout_b="col",
        options=dict(cta_group=2, cluster_m=2, cluster_n=1, block_n=256),
        description="GEMM 4096^3 as above on a 2x1 cluster running the cta_group::2 pair MMA: 256x256 "
                    "tiles, each CTA loading its 128 rows of A and half of every B tile"),
    "gemm4096_bf16_unicast": Workload(
        "gemm4096_bf16_unicast", 4096, 4096, 4096, dist="uniform", layout_a="row", layout_b="col",
        options=dict(mode="unicast", cluster_m=1, cluster_n=1, cta_group=1, block_n=256),
        description="GEMM 4096^3 as above with unicast loads and single-CTA 128x256 tiles (the baseline for "
                    "the 4096^3 sharing modes' L2->SM operand-byte comparison)"),
    "gemm8192_bf16_pair_mcastB4": Workload(
        "gemm8192_bf16_pair_mcastB4", 8192, 8192, 8192, dist="normal", scale=1.0 / math.sqrt(8192),
        out="bf16", beta=0.5,
        options=dict(mode="mcast", mcast_b=1, cluster_m=4, cluster_n=1, cta_group=2, block_n=256),
        description="GEMM 8192^3, N(0,1)/sqrt(K), bf16 out, beta=0.5 with bf16 C ~ N(0,1), "
                    "cta_group::2 256x256 tiles, 4-CTA cluster multicasting B"),
    "gemm8192_bf16_unicast": Workload(
        "gemm8192_bf16_unicast", 8192, 8192, 8192, dist="normal", scale=1.0 / math.sqrt(8192),
        out="bf16", beta=0.5,
        options=dict(mode="unicast", cluster_m=1, cluster_n=1, cta_group=1, block_n=256),
        description="the 8192^3 GEMM above with unicast loads and single-CTA 128x256 tiles (the baseline "
                    "for the L2->SM operand-byte comparison)"),
    "scores_8x16x4096x4096x128": Workload(
        "scores_8x16x4096x4096x128", 4096, 4096, 128, batch=128, dist="normal", layout_a="row",
        layout_b="col", out="f32",
        options=dict(mode="mcast", mcast_b=1, cluster_m=4, cluster_n=1),
        description="attention scores S = Q K^T, batch 8 x heads 16, seq 4096, head dim 128, "
                    "N(0,1) bf16 Q/K, fp32 S, each K tile multicast across the 4 Q-tile CTAs of a cluster"),
    "skinny_16384x128x8192": Workload(
        "skinny_16384x128x8192", 16384, 128, 8192, dist="uniform",
        options=dict(mode="mcast", mcast_b=1, cluster_m=4, cluster_n=1, cta_group=2, block_n=128),
        description="skinny GEMM M=16384, N=128, K=8192, U(-1,1), bf16 out, cta_group::2 256x128 tiles, small B "
                    "multicast along M across the two pairs of a 4-CTA cluster"),
    "skinny_128x16384x8192": Workload(
        "skinny_128x16384x8192", 128, 16384, 8192, dist="uniform",
        options=dict(mode="mcast", mcast_a=1, cluster_m=1, cluster_n=2, block_n=128),
        description="skinny GEMM M=128, N=16384, K=8192, U(-1,1), bf16 out, small A multicast along N across "
                    "the 2 CTAs of a cluster"),
}

# The bench's default: the largest single-GPU GEMM, on the pair MMA with 4-CTA B multicast.
DEFAULT = "gemm8192_bf16_pair_mcastB4"

# The unicast workload that computes the same output with every CTA fetching its own
# tiles: the measured L2->SM operand bytes of a sharing mode are compared with it.
UNICAST_TWIN = {
    "gemm4096_bf16_cluster2x1": "gemm4096_bf16_unicast",
    "gemm4096_bf16_cluster2x2": "gemm4096_bf16_unicast",
    "gemm4096_bf16_pair2x1": "gemm4096_bf16_unicast",
    "gemm8192_bf16_pair_mcastB4": "gemm8192_bf16_unicast",
}


@dataclass(frozen=True)
class AttentionWorkload:
    """Fused attention forward O = softmax(scale Q K^T) V over batch x heads independent heads."""
    name: str
    batch: int                      # batch x heads
    sq: int
    sk: int
    d: int = 128
    cluster: int = 2                # CTAs sharing each K/V tile
    cta_group: int = 1              # 1: multicast of whole K/V tiles; 2: pair MMA over half tiles
    out: str = "bf16"
    dist: str = "normal"
    causal: bool = False            # query i attends keys 0..i only
    description: str = ""

    @property
    def pairs(self) -> int:
        """(query, key) pairs scored per head."""
        if not self.causal:
            return self.sq * self.sk
        full = max(0, self.sq - self.sk)                          # rows past the last key see every key
        n = min(self.sq, self.sk)
        return n * (n + 1) // 2 + full * self.sk

    @property
    def flops(self) -> int:
        return 4 * self.batch * self.pairs * self.d               # Q K^T and P V over the scored pairs

    def min_hbm_bytes(self) -> int:
        """Q, K, V read once; O and the row log-sum-exp written once."""
        esc = 4 if self.out == "f32" else 2
        return self.batch * (2 * (self.sq + 2 * self.sk) * self.d + esc * self.sq * self.d + 4 * self.sq)


ATTENTION_WORKLOADS = {
    "attention_fwd_8x16x4096x4096x128": AttentionWorkload(
        "attention_fwd_8x16x4096x4096x128", 128, 4096, 4096, cluster=2,
        description="fused attention forward O = softmax(Q K^T / sqrt(128)) V with the row log-sum-exp, "
                    "batch 8 x heads 16, seq 4096, head dim 128, N(0,1) bf16 Q/K/V, bf16 O, each K/V tile "
                    "multicast across the 2 query-block CTAs of a cluster"),
    "attention_fwd_causal_8x16x4096x4096x128": AttentionWorkload(
        "attention_fwd_causal_8x16x4096x4096x128", 128, 4096, 4096, cluster=1, causal=True,
        description="the attention forward above with the causal mask (query i attends keys 0..i): half the "
                    "score pairs, FLOPs counted over the pairs scored; one CTA per cluster (the query blocks "
                    "of a cluster would need different numbers of key tiles)"),
}
