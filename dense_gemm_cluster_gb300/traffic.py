"""Analytic operand-traffic accounting (measurement side, host only).

"Hopper TMA Multicast 深度解析与实测", section 实机运行与 NCU 验证: the page
counts the bytes that land in every CTA's shared memory (delivered) against the
bytes fetched from L2 (issued). With unicast each CTA fetches its own copy; with
a multicast of cluster size c one fetch serves c CTAs, so the issued bytes drop
by the factor c (50% for c = 2). ``tma_scenario_bytes`` states that accounting;
``tests/golden/tma_multicast_h100.json`` pins it to the page's printed figures.

``l2_to_sm_operand_bytes`` applies the same accounting to the tiled GEMM: per
CTA tile and k-block, the A tile (128 rows) is fetched once per A-sharing group
of size gA, and the B tile (BN/G columns for the pair MMA with G = 2) once per
B-sharing group of size gB. ("Clusters, distributed shared memory & cluster
launch control", "Two CTAs, one MMA -- cta_group::2": B per FLOP halves;
"TMA multicast": N copies of a shared tile become one.)
"""
from __future__ import annotations

BLOCK_M = 128   # rows of C per CTA
BLOCK_K = 64    # K elements per pipeline stage (one 128-byte swizzle row of bf16)


def tma_scenario_bytes(ctas: int, cluster: int, iters: int, tile_bytes: int) -> dict:
    """Delivered and issued bytes of the page-1 TMA load microbenchmark.

    Every CTA receives ``tile_bytes`` per iteration. Unicast issues one fetch per
    CTA; multicast issues one fetch per cluster.
    """
    if ctas % cluster:
        raise ValueError("the grid must be a whole number of clusters")
    delivered = ctas * iters * tile_bytes
    return {
        "delivered": delivered,
        "issued_unicast": delivered,
        "issued_multicast": (ctas // cluster) * iters * tile_bytes,
    }


def _ceil(a: int, b: int) -> int:
    return -(-a // b)


def l2_to_sm_operand_bytes(M: int, N: int, K: int, *, batch: int = 1, cta_group: int = 1,
                           block_n: int = 256, group_a: int = 1, group_b: int = 1,
                           elem_bytes: int = 2) -> int:
    """Operand bytes the TMA engines fetch from L2 for one GEMM launch.

    ``block_n`` is the N extent of one MMA tile (the pair's tile for cta_group 2);
    ``group_a`` / ``group_b`` are the numbers of CTAs one A / B fetch serves.
    Partial tiles and the K tail are counted as full boxes, since a TMA load
    moves the whole box (zero-filled outside the tensor).
    """
    if cta_group not in (1, 2):
        raise ValueError("cta_group is 1 or 2")
    k_pad = _ceil(K, BLOCK_K) * BLOCK_K
    cta_tiles = _ceil(M, BLOCK_M * cta_group) * cta_group * _ceil(N, block_n) * batch
    per_cta = k_pad * elem_bytes * (BLOCK_M // group_a + (block_n // cta_group) // group_b)
    return cta_tiles * per_cta
