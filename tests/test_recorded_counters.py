"""The ncu counters recorded under profiles/ against the analytic byte accounting.

`profiles/ncu_traffic.json` holds, per workload, the DRAM bytes and the L2 -> SM
operand sectors of one launch as ncu measured them on GB300. These tests hold
those measurements to the design's claims: the pair MMA plus 4-CTA multicast of B
cuts the measured L2 -> SM operand bytes of the 8192^3 GEMM at least 1.8x against
unicast tiles, and the measured bytes follow the planner's analytic accounting.
(No GPU needed: the numbers are read from the committed record.)
"""
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def records():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def analytic():
    from dense_gemm_cluster_gb300 import build
    build.build()
    from dense_gemm_cluster_gb300 import gemm
    from dense_gemm_cluster_gb300.workloads import WORKLOADS
    out = {}
    for name, w in WORKLOADS.items():
        opts = gemm.make_options(layout_a=w.layout_a, layout_b=w.layout_b, layout_c=w.layout_c, out_type=w.out,
                                 **w.options)
        s, p = gemm.gemm_plan(opts, w.M, w.N, w.K, w.batch, 152)
        assert s == 0
        out[name] = (w, p)
    return out


def test_multicast_and_pair_cut_measured_l2_to_sm_bytes(records, analytic):
    uni = records["gemm8192_bf16_unicast"]["lts_bytes"]
    shared = records["gemm8192_bf16_pair_mcastB4"]["lts_bytes"]
    measured = uni / shared
    expected = (analytic["gemm8192_bf16_unicast"][1].l2_to_sm_operand_bytes /
                analytic["gemm8192_bf16_pair_mcastB4"][1].l2_to_sm_operand_bytes)
    assert expected == pytest.approx(2.0)
    assert measured >= 1.8, f"measured L2->SM reduction {measured:.2f}x"
    assert abs(measured / expected - 1.0) < 0.25


@pytest.mark.parametrize("name", ["gemm4096_bf16_cluster2x1", "gemm4096_bf16_cluster2x2", "gemm4096_bf16_pair2x1",
                                  "gemm4096_bf16_unicast", "gemm8192_bf16_pair_mcastB4",
                                  "gemm8192_bf16_unicast", "scores_8x16x4096x4096x128", "skinny_16384x128x8192",
                                  "skinny_128x16384x8192"])
def test_measured_l2_to_sm_bytes_follow_the_analytic_accounting(records, analytic, name):
    # Measured L2 -> SM reads sit a little below the analytic operand fetches where
    # requests for the same tile arrive close together (served once), and a little above
    # where the stream-K partials and beta * C reads come on top of the operands.
    w, p = analytic[name]
    ratio = records[name]["lts_bytes"] / p.l2_to_sm_operand_bytes
    assert 0.75 <= ratio <= 1.3, f"{name}: measured / analytic L2->SM bytes = {ratio:.3f}"


@pytest.mark.parametrize("name", ["scores_8x16x4096x4096x128", "skinny_16384x128x8192", "skinny_128x16384x8192",
                                  "attention_fwd_8x16x4096x4096x128"])
def test_dram_traffic_of_bandwidth_sensitive_workloads_stays_near_the_algorithmic_bytes(records, analytic, name):
    # The HBM-bound workloads read each input from DRAM about once: no wasted re-reads.
    # (Part of the output may still sit in L2 when the kernel ends, so the lower bound is
    # loose.)
    if name.startswith("attention"):
        from dense_gemm_cluster_gb300.workloads import ATTENTION_WORKLOADS
        algorithmic = ATTENTION_WORKLOADS[name].min_hbm_bytes()
    else:
        algorithmic = analytic[name][0].min_hbm_bytes()
    ratio = records[name]["dram_bytes"] / algorithmic
    assert 0.8 <= ratio <= 1.2, f"{name}: DRAM bytes / algorithmic bytes = {ratio:.3f}"


def test_pair_and_multicast_share_b_alike_on_4096(records, analytic):
    # A 2x1 cluster shares B either by multicast (each CTA receives the whole tile) or
    # through the pair MMA (each CTA loads half); both read B from L2 once per cluster.
    mc = records["gemm4096_bf16_cluster2x1"]["lts_bytes"]
    pair = records["gemm4096_bf16_pair2x1"]["lts_bytes"]
    assert (analytic["gemm4096_bf16_pair2x1"][1].l2_to_sm_operand_bytes ==
            analytic["gemm4096_bf16_cluster2x1"][1].l2_to_sm_operand_bytes)
    assert abs(pair / mc - 1.0) < 0.1
    # the pair also halves what crosses into each SM's shared memory for B
    assert records["gemm4096_bf16_pair2x1"]["xbar2sm_tma_bytes"] < 0.75 * records["gemm4096_bf16_cluster2x1"]["xbar2sm_tma_bytes"]


@pytest.mark.parametrize("name", ["gemm4096_bf16_cluster2x1", "gemm4096_bf16_cluster2x2", "gemm4096_bf16_pair2x1"])
def test_l2_resident_gemm_reads_its_inputs_once_plus_the_stream_k_partials(records, analytic, name):
    # 4096^3 fits in L2: DRAM sees A and B read once and C written once, plus at most one
    # round trip of the stream-K partials (each CTA parks at most one 128 x block_n fp32
    # partial at the start of the launch; the finisher reads it back tens of microseconds
    # later, after other tiles' operands may have pushed it out of L2).
    w, p = analytic[name]
    assert p.stream_k_tiles > 0
    ctas = p.clusters * p.cluster_m * p.cluster_n
    partials = ctas * p.block_m * p.block_n * 4
    got = records[name]["dram_bytes"]
    assert 0.8 * w.min_hbm_bytes() <= got <= 1.05 * (w.min_hbm_bytes() + 2 * partials), (
        f"{name}: {got / 1e6:.1f} MB of DRAM traffic against {w.min_hbm_bytes() / 1e6:.1f} MB of inputs and "
        f"output and {partials / 1e6:.1f} MB of partial slots")


def test_every_workload_has_a_record_taken_on_the_current_kernel_sources(records):
    # bench.py reports `traffic` and the measured L2 -> SM reduction only from records whose
    # source hash matches the kernels being built; every workload must have one.
    import bench
    from dense_gemm_cluster_gb300.workloads import ATTENTION_WORKLOADS, WORKLOADS
    gemm_sha = bench.kernel_source_hash()
    attn_sha = bench.kernel_source_hash(bench.ATTN_KERNEL_SOURCES)
    for name in WORKLOADS:
        assert records[name]["kernel_sha"] == gemm_sha, f"{name}: counters taken on other kernel sources"
        assert bench.recorded_traffic(name) is not None
    for name in ATTENTION_WORKLOADS:
        assert records[name]["kernel_sha"] == attn_sha, f"{name}: counters taken on other kernel sources"


def test_sharing_modes_cut_measured_l2_to_sm_bytes_against_their_unicast_twins(records, analytic):
    # Each sharing workload against the unicast workload that computes the same output:
    # the measured reduction tracks the analytic one (1.5x for a 2x1 cluster sharing B,
    # 2x for 2x2 multicast and for the pair with 4-CTA B multicast).
    from dense_gemm_cluster_gb300.workloads import UNICAST_TWIN
    for name, twin in UNICAST_TWIN.items():
        measured = records[twin]["lts_bytes"] / records[name]["lts_bytes"]
        expected = analytic[twin][1].l2_to_sm_operand_bytes / analytic[name][1].l2_to_sm_operand_bytes
        assert expected >= 1.5
        assert abs(measured / expected - 1.0) < 0.25, f"{name}: measured {measured:.2f}x, analytic {expected:.2f}x"
