"""Host-side pins: the seeded generator and the analytic byte accounting."""
import json
import os

import numpy as np
import pytest

from dense_gemm_cluster_gb300 import inputs, traffic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_outputs():
    # First outputs of splitmix64 from state 0 (Steele, Lea, Flood 2014; the
    # reference C implementation by Vigna prints these for seed 0).
    got = [int(x) for x in inputs.splitmix64(0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # counter-based: any window equals the same slice of a longer draw
    assert np.array_equal(inputs.splitmix64(7, 5, offset=10), inputs.splitmix64(7, 15)[10:])


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -2.5, 0.0])
    assert list(inputs.f64_to_bf16_bits(x)) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000]
    bits = np.arange(0, 0x7F80, 97, dtype=np.uint16)       # finite positive patterns
    assert np.array_equal(inputs.f64_to_bf16_bits(inputs.bf16_bits_to_f32(bits).astype(np.float64)), bits)


def test_distributions_have_the_named_moments():
    n = 1 << 18
    z = inputs.normal(0, n)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1.0) < 0.01
    u = 2.0 * inputs.uniform01(1, n) - 1.0
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1.0 / 3.0) < 0.01
    s = inputs.bf16_matrix(64, 64, "normal", 3, scale=1.0 / 64.0)
    v = inputs.bf16_bits_to_f32(s)
    assert abs(v.std() - 1.0 / 64.0) < 0.002


def test_streams_are_deterministic_and_distinct():
    a = inputs.bf16_matrix(16, 16, "uniform", 0)
    assert np.array_equal(a, inputs.bf16_matrix(16, 16, "uniform", 0))
    assert not np.array_equal(a, inputs.bf16_matrix(16, 16, "uniform", 1))


def test_store_layouts_round_trip():
    m = inputs.bf16_matrix(5, 9, "normal", 4)
    r, ldr = inputs.store(m, "row")
    c, ldc = inputs.store(m, "col")
    assert ldr == 16 and ldc == 8
    assert np.array_equal(r[:, :9], m) and np.array_equal(c[:, :5].T, m)


def test_page1_traffic_accounting_matches_printed_figures():
    g = json.load(open(os.path.join(GOLDEN, "tma_multicast_h100.json")))
    assert g["tile_rows"] * g["tile_cols"] * g["elem_bytes"] == g["tile_bytes"]
    b = traffic.tma_scenario_bytes(g["ctas"], g["cluster"], g["iters"], g["tile_bytes"])
    assert b["issued_unicast"] / 1e6 == pytest.approx(g["unicast_MB"], abs=1e-9)
    assert b["issued_multicast"] / 1e6 == pytest.approx(g["multicast_MB"], abs=1e-9)
    assert 100.0 * (1 - b["issued_multicast"] / b["issued_unicast"]) == pytest.approx(g["reduction_pct"])
    # delivered bandwidth = delivered bytes / time (the printed example agrees to 0.2%)
    assert b["delivered"] / (g["unicast_ms"] * 1e-3) / 1e9 == pytest.approx(g["unicast_GBps"], rel=2e-3)
    assert b["delivered"] / (g["multicast_ms"] * 1e-3) / 1e9 == pytest.approx(g["multicast_GBps"], rel=2e-3)
    assert g["unicast_ms"] / g["multicast_ms"] == pytest.approx(g["speedup"], abs=0.005)


def test_gemm_operand_bytes_closed_forms():
    # 8192^3: unicast 128x256 tiles vs the pair + 4-CTA B multicast: exactly 2x
    uni = traffic.l2_to_sm_operand_bytes(8192, 8192, 8192, block_n=256)
    pair = traffic.l2_to_sm_operand_bytes(8192, 8192, 8192, cta_group=2, block_n=256, group_b=2)
    assert uni == 64 * 32 * 8192 * 2 * (128 + 256)
    assert uni == 2 * pair
    # 4096^3 with a 2-CTA cluster along M sharing B: (128+256)/(128+128) = 1.5x
    a = traffic.l2_to_sm_operand_bytes(4096, 4096, 4096)
    b = traffic.l2_to_sm_operand_bytes(4096, 4096, 4096, group_b=2)
    assert a / b == pytest.approx(1.5)
    # K tail counted as a whole box
    assert traffic.l2_to_sm_operand_bytes(128, 256, 1) == 64 * 2 * 384
    with pytest.raises(ValueError):
        traffic.tma_scenario_bytes(3, 2, 1, 1)
