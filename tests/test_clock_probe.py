"""GPU: the clock probe (options clock_probe = 1) counts every CTA of every launch, reads
the SM clock the kernel ran at, clears on read, and leaves the product unchanged.

The probe is measurement plumbing: the pages state no clock. What it reports is the ratio of
the SM cycle counter to the global nanosecond timer over each CTA's life, summed over CTAs.
"""
import numpy as np
import pytest

from gpu_cases import Problem, assert_close, options_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import torch
    from dense_gemm_cluster_gb300 import gemm
    assert torch.cuda.is_available()
    return gemm


@pytest.mark.parametrize("opts", [dict(), dict(cta_group=2, cluster_m=4, mode="mcast", mcast_b=1),
                                  dict(schedule="stream_k", mode="mcast", mcast_b=1, cluster_m=2)])
def test_probe_counts_every_cta_and_keeps_the_product(G, opts):
    p = Problem(1100, 1300, 512, la="row", lb="col", out="bf16", beta=0.5, seed=31)
    g = G.Gemm(0, clock_probe=1, **options_for(p, **opts))
    try:
        first = g.read_clock()                     # nothing launched yet
        assert (first["cycles"], first["ns"], first["ctas"]) == (0, 0, 0)
        dC = p.run(g, 1.0, 0.5)
        assert g.query_status() == G.GEMM_OK, G.gemm_last_error(g.handle)
        one = g.read_clock()
        cs = opts.get("cluster_m", 1) * opts.get("cluster_n", 1)
        assert 0 < one["ctas"] <= 152 and one["ctas"] % cs == 0
        assert one["cycles"] > 0 and one["ns"] > 0
        assert 0.5 < one["ghz"] < 3.0, one
        assert_close(p.result(dC), p.reference(1.0, 0.5), 512, "bf16", f"clock probe {opts}")
        for _ in range(3):
            p.run(g, 1.0, 0.5)
        three = g.read_clock()
        assert three["ctas"] == 3 * one["ctas"]
        again = g.read_clock()
        assert (again["cycles"], again["ns"], again["ctas"]) == (0, 0, 0)
    finally:
        g.close()


def test_probe_matches_an_unprobed_launch_bit_for_bit(G):
    p = Problem(700, 900, 448, la="row", lb="row", out="f32", beta=0.0, seed=32)
    outs = []
    for probe in (0, 1):
        g = G.Gemm(0, clock_probe=probe, **options_for(p, cta_group=2, cluster_m=2))
        try:
            dC = p.run(g)
            assert g.query_status() == G.GEMM_OK
            outs.append(p.result(dC))
        finally:
            g.close()
    assert np.array_equal(outs[0], outs[1])


def test_read_clock_needs_a_probed_handle(G):
    g = G.Gemm(0)
    try:
        with pytest.raises(G.GemmError) as ei:
            g.read_clock()
        assert ei.value.status == G.GEMM_ERR_INVALID_ARG
    finally:
        g.close()
