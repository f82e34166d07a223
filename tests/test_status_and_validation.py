"""Failure detection and argument checks through the C ABI.

The timeout test plants a mistake in the arming protocol (16 bytes announced
that never arrive, GEMM_DEBUG_EXTRA_TX), so the MMA warp's bounded wait on the
first stage must run out. The kernel records the reason in its status word and
every role stops; nothing faults, traps or spins without a limit, and the same
context then runs a normal GEMM correctly.
"""
import numpy as np
import pytest

from gpu_cases import Problem, assert_close, options_for, torch_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import torch
    from dense_gemm_cluster_gb300 import gemm
    assert torch.cuda.is_available()
    return gemm


@pytest.mark.parametrize("mode", [dict(), dict(mode="mcast", mcast_b=1, cluster_m=2),
                                  dict(cta_group=2, cluster_m=2)])
def test_bounded_wait_reports_timeout_then_context_still_works(G, mode):
    p = Problem(256, 256, 256, la="row", lb="col", out="f32", seed=31)
    g = G.Gemm(0, debug_flags=G.GEMM_DEBUG_EXTRA_TX, wait_timeout_ns=20_000_000, **options_for(p, **mode))
    dC = torch_dev(p.C_in)
    g.run(p.M, p.N, p.K, torch_dev(p.A), p.lda, torch_dev(p.B), p.ldb, dC, p.ldc)
    s = g.query_status()
    assert s == G.GEMM_ERR_DEVICE_TIMEOUT
    assert "bounded wait expired" in G.gemm_last_error(g.handle)
    assert g.query_status() == G.GEMM_OK          # the status word was cleared
    g.close()
    # the context is intact: a normal run on it is correct
    g2 = G.Gemm(0, **options_for(p, **mode))
    got = p.result(p.run(g2))
    assert g2.query_status() == G.GEMM_OK
    assert_close(got, p.reference(), p.K, "f32", "after timeout")
    g2.close()


def test_argument_errors_come_back_before_launch(G):
    import torch
    g = G.Gemm(0, layout_a="row", layout_b="col", out_type="bf16")
    A = torch.zeros(256 * 64, dtype=torch.int16, device="cuda")
    B = torch.zeros(256 * 64, dtype=torch.int16, device="cuda")
    C = torch.zeros(256 * 256, dtype=torch.int16, device="cuda")
    n0 = g.launches
    run = lambda *a: G.gemm_run(g.handle, *a)
    assert run(256, 256, 64, A, 63, B, 64, C, 256, 1.0, 0.0) == G.GEMM_ERR_INVALID_ARG    # lda < K
    assert run(256, 256, 64, A, 72 + 1, B, 64, C, 256, 1.0, 0.0) == G.GEMM_ERR_ALIGNMENT   # lda*2 % 16
    assert run(256, 256, 64, A.data_ptr() + 2, 64, B, 64, C, 256, 1.0, 0.0) == G.GEMM_ERR_ALIGNMENT
    assert run(256, 256, 64, None, 64, B, 64, C, 256, 1.0, 0.0) == G.GEMM_ERR_INVALID_ARG
    assert run(256, 256, 64, A, 64, B, 64, None, 256, 1.0, 0.0) == G.GEMM_ERR_INVALID_ARG
    assert run(-1, 256, 64, A, 64, B, 64, C, 256, 1.0, 0.0) == G.GEMM_ERR_INVALID_ARG
    assert run(0, 256, 64, A, 64, B, 64, C, 256, 1.0, 0.0) == G.GEMM_OK                   # empty: no-op
    assert g.launches == n0
    assert G.gemm_run(0, 1, 1, 1, A, 8, B, 8, C, 8, 1.0, 0.0) == G.GEMM_ERR_INVALID_ARG   # null handle
    g.close()


def test_create_rejects_impossible_modes(G):
    with pytest.raises(G.GemmError) as e:
        G.Gemm(0, cta_group=2, cluster_m=1)
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED
    with pytest.raises(G.GemmError):
        G.Gemm(0, cluster_m=4, cluster_n=4)


def test_multicast_refused_in_a_multi_gpu_job(G, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(G.GemmError) as e:
        G.Gemm(0, mode="mcast", mcast_b=1, cluster_m=2)
    assert e.value.status == G.GEMM_ERR_UNSUPPORTED
    G.Gemm(0, cta_group=2, cluster_m=2).close()          # the pair MMA without multicast is fine


def test_host_buffer_entry_point(G):
    p = Problem(300, 260, 192, la="row", lb="row", out="bf16", beta=0.5, seed=32)
    g = G.Gemm(0, **options_for(p, mode="mcast", mcast_b=1, cluster_m=2))
    C = p.C_in.copy()
    g.run_host(p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, C, p.ldc, 1.0, 0.5)
    from gpu_cases import decode
    assert_close(decode(C, p.M, p.N, "row"), p.reference(1.0, 0.5), p.K, "bf16", "host buffers")
    g.close()
