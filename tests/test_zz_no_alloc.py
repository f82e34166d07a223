"""gemm_run_noalloc: the handle-free GEMM entry point for callers that cannot
allocate device memory (code running while a pool holds the device's memory,
allocator callbacks, hosts that forbid allocation). Its status record lives in
a static device array; nothing is allocated.

Every call is checked against the fp64 oracle and against the handle entry
point's output, within the workloads' tolerance, on two calls in a row.

Collected last on purpose (file name), so that a failure here does not hide the
results of the other tests in a run that stops at the first failure. It must
pass both alone in a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

from gpu_cases import Problem, max_rel_err, options_for, tolerance, torch_dev

pytestmark = pytest.mark.gpu


def _handle_result(p, opts, alpha, beta):
    from dense_gemm_cluster_gb300 import gemm
    g = gemm.Gemm(0, **opts)
    try:
        dC = p.run(g, alpha, beta)
        assert g.query_status() == gemm.GEMM_OK
        return p.result(dC)
    finally:
        g.close()


@pytest.mark.parametrize("mode", [dict(mode="mcast", mcast_b=1, cluster_m=2, cluster_n=1),
                                  dict(cta_group=2, cluster_m=2, cluster_n=1, block_n=256),
                                  dict(mode="mcast", mcast_b=1, cta_group=2, cluster_m=4, cluster_n=1)])
def test_noalloc_matches_the_oracle_and_gemm_run_on_two_calls(mode):
    import torch
    from dense_gemm_cluster_gb300 import gemm

    assert torch.cuda.is_available()
    p = Problem(700, 900, 320, la="row", lb="row", out="bf16", beta=0.5, seed=21)
    opts = options_for(p, **mode)
    ref = p.reference(1.0, 0.5)
    via_handle = _handle_result(p, opts, 1.0, 0.5)
    tol = tolerance(p.K, "bf16")
    assert max_rel_err(via_handle, ref) <= tol

    o = gemm.make_options(**opts)
    dA, dB = torch_dev(p.A), torch_dev(p.B)
    for call in range(2):
        dC = torch_dev(p.C_in)                    # fresh C each call: beta reads it
        status = (ctypes.c_uint32 * 4)(99, 99, 99, 99)
        s = gemm.gemm_run_noalloc(o, 0, p.M, p.N, p.K, dA, p.lda, dB, p.ldb, dC, p.ldc, 1.0, 0.5, None, status)
        assert s == gemm.GEMM_OK, gemm.gemm_last_error(None)
        assert list(status) == [0, 0, 0, 0]       # cleared before the launch, still clear after it
        got = p.result(dC)
        assert np.isfinite(got).all()
        assert max_rel_err(got, ref) <= tol, f"call {call} against the oracle"
        assert max_rel_err(got, via_handle) <= tol, f"call {call} against gemm_run"


def test_noalloc_async_call_then_rejections():
    import torch
    from dense_gemm_cluster_gb300 import gemm

    p = Problem(256, 384, 128, la="row", lb="col", out="f32", seed=22)
    o = gemm.make_options(**options_for(p))
    dA, dB, dC = torch_dev(p.A), torch_dev(p.B), torch_dev(p.C_in)
    assert gemm.gemm_run_noalloc(o, 0, p.M, p.N, p.K, dA, p.lda, dB, p.ldb, dC, p.ldc, 1.0, 0.0) == gemm.GEMM_OK
    torch.cuda.synchronize()
    assert max_rel_err(p.result(dC), p.reference()) <= tolerance(p.K, "f32")
    # argument checks still apply: a misaligned leading dimension is refused before any launch
    s = gemm.gemm_run_noalloc(o, 0, p.M, p.N, p.K, dA, p.lda + 1, dB, p.ldb, dC, p.ldc, 1.0, 0.0)
    assert s == gemm.GEMM_ERR_ALIGNMENT and gemm.gemm_last_error(None)
    # K = 0 launches no GEMM kernel: C <- beta * C, and the status record reads clear
    status = (ctypes.c_uint32 * 4)(7, 7, 7, 7)
    C0 = torch.full((p.M, p.N), 2.0, dtype=torch.float32, device="cuda")
    s = gemm.gemm_run_noalloc(o, 0, p.M, p.N, 0, None, 8, None, p.ldb, C0, p.N, 1.0, 0.25, None, status)
    assert s == gemm.GEMM_OK and list(status) == [0, 0, 0, 0]
    assert bool((C0 == 0.5).all())


def test_noalloc_timeout_is_reported_then_the_next_call_is_clean():
    # A host-planted protocol mistake (16 bytes announced that never arrive) makes the
    # MMA's bounded wait run out; the kernel records it in the static record and returns.
    from dense_gemm_cluster_gb300 import gemm

    p = Problem(256, 256, 256, la="row", lb="col", out="f32", seed=23)
    bad = gemm.make_options(debug_flags=gemm.GEMM_DEBUG_EXTRA_TX, wait_timeout_ns=20_000_000,
                            **options_for(p, mode="mcast", mcast_b=1, cluster_m=2))
    dA, dB = torch_dev(p.A), torch_dev(p.B)
    status = (ctypes.c_uint32 * 4)(0, 0, 0, 0)
    s = gemm.gemm_run_noalloc(bad, 0, p.M, p.N, p.K, dA, p.lda, dB, p.ldb, torch_dev(p.C_in), p.ldc, 1.0, 0.0,
                              None, status)
    assert s == gemm.GEMM_ERR_DEVICE_TIMEOUT
    assert status[0] != 0 and "bounded wait expired" in gemm.gemm_last_error(None)
    good = gemm.make_options(**options_for(p, mode="mcast", mcast_b=1, cluster_m=2))
    status = (ctypes.c_uint32 * 4)(99, 99, 99, 99)
    dC = torch_dev(p.C_in)
    s = gemm.gemm_run_noalloc(good, 0, p.M, p.N, p.K, dA, p.lda, dB, p.ldb, dC, p.ldc, 1.0, 0.0, None, status)
    assert s == gemm.GEMM_OK and list(status) == [0, 0, 0, 0]
    assert max_rel_err(p.result(dC), p.reference()) <= tolerance(p.K, "f32")
