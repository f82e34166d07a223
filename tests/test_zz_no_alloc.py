"""gemm_run_noalloc: the handle-free GEMM entry point for callers that cannot
allocate device memory (its status record lives in a static device array).

Collected last on purpose (file name), so that a failure here does not hide the
results of the other tests in a run that stops at the first failure. It must
pass both alone in a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

from gpu_cases import Problem, max_rel_err, options_for, tolerance, torch_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_gemm_run_on_two_calls():
    import torch
    from dense_gemm_cluster_gb300 import gemm

    assert torch.cuda.is_available()
    p = Problem(700, 900, 320, la="row", lb="row", out="bf16", beta=0.5, seed=21)
    opts = options_for(p, mode="mcast", mcast_b=1, cluster_m=2, cluster_n=1)

    # The existing entry point, through a handle.
    g = gemm.Gemm(0, **opts)
    ref_dev = p.run(g, 1.0, 0.5)
    assert g.query_status() == gemm.GEMM_OK
    ref = p.result(ref_dev)
    g.close()

    o = gemm.make_options(**opts)
    dA, dB = torch_dev(p.A), torch_dev(p.B)
    for call in range(2):
        dC = torch_dev(p.C_in)                    # fresh C each call: beta reads it
        status = (ctypes.c_uint32 * 4)(99, 99, 99, 99)
        s = gemm.gemm_run_noalloc(o, 0, p.M, p.N, p.K, dA, p.lda, dB, p.ldb, dC, p.ldc, 1.0, 0.5, None, status)
        assert s == gemm.GEMM_OK, gemm.gemm_last_error(None)
        assert list(status) == [0, 0, 0, 0]       # cleared before the launch, still clear after it
        got = p.result(dC)
        err = max_rel_err(got, ref)
        assert err <= tolerance(p.K, "bf16"), f"call {call}: {err}"
        assert np.isfinite(got).all()


def test_noalloc_async_call_then_rejections():
    import torch
    from dense_gemm_cluster_gb300 import gemm

    p = Problem(256, 384, 128, la="row", lb="col", out="f32", seed=22)
    o = gemm.make_options(**options_for(p))
    dA, dB, dC = torch_dev(p.A), torch_dev(p.B), torch_dev(p.C_in)
    assert gemm.gemm_run_noalloc(o, 0, p.M, p.N, p.K, dA, p.lda, dB, p.ldb, dC, p.ldc, 1.0, 0.0) == gemm.GEMM_OK
    torch.cuda.synchronize()
    ref = p.reference()
    assert max_rel_err(p.result(dC), ref) <= tolerance(p.K, "f32")
    # argument checks still apply: a misaligned leading dimension is refused before any launch
    s = gemm.gemm_run_noalloc(o, 0, p.M, p.N, p.K, dA, p.lda + 1, dB, p.ldb, dC, p.ldc, 1.0, 0.0)
    assert s == gemm.GEMM_ERR_ALIGNMENT and gemm.gemm_last_error(None)
