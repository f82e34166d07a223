"""GPU parity of the cluster halo-exchange stencil against the fp64 oracle.

Halos inside a cluster come from the neighbours' shared memory (DSMEM); halos
at cluster edges from global memory; the result must not depend on which.
Dyadic inputs make every fp32 operation exact, so those cases compare bit for
bit; random inputs are held to two fp32 roundings of the terms' magnitudes.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _run(x, cluster):
    import torch
    from dense_gemm_cluster_gb300 import gemm
    dx = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    dy = torch.full_like(dx, float("nan"))
    assert gemm.stencil_1d_run(dx, dy, x.shape[0], cluster) == gemm.GEMM_OK
    assert gemm.stencil_1d_query_status() == gemm.GEMM_OK
    return dy.cpu().numpy().astype(np.float64)


TILE = 8192


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
@pytest.mark.parametrize("n", [1, 3, 5, TILE - 1, TILE, TILE + 1, 3 * TILE + 7, 9 * TILE, 20 * TILE + 4093])
def test_dyadic_inputs_bit_exact(cluster, n):
    import oracle
    rng = np.random.default_rng(n * 8 + cluster)
    x = (rng.integers(-512, 512, size=n) * 4.0).astype(np.float32)     # multiples of 4: every step exact
    assert np.array_equal(_run(x, cluster), oracle.stencil_1d(x))


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
def test_random_inputs_within_two_roundings(cluster):
    import oracle
    from dense_gemm_cluster_gb300 import inputs
    n = 37 * TILE + 1001
    x = (2.0 * inputs.uniform01(3, n) - 1.0).astype(np.float32)
    got = _run(x, cluster)
    ref = oracle.stencil_1d(x)
    xa = np.abs(x.astype(np.float64))
    mag = 0.5 * xa
    mag[1:] += 0.25 * xa[:-1]
    mag[:-1] += 0.25 * xa[1:]
    assert np.all(np.abs(got - ref) <= 2.0 ** -22 * mag + 1e-30)


def test_halo_values_cross_tiles_and_clusters():
    # a unit impulse on each side of every tile and cluster edge must spread into the neighbour tile
    import oracle
    n = 16 * TILE
    x = np.zeros(n, np.float32)
    for t in range(1, 16):
        x[t * TILE - 1] = 4.0
        x[t * TILE] = 8.0
    for c in (1, 2, 4, 8):
        assert np.array_equal(_run(x, c), oracle.stencil_1d(x))


def test_argument_errors():
    import torch
    from dense_gemm_cluster_gb300 import gemm
    x = torch.zeros(64, device="cuda")
    y = torch.zeros(64, device="cuda")
    assert gemm.stencil_1d_run(x, y, 64, 3) == gemm.GEMM_ERR_UNSUPPORTED
    assert gemm.stencil_1d_run(x.data_ptr() + 4, y, 60, 2) == gemm.GEMM_ERR_ALIGNMENT
    assert gemm.stencil_1d_run(x, x, 64, 2) == gemm.GEMM_ERR_INVALID_ARG
    assert gemm.stencil_1d_run(x, y, 0, 2) == gemm.GEMM_OK
