"""GPU checks of the TMA unicast / multicast microbenchmark: every tile lands
where the 128-byte swizzle puts it, in every mode, and the byte accounting
follows the page-1 rule (multicast issues 1/cluster of what it delivers)."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,cluster,box_rows,stages,stride", [
    ("unicast", 1, 128, 4, 0), ("unicast", 2, 128, 4, 1), ("multicast", 2, 128, 4, 0),
    ("multicast", 4, 64, 8, 1), ("multicast_sliced", 2, 128, 4, 0), ("multicast_sliced", 4, 256, 2, 1),
    ("multicast", 2, 8, 1, 0)])
def test_tiles_land_and_bytes_add_up(mode, cluster, box_rows, stages, stride):
    from dense_gemm_cluster_gb300 import tma_bench
    r = tma_bench.run(mode, cluster, box_rows, stages, iters=300, warmup=10, stride=stride, rows=2048, cols=1024)
    assert r["verify_errors"] == 0
    assert r["delivered_bytes"] == r["ctas"] * 300 * box_rows * 128
    if mode == "unicast" or cluster == 1:
        assert r["issued_bytes"] == r["delivered_bytes"]
    else:
        assert r["issued_bytes"] * cluster == r["delivered_bytes"]
    assert r["kernel_ms"] > 0 and r["bytes_per_sm_cycle"] > 0


def _unswizzle(tile: "np.ndarray", rows: int) -> "np.ndarray":
    # 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8) of that row.
    import numpy as np
    t = tile.reshape(rows, 8, 16)
    out = np.empty_like(t)
    for r in range(rows):
        out[r, np.arange(8) ^ (r % 8)] = t[r]
    return out.reshape(rows, 128).view(np.int16)


@pytest.mark.parametrize("mode,cluster,box_rows,stages,stride", [
    ("unicast", 2, 128, 4, 1), ("multicast", 2, 128, 4, 0), ("multicast", 4, 64, 8, 1),
    ("multicast_sliced", 2, 128, 4, 1), ("multicast_sliced", 4, 256, 2, 0)])
def test_every_element_of_the_last_landed_tile_matches_the_source(mode, cluster, box_rows, stages, stride):
    # Each CTA copies its last landed tile out of shared memory; every element, un-swizzled,
    # must equal the source at the tile's origin (in every CTA of a multicast cluster).
    import numpy as np
    import torch
    from dense_gemm_cluster_gb300 import tma_bench
    rows, cols = 2048, 1024
    src = (torch.arange(rows * cols, device="cuda", dtype=torch.int32) % 65521).to(torch.int16)
    r = tma_bench.run(mode, cluster, box_rows, stages, iters=97, warmup=3, stride=stride, rows=rows, cols=cols,
                      src=src, landed=True)
    host = src.cpu().numpy().reshape(rows, cols)
    assert r["verify_errors"] == 0 and r["ctas"] > 0
    for i in range(r["ctas"]):
        x, y = (int(v) for v in r["origin"][i])
        assert 0 <= x <= cols - 64 and 0 <= y <= rows - box_rows
        got = _unswizzle(r["landed"][i], box_rows)
        assert np.array_equal(got, host[y:y + box_rows, x:x + 64]), f"CTA {i} tile at ({x}, {y})"


def test_rejects_bad_options():
    from dense_gemm_cluster_gb300 import gemm, tma_bench
    with pytest.raises(gemm.GemmError):
        tma_bench.run("multicast_sliced", 4, 8, 2, iters=10, rows=1024, cols=1024)   # 8 rows cannot split in 4
    with pytest.raises(gemm.GemmError):
        tma_bench.run("unicast", 3, 128, 2, iters=10, rows=1024, cols=1024)
