"""The persistent kernel's work partition, replayed on the host (no GPU).

``gemm_schedule_work`` runs the kernel's own work iterator compiled for the host.
Over hundreds of (tiles, whole tiles, k-blocks, clusters) shapes these tests
check what the stream-K finisher waits rely on ("Clusters, distributed shared
memory & cluster launch control", section "The second wall": the k-blocks of
the last waves are split evenly over every cluster):

* every k-block of every tile is computed exactly once, whole tiles by a
  static stride;
* a split tile has exactly one finisher, the cluster holding its first k-block,
  and the contributors it names are exactly the clusters holding its other
  parts (later clusters, consecutive);
* a contributor's part is the first unit of its cluster, so every partial is
  parked at the start of the launch, each cluster parks at most one (one
  workspace slot per CTA suffices), and split pieces come before whole tiles;
* no finisher waits on a part computed after its own: a simulation of the
  clusters advancing in order, a finisher blocking until its contributors'
  partials exist, always runs to completion.
"""
import random

import pytest

WHOLE, PARTIAL, FINISHER = 0, 1, 2


@pytest.fixture(scope="module")
def G():
    from dense_gemm_cluster_gb300 import build
    build.build()
    from dense_gemm_cluster_gb300 import gemm
    return gemm


def schedule(G, tiles, dp, num_kb, clusters):
    return [G.gemm_schedule_work(tiles, dp, num_kb, clusters, c) for c in range(clusters)]


def check_partition(work, tiles, dp, num_kb, clusters):
    covered = {}
    for c, items in enumerate(work):
        seen_whole = False
        partials = 0
        for i, (t, kb0, kb1, kind, cf, cn, last) in enumerate(items):
            assert 0 <= t < tiles and 0 <= kb0 < kb1 <= num_kb, (c, i)
            assert last == (i == len(items) - 1), (c, i, "last flag")
            for kb in range(kb0, kb1):
                assert (t, kb) not in covered, f"k-block {kb} of tile {t} twice"
                covered[(t, kb)] = (c, i)
            if kind == WHOLE:
                assert kb0 == 0 and kb1 == num_kb
                if t < dp:
                    assert t % clusters == c, "whole tiles go by a static stride"
                    seen_whole = True
            else:
                assert t >= dp, "only tiles past the whole ones are split"
                assert not seen_whole, "split pieces come before whole tiles"
            if kind == PARTIAL:
                partials += 1
                assert kb0 > 0
                assert i == 0, "a contributor's part is the first unit of its cluster"
            if kind == FINISHER:
                assert kb0 == 0 and kb1 < num_kb and cn >= 1 and cf == c + 1
                assert i == len(items) - 1 or items[i + 1][3] == WHOLE
        assert partials <= 1, "one parked partial per cluster (one workspace slot)"
    assert len(covered) == tiles * num_kb, "every k-block of every tile exactly once"
    # Finishers name exactly the clusters that hold the tile's other parts.
    for c, items in enumerate(work):
        for t, kb0, kb1, kind, cf, cn, last in items:
            if kind != FINISHER:
                continue
            holders = sorted({covered[(t, kb)][0] for kb in range(kb1, num_kb)})
            assert holders == list(range(cf, cf + cn)), (t, holders, cf, cn)
            for h in holders:
                assert work[h][0][0] == t and work[h][0][3] == PARTIAL


def runs_to_completion(work):
    """Clusters advance through their units in order; a finisher's unit completes only
    once every contributor has parked its partial (finished that unit)."""
    pos = [0] * len(work)
    parked = set()
    while True:
        progressed = False
        for c, items in enumerate(work):
            if pos[c] >= len(items):
                continue
            t, kb0, kb1, kind, cf, cn, last = items[pos[c]]
            if kind == FINISHER and not all((h, t) in parked for h in range(cf, cf + cn)):
                continue
            if kind == PARTIAL:
                parked.add((c, t))
            pos[c] += 1
            progressed = True
        if all(pos[c] >= len(items) for c, items in enumerate(work)):
            return True
        if not progressed:
            return False


def test_known_split():
    # 7 tiles of 10 k-blocks on 3 clusters, the first 3 whole: 40 k-blocks split 14/13/13.
    from dense_gemm_cluster_gb300 import build
    build.build()
    from dense_gemm_cluster_gb300 import gemm as G
    w = schedule(G, 7, 3, 10, 3)
    assert w[0] == [(3, 0, 10, WHOLE, -1, 0, 0), (4, 0, 4, FINISHER, 1, 1, 0), (0, 0, 10, WHOLE, -1, 0, 1)]
    assert w[1] == [(4, 4, 10, PARTIAL, -1, 0, 0), (5, 0, 7, FINISHER, 2, 1, 0), (1, 0, 10, WHOLE, -1, 0, 1)]
    assert w[2] == [(5, 7, 10, PARTIAL, -1, 0, 0), (6, 0, 10, WHOLE, -1, 0, 0), (2, 0, 10, WHOLE, -1, 0, 1)]


def test_partition_over_many_shapes(G):
    rng = random.Random(5)
    shapes = []
    for clusters in (1, 2, 3, 5, 19, 36, 38, 76, 152):
        for _ in range(40):
            tiles = rng.randint(0, 6 * clusters + 7)
            num_kb = rng.choice([1, 2, 3, 4, 7, 16, 33, 64, 128])
            waves = tiles // clusters
            dp = rng.randint(0, waves) * clusters
            shapes.append((tiles, dp, num_kb, clusters))
    # the planner's choices (whole waves less one, or everything whole) and sub-wave spreads
    for tiles, num_kb, clusters in [(512, 128, 36), (512, 64, 38), (128, 64, 38), (1024, 64, 152), (4, 4, 76),
                                    (65536, 2, 38), (24, 96, 19), (5, 200, 76)]:
        full = tiles // clusters
        shapes += [(tiles, max(0, full - 1) * clusters, num_kb, clusters), (tiles, tiles, num_kb, clusters)]
    for tiles, dp, num_kb, clusters in shapes:
        work = schedule(G, tiles, dp, num_kb, clusters)
        check_partition(work, tiles, dp, num_kb, clusters)
        assert runs_to_completion(work), (tiles, dp, num_kb, clusters)
    assert len(shapes) >= 300


def test_the_simulation_catches_a_finisher_that_waits_on_a_later_part():
    # A planted order (the contributor's partial after a unit that waits on the
    # finisher's cluster) must deadlock the simulation: the check is not vacuous.
    # Cluster 0 finishes tile 1 with cluster 1's partial, but cluster 1 first waits for
    # a partial of tile 2 from cluster 0, which is never parked.
    work = [[(1, 0, 5, FINISHER, 1, 1, 0), (0, 0, 10, WHOLE, -1, 0, 1)],
            [(2, 0, 5, FINISHER, 0, 1, 0), (1, 5, 10, PARTIAL, -1, 0, 1)]]
    assert not runs_to_completion(work)


def test_rejects_bad_arguments(G):
    from dense_gemm_cluster_gb300 import gemm
    with pytest.raises(ValueError):
        gemm.gemm_schedule_work(10, 11, 4, 2, 0)
    with pytest.raises(ValueError):
        gemm.gemm_schedule_work(10, 0, 4, 2, 2)
    assert gemm.gemm_schedule_work(0, 0, 4, 3, 1) == []
