"""The C-ABI library builds, loads, and exports every entry point the headers under include/ declare.

Also checks the host-only planner (no GPU needed): validation and launch plans.
"""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_cluster_gb300 import build
    build.build()
    from dense_gemm_cluster_gb300 import gemm
    return gemm


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b((?:gemm|tma_bench|stencil_1d|attention_forward)_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "gemm_run" in names and "gemm_create" in names and len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", lib.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib._lib, n)


def test_headers_are_plain_c(tmp_path):
    # The ABI is C: every header compiles on its own as C99 and C11, pedantically, without CUDA's
    # headers (streams cross the boundary as void *).
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    headers = sorted(fn for fn in os.listdir(os.path.join(ROOT, "include")) if fn.endswith(".h"))
    src = tmp_path / "h.c"
    src.write_text("".join(f'#include "{h}"\n' for h in headers) + "int main(void) { return 0; }\n")
    for std in ("c99", "c11"):
        r = subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                            "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


C_PROGRAM = r"""
#include <stdio.h>
#include "densegemm.h"
int main(void) {
    gemm_options_t o;
    gemm_options_default(&o);
    o.cta_group = 0; o.cluster_m = 4; o.mode = GEMM_MODE_MCAST; o.mcast_b = 1;
    gemm_plan_t p;
    gemm_status_t s = gemm_plan(&o, 8192, 8192, 8192, 1, 152, &p);
    if (s != GEMM_OK) { printf("plan %s\n", gemm_status_string(s)); return 1; }
    gemm_work_item_t items[64];
    int64_t n = gemm_schedule_work(p.tiles, 504, 64, 36, 0, items, 64);
    o.cta_group = 3;
    gemm_status_t bad = gemm_plan(&o, 8192, 8192, 8192, 1, 152, &p);
    printf("%d %d %lld %lld %d %d %s\n", p.cta_group, p.group_b, (long long)p.tiles, (long long)n,
           (int)items[0].kind, (int)bad, gemm_last_error(NULL));
    return 0;
}
"""


def test_a_c_program_links_against_the_library_and_plans(lib, tmp_path):
    # The boundary seen from C: the header, the shared library and the host-only calls, no GPU.
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from dense_gemm_cluster_gb300 import build
    so_dir = build.BUILD_DIR
    src, exe = tmp_path / "abi.c", tmp_path / "abi"
    src.write_text(C_PROGRAM)
    r = subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-L", so_dir, "-ldensegemm",
                        f"-Wl,-rpath,{so_dir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    cta_group, group_b, tiles, n_items, kind0, bad, *msg = out.stdout.split()
    # Automatic pair on an even cluster extent; 36 clusters walk 512 tiles: the first takes its
    # stream-K pieces first (kind 1 or 2), then 14 whole tiles.
    assert (cta_group, group_b, tiles) == ("2", "2", "512")
    assert int(n_items) == 14 + 1 and kind0 in ("1", "2")
    assert bad == "2" and "cta_group" in " ".join(msg)


def test_status_strings(lib):
    assert lib.gemm_status_string(0) == "GEMM_OK"
    assert lib.gemm_status_string(5) == "GEMM_ERR_DEVICE_TIMEOUT"
    assert lib.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


def test_options_default(lib):
    o = lib.gemm_options_default()
    assert (o.mode, o.cluster_m, o.cluster_n, o.cta_group) == (0, 1, 1, 1)
    assert (o.layout_a, o.layout_b, o.layout_c, o.out_type) == (0, 1, 0, 0)


def plan(lib, M, N, K, batch=1, sm=152, **kw):
    s, p = lib.gemm_plan(lib.make_options(**kw), M, N, K, batch, sm)
    return s, p


def test_plan_4096_cluster2x1(lib):
    s, p = plan(lib, 4096, 4096, 4096, mode="mcast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=1)
    assert s == 0
    assert (p.block_m, p.block_n, p.block_k) == (128, 256, 64)
    assert p.group_a == 1 and p.group_b == 2          # a 2x1 cluster shares only B
    assert p.tiles == (4096 // 256) * (4096 // 256)
    assert p.clusters == 76                           # 152 SMs in 2-CTA clusters
    assert p.smem_bytes <= 232448 and p.stages == 4
    from dense_gemm_cluster_gb300 import traffic
    assert p.l2_to_sm_operand_bytes == traffic.l2_to_sm_operand_bytes(4096, 4096, 4096, group_b=2)


def test_plan_pair_with_b_multicast(lib):
    s, p = plan(lib, 8192, 8192, 8192, cta_group=2, cluster_m=4, mode="mcast", mcast_b=1)
    assert s == 0 and p.group_b == 2 and p.group_a == 1
    assert p.block_k == 128 and p.stages == 3          # 64 KB stages: three fit
    s, p = plan(lib, 8192, 8192, 8192, cta_group=2, cluster_m=4, mode="mcast", mcast_b=1, block_k=64)
    assert s == 0 and p.block_k == 64 and p.stages == 6
    from dense_gemm_cluster_gb300 import traffic
    uni = traffic.l2_to_sm_operand_bytes(8192, 8192, 8192)
    assert uni == 2 * p.l2_to_sm_operand_bytes


def test_plan_column_major_c_swaps_roles(lib):
    s, p = plan(lib, 1000, 300, 64, layout_c="col", cluster_m=1, cluster_n=2, mode="mcast", mcast_a=1)
    assert s == 0 and p.transposed == 1
    assert (p.cluster_m, p.cluster_n) == (2, 1) and p.group_b == 2 and p.group_a == 1


def test_plan_auto_cta_group_pairs_even_cluster_rows(lib):
    # cta_group 0: the pair MMA wherever the cluster's extent along M is even, as launched
    # (column-major C runs C^T, so there it is cluster_n that must be even).
    for kw, want in [(dict(cluster_m=2), 2), (dict(cluster_m=4, mode="mcast", mcast_b=1), 2),
                     (dict(cluster_m=2, cluster_n=2, mode="mcast", mcast_a=1), 2), (dict(), 1),
                     (dict(cluster_n=2, mode="mcast", mcast_a=1), 1),
                     (dict(cluster_n=2, layout_c="col"), 2), (dict(cluster_m=2, layout_c="col"), 1)]:
        s, p = plan(lib, 4096, 4096, 4096, cta_group=0, **kw)
        assert s == 0 and p.cta_group == want, kw
    # The auto pair shares B within the pair: a 4-CTA cluster multicasts it across 2 pairs.
    s, p = plan(lib, 4096, 4096, 4096, cta_group=0, cluster_m=4, mode="mcast", mcast_b=1)
    assert s == 0 and p.group_b == 2


@pytest.mark.parametrize("kw,code", [
    (dict(cta_group=-1), 2),
    (dict(clock_probe=2), 1),
    (dict(cta_group=3), 2),
    (dict(cluster_m=3), 2),
    (dict(cluster_m=4, cluster_n=4), 2),
    (dict(cta_group=2, cluster_m=1), 2),
    (dict(block_n=96), 2),
    (dict(stages=1), 2),
    (dict(stages=9), 2),
    (dict(layout_a=2), 1),
    (dict(out_type=7), 1),
    (dict(mode=5), 1),
    (dict(host_parts=9), 1),
    (dict(host_parts=-1), 1),
])
def test_plan_rejects_bad_options(lib, kw, code):
    s, _ = plan(lib, 128, 128, 128, **kw)
    assert s == code, lib.gemm_last_error()
    assert lib.gemm_last_error()


def test_plan_rejects_bad_sizes(lib):
    assert plan(lib, -1, 4, 4)[0] == 1
    assert plan(lib, 1 << 31, 4, 4)[0] == 1
    s, p = plan(lib, 0, 0, 0)
    assert s == 0 and p.tiles == 0


def test_block_k_choice(lib):
    # K-major operands with K not a multiple of 64 cannot use the k-split map
    s, p = plan(lib, 512, 512, 200, cta_group=2, cluster_m=2)
    assert s == 0 and p.block_k == 64
    assert plan(lib, 512, 512, 200, cta_group=2, cluster_m=2, block_k=128)[0] == 2
    # both operands MN-major: any K works with 128-wide stages
    s, p = plan(lib, 512, 512, 200, cta_group=2, cluster_m=2, layout_a="col", layout_b="row", block_k=128)
    assert s == 0 and p.block_k == 128
    # 128x256 single-CTA tiles: 96 KB stages leave room for two only, so auto keeps 64
    s, p = plan(lib, 4096, 4096, 4096)
    assert p.block_k == 64 and p.stages == 4
    assert plan(lib, 64, 64, 64, block_k=32)[0] == 2


def test_unicast_mode_ignores_multicast_flags(lib):
    s, p = plan(lib, 512, 512, 512, mode="unicast", mcast_a=1, mcast_b=1, cluster_m=2, cluster_n=2)
    assert s == 0 and p.group_a == 1 and p.group_b == 1


def test_plan_stream_k_tail(lib):
    # 4096^3, 2x1 clusters: 256 cluster tiles on 76 clusters -> 3.37 waves; auto splits the tail
    s, p = plan(lib, 4096, 4096, 4096, sm=152, mode="mcast", mcast_b=1, cluster_m=2)
    assert s == 0 and p.clusters == 76
    assert p.stream_k_tiles == 256 - 2 * 76
    s, p = plan(lib, 4096, 4096, 4096, sm=152, mode="mcast", mcast_b=1, cluster_m=2, schedule="dp")
    assert p.stream_k_tiles == 0
    # a full last wave keeps whole tiles; a single k-block cannot be split
    s, p = plan(lib, 128 * 152, 256, 4096, sm=152)
    assert p.stream_k_tiles == 0
    s, p = plan(lib, 4096, 4096, 64, sm=152)
    assert p.stream_k_tiles == 0
    assert plan(lib, 64, 64, 64, schedule=4)[0] == 1
    s, p = plan(lib, 4096, 4096, 4096, sm=152, schedule="clc")
    assert s == 0 and p.stream_k_tiles == 0


def test_plan_sub_wave_spread(lib):
    # 6 tiles of 128x128 with 64 k-blocks each on 152 SMs: split 16 k-blocks a cluster
    s, p = plan(lib, 768, 128, 8192, sm=152, block_n=128)
    assert s == 0 and p.tiles == 6 and p.clusters == 24 and p.stream_k_tiles == 6
    s, p = plan(lib, 256, 256, 2048, sm=152)       # 2 tiles x 32 k-blocks: 4 clusters of 16
    assert p.tiles == 2 and p.clusters == 4 and p.stream_k_tiles == 2
    # whole tiles: more than half the clusters busy, a whole-tile schedule, or < 16 k-blocks a cluster
    s, p = plan(lib, 16384, 128, 8192, sm=152, block_n=128)
    assert p.tiles == 128 and p.clusters == 128 and p.stream_k_tiles == 0
    s, p = plan(lib, 768, 128, 8192, sm=152, block_n=128, schedule="dp")
    assert p.clusters == 6 and p.stream_k_tiles == 0
    # an explicit stream-K schedule spreads even when more than half the clusters are busy
    s, p = plan(lib, 16384, 128, 8192, sm=152, block_n=128, schedule="stream_k")
    assert p.tiles == 128 and p.clusters == 152 and p.stream_k_tiles == 128
    s, p = plan(lib, 16384, 128, 8192, sm=152, block_n=128, cta_group=2, cluster_m=2, schedule="stream_k")
    assert p.tiles == 64 and p.clusters == 76 and p.stream_k_tiles == 64
    s, p = plan(lib, 256, 256, 256, sm=152, mode="mcast", mcast_b=1, cluster_m=2)
    assert p.tiles == 1 and p.clusters == 1


def test_attention_validation_before_launch(lib):
    # Every one of these returns before any CUDA call (no GPU needed); the fake device
    # addresses are never dereferenced.
    a, m = 1 << 20, (1 << 20) + 2                # 16-byte aligned / misaligned fake addresses
    run = lib.attention_forward_run
    assert run(a, a, a, a, None, 1, 128, 128, 96) == lib.GEMM_ERR_UNSUPPORTED          # head dim
    assert run(a, a, a, a, None, 1, 128, 128, 64, 0.0, 0, 2, 2) == lib.GEMM_ERR_UNSUPPORTED   # pair needs 128
    assert run(a, a, a, a, None, 1, 128, 128, 128, 0.0, 0, 3) == lib.GEMM_ERR_UNSUPPORTED
    assert run(a, a, a, a, None, 1, 128, 128, 128, 0.0, 0, 4, 2) == lib.GEMM_ERR_UNSUPPORTED         # pair needs 2
    assert run(a, a, a, a, None, 1, 128, 128, 128, 0.0, 0, 2, 3) == lib.GEMM_ERR_UNSUPPORTED
    assert run(a, a, a, a, None, 1, 128, 0, 128) == lib.GEMM_ERR_INVALID_ARG              # no keys
    assert run(a, a, a, a, None, -1, 128, 128, 128) == lib.GEMM_ERR_INVALID_ARG
    assert run(None, a, a, a, None, 1, 128, 128, 128) == lib.GEMM_ERR_INVALID_ARG
    assert run(m, a, a, a, None, 1, 128, 128, 128) == lib.GEMM_ERR_ALIGNMENT
    assert run(a, a, a, a, m, 1, 128, 128, 128) == lib.GEMM_ERR_ALIGNMENT               # lse
    assert run(a, a, a, a, None, 1 << 31, 128, 128, 128) == lib.GEMM_ERR_INVALID_ARG      # batch limit
    assert run(a, a, a, a, None, 0, 128, 128, 128) == lib.GEMM_OK                         # nothing to do
    assert run(a, a, a, a, None, 3, 0, 128, 128) == lib.GEMM_OK
    # the host-buffer entry point checks its workspace and arguments before any copy
    need = lib.attention_forward_host_workspace_bytes(2, 300, 500, 128, 0)
    assert need >= 2 * (300 + 2 * 500) * 128 * 2 + 2 * 300 * (128 * 2 + 4)
    assert lib.attention_forward_host_workspace_bytes(0, 300, 500, 128, 0) == 0
    host = lib.attention_forward_run_host
    assert host(a, a, a, a, None, 2, 300, 500, 128, a, need - 1) == lib.GEMM_ERR_INVALID_ARG     # short
    assert host(a, a, a, a, None, 2, 300, 500, 128, None, need) == lib.GEMM_ERR_INVALID_ARG      # missing
    assert host(a, a, a, a, None, 2, 300, 500, 128, a + 16, need) == lib.GEMM_ERR_ALIGNMENT     # not 256-B aligned
    assert host(a, a, a, a, None, 2, 300, 500, 96, a, need) == lib.GEMM_ERR_UNSUPPORTED
    assert host(a, a, a, a, None, 2, 300, 500, 64, a, need, cluster=2, cta_group=2) == lib.GEMM_ERR_UNSUPPORTED
    assert host(a, a, a, a, None, 2, 300, 500, 128, a, need, cluster=4, cta_group=2) == lib.GEMM_ERR_UNSUPPORTED
    assert host(a, a, a, a, None, 0, 300, 500, 128, None, 0) == lib.GEMM_OK                     # nothing to do


def test_gemm_class_rejects_bad_options_before_any_device_call(lib):
    # resolve() refuses the options before the device is queried, so this needs no GPU
    with pytest.raises(lib.GemmError) as ei:
        lib.Gemm(0, cluster_m=16)
    assert ei.value.status == lib.GEMM_ERR_UNSUPPORTED
    with pytest.raises(TypeError):
        lib.Gemm(0, no_such_field=1)


def test_gemm_entry_points_refuse_a_null_handle_before_any_cuda_call(lib):
    a = 1 << 20                                   # fake aligned address, never dereferenced
    assert lib.gemm_run(None, 8, 8, 8, a, 8, a, 8, a, 8, 1.0, 0.0) == lib.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_strided_batched(None, 8, 8, 8, a, 8, 64, a, 8, 64, a, 8, 64, 2, 1.0, 0.0) == \
        lib.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_host(None, 8, 8, 8, a, 8, a, 8, a, 8, 1.0, 0.0) == lib.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_strided_batched_host(None, 8, 8, 8, a, 8, 64, a, 8, 64, a, 8, 64, 2, 1.0, 0.0) == \
        lib.GEMM_ERR_INVALID_ARG
    assert lib.gemm_query_status(None) == lib.GEMM_ERR_INVALID_ARG
    assert lib.gemm_read_clock(None)[0] == lib.GEMM_ERR_INVALID_ARG
    assert lib.gemm_destroy(None) == lib.GEMM_OK
    assert lib.gemm_launch_count(None) == -1


def test_multicast_refused_in_a_multi_gpu_job_before_any_cuda_call(lib, monkeypatch):
    # Cluster-multicast TMA loads are single-GPU only. With WORLD_SIZE > 1 every entry
    # point that would issue them refuses before touching the device (no GPU here; the
    # fake addresses are never dereferenced).
    a = 1 << 20
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert lib.attention_forward_run(a, a, a, a, None, 1, 256, 256, 128, 0.0, 0, 2, 1) == lib.GEMM_ERR_UNSUPPORTED
    assert lib.attention_forward_run(a, a, a, a, None, 1, 256, 256, 64, 0.0, 0, 4, 1) == lib.GEMM_ERR_UNSUPPORTED
    need = lib.attention_forward_host_workspace_bytes(2, 300, 500, 128, 0)
    assert lib.attention_forward_run_host(a, a, a, a, None, 2, 300, 500, 128, a, need, cluster=2) == \
        lib.GEMM_ERR_UNSUPPORTED
    for mode in (1, 2):
        o = lib.tma_bench_options_t(mode=mode, cluster=2, ctas=0, box_rows=128, stages=4, iters=8, warmup=0,
                                    streaming_stride=0, wait_timeout_ns=0)
        s, *_ = lib.tma_bench_run(o, a, 4096, 4096, 4096, a, a, a)
        assert s == lib.GEMM_ERR_UNSUPPORTED and "single-GPU" in lib.tma_bench_last_error()
    mc = lib.make_options(mode="mcast", mcast_b=1, cluster_m=2)
    assert lib.gemm_run_noalloc(mc, 0, 256, 256, 256, a, 256, a, 256, a, 256, 1.0, 0.0) == lib.GEMM_ERR_UNSUPPORTED
    assert "WORLD_SIZE" in lib.gemm_last_error(None)
    with pytest.raises(lib.GemmError) as ei:
        lib.Gemm(0, mode="mcast", mcast_b=1, cluster_m=2)
    assert ei.value.status == lib.GEMM_ERR_UNSUPPORTED


def test_noalloc_checks_options_before_the_device(lib):
    # Impossible options and sizes come back as such (not as a CUDA error) without a GPU:
    # gemm_run_noalloc validates before its one-time device set-up.
    a = 1 << 20
    run = lib.gemm_run_noalloc
    assert run(lib.make_options(cluster_m=16), 0, 256, 256, 256, a, 256, a, 256, a, 256, 1.0, 0.0) == \
        lib.GEMM_ERR_UNSUPPORTED
    assert run(lib.make_options(cta_group=2, cluster_m=1), 0, 256, 256, 256, a, 256, a, 256, a, 256, 1.0, 0.0) == \
        lib.GEMM_ERR_UNSUPPORTED
    assert run(lib.make_options(schedule="stream_k"), 0, 256, 256, 256, a, 256, a, 256, a, 256, 1.0, 0.0) == \
        lib.GEMM_ERR_UNSUPPORTED
    assert "workspace" in lib.gemm_last_error(None)
    assert run(lib.make_options(clock_probe=1), 0, 256, 256, 256, a, 256, a, 256, a, 256, 1.0, 0.0) == \
        lib.GEMM_ERR_UNSUPPORTED
    assert "clock probe" in lib.gemm_last_error(None)
    assert run(lib.make_options(), 0, -1, 256, 256, a, 256, a, 256, a, 256, 1.0, 0.0) == lib.GEMM_ERR_INVALID_ARG
    assert run(lib.make_options(), 99, 256, 256, 256, a, 256, a, 256, a, 256, 1.0, 0.0) == lib.GEMM_ERR_INVALID_ARG


def test_plan_l2_hints_and_k_rotation(lib):
    # One tile along N: A streams once (evict first), B is read by every tile (evict last),
    # and K-major A rows start at tile-dependent k-blocks.
    s, p = plan(lib, 16384, 128, 8192, layout_a="row", layout_b="row", cta_group=2, cluster_m=4, block_n=128,
                mode="mcast", mcast_b=1)
    assert s == 0 and (p.l2_hint_a, p.l2_hint_b, p.k_rotate) == (1, 2, 1)
    # One tile along M: the mirror; a row-major (MN-major) B is walked in lockstep.
    s, p = plan(lib, 128, 16384, 8192, layout_a="row", layout_b="row", block_n=128)
    assert s == 0 and (p.l2_hint_a, p.l2_hint_b, p.k_rotate) == (2, 1, 0)
    s, p = plan(lib, 128, 16384, 8192, layout_a="row", layout_b="col", block_n=128)
    assert s == 0 and (p.l2_hint_a, p.l2_hint_b, p.k_rotate) == (2, 1, 0)
    s, p = plan(lib, 16384, 128, 8192, layout_a="col", layout_b="row", block_n=128)
    assert s == 0 and (p.l2_hint_a, p.l2_hint_b, p.k_rotate) == (1, 2, 0)     # MN-major A: in order
    # Column-major C runs C^T = B^T A^T: the launched operands swap roles.
    s, p = plan(lib, 16384, 128, 8192, layout_a="row", layout_b="row", layout_c="col", block_n=128)
    assert s == 0 and p.transposed == 1 and (p.l2_hint_a, p.l2_hint_b) == (2, 1)
    # Tiles along both dimensions, or a batch: no hints, no rotation.
    for args, kw in [((8192, 8192, 8192), dict(cta_group=2, cluster_m=4, mode="mcast", mcast_b=1)),
                     ((4096, 4096, 4096), dict(cluster_m=2, mode="mcast", mcast_b=1)),
                     ((128, 128, 8192), dict())]:
        s, p = plan(lib, *args, **kw)
        assert s == 0 and (p.l2_hint_a, p.l2_hint_b, p.k_rotate) == (0, 0, 0), args
    s, p = plan(lib, 4096, 4096, 128, batch=128, layout_b="col", cluster_m=4, mode="mcast", mcast_b=1)
    assert s == 0 and (p.l2_hint_a, p.l2_hint_b, p.k_rotate) == (0, 0, 0)


def test_plan_serpentine_k_walk(lib):
    # Long K and at least two waves of whole tiles: successive tiles alternate direction.
    s, p = plan(lib, 8192, 8192, 8192, cta_group=2, cluster_m=4, mode="mcast", mcast_b=1)
    assert s == 0 and p.k_serpentine == 1 and p.k_rotate == 0
    # Short K (the score form's 2 k-blocks; 5 k-blocks), one wave, or a one-tile-wide grid: in order.
    for args, kw in [((4096, 4096, 128), dict(batch=128, layout_b="col", cluster_m=4, mode="mcast", mcast_b=1)),
                     ((3072, 4096, 320), dict()),
                     ((1024, 1024, 8192), dict()),
                     ((16384, 128, 8192), dict(cta_group=2, cluster_m=4, mode="mcast", mcast_b=1, block_n=128))]:
        s, p = plan(lib, *args, **kw)
        assert s == 0 and p.k_serpentine == 0, args


def test_plan_l2_prefetch_depth(lib):
    # A ring's worth of k-blocks in general; three on one-tile-wide grids, where each
    # tile streams an operand of its own; none with cluster launch control.
    s, p = plan(lib, 8192, 8192, 8192, cta_group=2, cluster_m=4, mode="mcast", mcast_b=1)
    assert s == 0 and p.prefetch_kb == p.stages
    s, p = plan(lib, 4096, 4096, 128, batch=128, layout_b="col", cluster_m=4, mode="mcast", mcast_b=1)
    assert s == 0 and p.prefetch_kb == p.stages
    for args, kw in [((16384, 128, 8192), dict(layout_b="row", cta_group=2, cluster_m=4, block_n=128, mode="mcast",
                                               mcast_b=1)),
                     ((128, 16384, 8192), dict(layout_b="row", cluster_n=2, block_n=128, mode="mcast", mcast_a=1))]:
        s, p = plan(lib, *args, **kw)
        assert s == 0 and p.l2_hint_a != 0 and p.prefetch_kb == 3 * p.stages, args
    s, p = plan(lib, 8192, 8192, 8192, schedule="clc")
    assert s == 0 and p.prefetch_kb == 0
