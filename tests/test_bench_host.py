"""Host logic of bench.py without a GPU: the whole-job aggregation over ranks
(max of elapsed time, sum of work) on a world_size-2 gloo group, the clock
sampler's parsing of nvidia-smi CSV, and the reference arm's JSON line."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed, units = bench.aggregate(dist, elapsed_s=1.0 + rank, units=10.0 * (rank + 1))
    out[rank] = (elapsed, units)
    dist.destroy_process_group()


def test_aggregate_is_max_time_and_sum_of_work_over_two_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == (2.0, 30.0)


def test_aggregate_single_process_passthrough():
    import bench
    assert bench.aggregate(None, 1.5, 7.0) == (1.5, 7.0)


def test_clock_sampler_parses_throttle_reasons(tmp_path):
    import bench
    s = bench.ClockSampler(0)
    f = tmp_path / "c.csv"
    f.write_text("0, 1980, 2070, 700.5, 0x0, Not Active, Not Active, Not Active, Active\n"
                 "0, 2000, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, Not Active\n")
    s.file = open(f, "a+")
    s.proc = object()
    summ = s.summary()
    assert summ["sm_mhz"] == 1990.0 and summ["sm_max_mhz"] == 2070.0
    assert summ["reasons"] == ["sw_power_cap"] and summ["samples"] == 2


def test_reference_arm_prints_one_contract_line_without_a_gpu():
    # `bench.py --impl reference` times the fp64 oracle on the host cores; it must print one
    # JSON line with the contract's keys, its own cpu_baseline and a zero-byte e2e.
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "gemm256_f32_mcastB",
                        "--steps", "2", "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "gemm256_f32_mcastB"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_l2_to_sm_report_divides_the_unicast_twins_measured_bytes():
    # The bench line's multicast evidence: the unicast twin's ncu L2 -> SM bytes over this
    # workload's, both from records taken on the current kernel sources.
    import bench
    from dense_gemm_cluster_gb300 import build
    build.build()
    from dense_gemm_cluster_gb300 import gemm
    from dense_gemm_cluster_gb300.workloads import WORKLOADS
    w = WORKLOADS["gemm8192_bf16_pair_mcastB4"]
    opts = gemm.make_options(layout_a=w.layout_a, layout_b=w.layout_b, layout_c=w.layout_c, out_type=w.out,
                             **w.options)
    _, plan = gemm.gemm_plan(opts, w.M, w.N, w.K, w.batch, 152)
    _, uni = gemm.gemm_plan(gemm.make_options(layout_a=w.layout_a, layout_b=w.layout_b, block_n=256),
                            w.M, w.N, w.K, w.batch, 152)
    rec = bench.recorded_traffic(w.name)
    r = bench.l2_to_sm_report(w, plan, uni, rec)
    assert r["unicast_workload"] == "gemm8192_bf16_unicast"
    assert r["reduction_vs_unicast"] == pytest.approx(2.0)
    twin = bench.recorded_traffic("gemm8192_bf16_unicast")
    assert r["reduction_measured"] == pytest.approx(twin["lts_bytes"] / rec["lts_bytes"])
    assert r["reduction_measured"] >= 1.8
    # without a record (stale or missing) nothing is claimed
    r = bench.l2_to_sm_report(w, plan, uni, None)
    assert r["measured"] is None and r["reduction_measured"] is None
    # a workload without a unicast twin reports the analytic ratio only
    s = WORKLOADS["scores_8x16x4096x4096x128"]
    r = bench.l2_to_sm_report(s, plan, uni, bench.recorded_traffic(s.name))
    assert r["unicast_workload"] is None and r["reduction_measured"] is None


def test_nvml_clock_summary_windows_and_reasons():
    # The in-process clock record: only samples inside the window count; the clock-event
    # reason bits decode to the names the throttle checks use.
    import bench
    c = bench.NvmlClocks.__new__(bench.NvmlClocks)
    c.ok, c.max_mhz, c.period_s = True, 2070.0, 0.001
    c.samples = [(0.5, 2070.0, 150.0, 0x0),                 # before the window
                 (1.0, 2070.0, 900.0, 0x0), (1.1, 1500.0, 1390.0, 0x4),
                 (1.2, 1480.0, 1395.0, 0x4 | 0x40), (2.5, 900.0, 100.0, 0x8)]   # the last after it
    s = c.summary(0.9, 1.3)
    assert s["samples"] == 3 and s["sm_mhz"] == 1500.0 and s["sm_mhz_min"] == 1480.0
    assert s["power_w_max"] == 1395.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    c.ok = False
    assert c.summary(0.0, 9.0)["reasons"] == ["nvml unavailable"]


def test_in_kernel_clock_and_the_tensor_peak_at_that_clock():
    import bench
    c = bench.in_kernel_clock({"cycles": 18_670_000_000, "ns": 10_000_000_000, "ctas": 2880}, 20)
    assert c["sm_ghz_in_kernel"] == pytest.approx(1.867) and c["ctas_per_launch"] == 144
    r = bench.tensor_peak_at_kernel_clock(1909.6, c, 152)
    assert r["peak_all_sms"] == pytest.approx(152 * 8192 * 1.867 / 1e3)
    assert r["peak_sms_used"] == pytest.approx(144 * 8192 * 1.867 / 1e3)
    assert r["frac_sms_used"] == pytest.approx(1909.6 / (144 * 8192 * 1.867 / 1e3))
    assert bench.in_kernel_clock({"cycles": 0, "ns": 0, "ctas": 0}, 20) == {"sm_ghz_in_kernel": None}
    assert bench.tensor_peak_at_kernel_clock(1000.0, {"sm_ghz_in_kernel": None}, 152) is None


def test_smem_port_bound_of_the_tile_shapes():
    # Per K = 16 step of one CTA: TMA writes and the MMA reads the A rows and the CTA's share of
    # B's columns; a 128 x 256 single-CTA tile moves 192 B per tensor clock through a 128 B port.
    import bench
    one = bench.smem_port_bound(128, 256, 1)
    assert one["bytes_per_tensor_clk"] == pytest.approx(192.0) and one["tensor_util_bound"] == pytest.approx(2 / 3)
    pair = bench.smem_port_bound(128, 256, 2)
    assert pair["bytes_per_tensor_clk"] == pytest.approx(128.0) and pair["tensor_util_bound"] == 1.0
    narrow = bench.smem_port_bound(128, 128, 1)
    assert narrow["bytes_per_tensor_clk"] == pytest.approx(256.0) and narrow["tensor_util_bound"] == pytest.approx(0.5)
