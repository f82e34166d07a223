"""Runs the TMA unicast / multicast load microbenchmark (include/tma_bench.h).

    python -m dense_gemm_cluster_gb300.tma_bench [--sweep] [--scenario l2|dram] [--mode M]

Default: the two scenarios of "Hopper TMA Multicast 深度解析与实测", section
实机运行与 NCU 验证 (a 4096 x 4096 bf16 matrix, 128 x 64 tiles, 2-CTA
clusters, 5000 loads per CTA; L2 reuse and DRAM streaming), unicast against
multicast, rewritten for sm_103a with a pipelined ring of loads;
``--scenario`` / ``--mode`` run one of them alone (for profiling). ``--sweep``
varies the tile height, the ring depth and the cluster size. One JSON line per
run: time, delivered and issued bytes, delivered GB/s, bytes per SM cycle.
"""
from __future__ import annotations

import argparse
import json
import statistics

MODES = {"unicast": 0, "multicast": 1, "multicast_sliced": 2}


def run(mode="unicast", cluster=2, box_rows=128, stages=4, iters=5000, warmup=50, stride=0, ctas=0,
        rows=4096, cols=4096, src=None, device=0, landed=False):
    """One benchmark launch. With landed=True the result also holds every CTA's last landed
    tile (uint8 array, ctas x box_rows x 128 bytes, swizzled as in shared memory) and its
    (x, y) origin in src (int array, ctas x 2), for a full check against src."""
    import torch
    from . import gemm
    dev = torch.device("cuda", device)
    if src is None:
        src = (torch.arange(rows * cols, device=dev, dtype=torch.int32) % 65521).to(torch.int16)
    o = gemm.tma_bench_options_t()
    o.mode, o.cluster, o.ctas, o.box_rows = MODES[mode], cluster, ctas, box_rows
    o.stages, o.iters, o.warmup, o.streaming_stride = stages, iters, warmup, stride
    nmax = 512
    cycles = torch.zeros(nmax, dtype=torch.int64, device=dev)
    ns = torch.zeros(nmax, dtype=torch.int64, device=dev)
    verify = torch.zeros(nmax, dtype=torch.int32, device=dev)
    if landed:
        land = torch.zeros(nmax * box_rows * 128, dtype=torch.uint8, device=dev)
        orig = torch.full((nmax * 2,), -1, dtype=torch.int32, device=dev)
        o.landed, o.origin = land.data_ptr(), orig.data_ptr()
    stream = torch.cuda.current_stream(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    s, n, delivered, issued = gemm.tma_bench_run(o, src, rows, cols, cols, cycles, ns, verify, stream)
    end.record(stream)
    if s != gemm.GEMM_OK:
        raise gemm.GemmError(s, gemm.tma_bench_last_error())
    s = gemm.tma_bench_query_status(stream)
    if s != gemm.GEMM_OK:
        raise gemm.GemmError(s, gemm.tma_bench_last_error())
    ms = start.elapsed_time(end)
    cyc = cycles[:n].cpu().tolist()
    nss = ns[:n].cpu().tolist()
    bad = verify[:n].cpu().tolist()
    per_cta_bytes = iters * box_rows * 128
    extra = {}
    if landed:
        extra = {"landed": land[:n * box_rows * 128].cpu().numpy().reshape(n, box_rows * 128),
                 "origin": orig[:2 * n].cpu().numpy().reshape(n, 2)}
    return {**extra,
        "mode": mode if cluster > 1 else "unicast", "cluster": cluster, "ctas": n, "box_rows": box_rows,
        "stages": stages, "iters": iters, "stride": stride, "kernel_ms": ms,
        "timed_ms_max": max(nss) / 1e6, "delivered_bytes": delivered, "issued_bytes": issued,
        "delivered_GBps": delivered / (max(nss) * 1e-9) / 1e9,
        "bytes_per_sm_cycle": per_cta_bytes / statistics.median(cyc),
        "verify_errors": int(sum(1 for b in bad if b != 0)),
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--scenario", choices=("l2", "dram"), default=None, help="one scenario (default: both)")
    ap.add_argument("--mode", choices=sorted(MODES), default=None, help="one mode (default: unicast, multicast)")
    args = ap.parse_args(argv)
    import torch
    dev = torch.device("cuda", 0)
    rows = cols = 4096
    src = (torch.arange(rows * cols, device=dev, dtype=torch.int32) % 65521).to(torch.int16)
    big = None
    if not args.sweep:
        big_rows = 131072                      # 1 GiB of bf16: larger than L2
        scenarios = ((0, "L2 reuse"), (1, "DRAM streaming"))
        if args.scenario:
            scenarios = scenarios[:1] if args.scenario == "l2" else scenarios[1:]
        for stride, label in scenarios:
            if stride:
                big = (torch.arange(big_rows * cols, device=dev, dtype=torch.int32) % 65521).to(torch.int16)
            for mode in ((args.mode,) if args.mode else ("unicast", "multicast")):
                r = run(mode, 2, 128, 4, 5000, 50, stride, rows=big_rows if stride else rows, cols=cols,
                        src=big if stride else src)
                r["scenario"] = label
                print(json.dumps(r), flush=True)
        return 0
    for cluster in (1, 2, 4):
        for mode in (("unicast",) if cluster == 1 else ("unicast", "multicast", "multicast_sliced")):
            for box_rows in (64, 128, 256):
                for stages in (2, 4, 8):
                    if stages * box_rows * 128 > 200 * 1024:
                        continue
                    r = run(mode, cluster, box_rows, stages, 2000, 50, 0, src=src)
                    print(json.dumps(r), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
