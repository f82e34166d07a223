"""Throughput of the fused attention forward (include/attention.h).

    python -m dense_gemm_cluster_gb300.attention [--batch B] [--sq S] [--sk S] [--d D] [--cluster C]
                                                 [--cta-group G] [--causal] [--steps K] [--warmup W]

One JSON line per cluster size: TFLOP/s (4 * batch * d per scored (query, key)
pair per launch: the two products; sq * sk pairs, or with --causal the pairs
with key <= query) against the tensor roofline. Inputs: seeded N(0,1) bf16.
"""
from __future__ import annotations

import argparse
import json
import os


def measure(batch=128, sq=4096, sk=4096, d=128, cluster=2, steps=10, warmup=3, device=0, cta_group=1, causal=False):
    import numpy as np
    import torch
    from . import gemm, inputs
    dev = torch.device("cuda", device)

    def mk(seed, rows):
        return torch.from_numpy(inputs.bf16_matrix(rows, d, "normal", seed).view(np.int16)).to(dev)

    Q, K, V = mk(0, batch * sq), mk(1, batch * sk), mk(2, batch * sk)
    O = torch.empty(batch * sq * d, dtype=torch.int16, device=dev)
    lse = torch.empty(batch * sq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        assert gemm.attention_forward_run(Q, K, V, O, lse, batch, sq, sk, d, 0.0, 0, cluster, cta_group,
                                          causal=causal, stream=stream) == 0
    st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        st[i].record(stream)
        gemm.attention_forward_run(Q, K, V, O, lse, batch, sq, sk, d, 0.0, 0, cluster, cta_group, causal=causal,
                                   stream=stream)
        en[i].record(stream)
    assert gemm.attention_forward_query_status(stream) == 0
    ms = sum(a.elapsed_time(b) for a, b in zip(st, en)) / steps
    n = min(sq, sk)
    pairs = n * (n + 1) // 2 + max(0, sq - sk) * sk if causal else sq * sk
    flops = 4.0 * batch * pairs * d
    peak = 1893.8
    try:
        with open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except (OSError, ValueError, KeyError):
        pass
    tf = flops / (ms * 1e-3) / 1e12
    return {"kernel": "attention_fwd", "batch": batch, "sq": sq, "sk": sk, "d": d, "cluster": cluster,
            "cta_group": cta_group, "causal": causal, "ms": ms,
            "TFLOPs": tf, "tensor_peak": peak, "frac": tf / peak}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--batch", type=int, default=128)
    ap.add_argument("--sq", type=int, default=4096)
    ap.add_argument("--sk", type=int, default=4096)
    ap.add_argument("--d", type=int, choices=(64, 128), default=128, help="head dimension")
    ap.add_argument("--cluster", type=int, choices=(1, 2, 4), default=None, help="one cluster size (default: all)")
    ap.add_argument("--cta-group", type=int, choices=(1, 2), default=1, help="2: pair MMA (cluster 2)")
    ap.add_argument("--causal", action="store_true", help="query i attends keys 0..i only")
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    args = ap.parse_args(argv)
    if args.cta_group == 2 and (args.d != 128 or args.cluster not in (None, 2)):
        ap.error("the pair MMA (--cta-group 2) needs --d 128 and a 2-CTA cluster")
    configs = [(args.cluster, args.cta_group)] if args.cluster else [(1, 1), (2, 1), (4, 1), (2, 2)]
    if args.d != 128:
        configs = [(c, g) for c, g in configs if g == 1]
    for c, g in configs:
        print(json.dumps(measure(args.batch, args.sq, args.sk, args.d, c, args.steps, args.warmup, cta_group=g,
                                 causal=args.causal)), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
