"""Run layout -> dispatch -> combine on one seeded workload a few times.

A minimal driver, e.g. for a profiler, that allocates only what the step
needs:

  python -m combine_ep_dispatch_gb300.run_step --workload dsv3 --iters 3

Combine reads the dispatched rows (identity experts; for the FP8 workload a
bf16 dispatch of the same routing provides them).  --order expert runs the
expert-major path (one row per (token, expert) pair, combine weighted by the
gate weights); --fused uses the one-launch layout + dispatch (rank order,
bf16, small batches); --with-layout uses the single layout + dispatch call
(rank order); --cast-transpose adds the FP8 cast and transposed cast of the
received rows (expert order); --regions dispatches into and combines from
per-rank regions, one allocation per rank (rank order, after the layout).
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import _lib
from .inputs import CONFIGS, make_inputs
from .pipeline import DispatchCombine


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="dsv3", choices=sorted(CONFIGS))
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--order", default="rank", choices=("rank", "expert"))
    ap.add_argument("--fused", action="store_true")
    ap.add_argument("--with-layout", action="store_true")
    ap.add_argument("--cast-transpose", action="store_true")
    ap.add_argument("--regions", action="store_true")
    args = ap.parse_args(argv)

    inp = make_inputs(args.workload, seed=args.seed)
    cfg = inp["cfg"]
    dev = torch.device("cuda")
    x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(inp["topk_idx"]).to(dev)
    w = torch.from_numpy(inp["topk_w"]).to(dev)
    quant = _lib.EP_QUANT_FP8_E4M3_B128 if cfg.quant == "fp8" else _lib.EP_QUANT_BF16
    order = args.order
    probe = DispatchCombine(cfg.T, 8, cfg.E, cfg.k, cfg.W, capacity_rows=0, device=dev,
                            order=order)
    probe.layout(idx)
    R = int(probe.rank_offset[cfg.W].item() if order == "rank" else
            probe.expert_offset[cfg.E].item())
    dc = DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W, capacity_rows=R, quant=quant,
                         device=dev, order=order)
    ident = dc if quant == _lib.EP_QUANT_BF16 else DispatchCombine(
        cfg.T, cfg.H, cfg.E, cfg.k, cfg.W, capacity_rows=R, device=dev, order=order)
    weights = w if order == "expert" else None
    scale = torch.full((cfg.E,), 112.0, dtype=torch.float32, device=dev)
    if args.regions:
        if order != "rank":
            raise SystemExit("--regions takes the rank-major layout")
        regions, y_regions = [], []
        dc.layout(idx)
        ident.layout(idx)
        ident.dispatch(x, idx, w)
        torch.cuda.synchronize()
        off = [int(v) for v in dc.rank_offset.cpu()]
        fp8 = quant != _lib.EP_QUANT_BF16
        for r in range(cfg.W):
            n = off[r + 1] - off[r]
            regions.append({
                "recv_x": torch.empty(n, cfg.H, dtype=torch.uint8 if fp8 else torch.bfloat16,
                                      device=dev),
                "recv_scale": (torch.empty(n, cfg.H // 128, dtype=torch.float32, device=dev)
                               if fp8 else None),
                "recv_topk_idx": torch.empty(n, cfg.k, dtype=torch.int32, device=dev),
                "recv_topk_w": torch.empty(n, cfg.k, dtype=torch.float32, device=dev),
                "recv_src": torch.empty(n, dtype=torch.int32, device=dev)})
            y_regions.append(ident.recv_x[off[r]:off[r + 1]].clone())
        for _ in range(args.iters):
            dc.layout(idx)
            _lib.ep_dispatch_regions(x, idx, w, dc.slot, dc.rank_offset, regions, quant,
                                     dc.status)
            _lib.ep_combine_regions(y_regions, dc.slot, dc.rank_offset, dc.out, dc.status)
        torch.cuda.synchronize()
        print(f"{args.workload} (rank, per-rank regions): T={cfg.T} H={cfg.H} E={cfg.E} k={cfg.k} "
              f"W={cfg.W} R={R} iters={args.iters} status={int(dc.status.item())}")
        return
    for _ in range(args.iters):
        if args.fused:
            dc.dispatch_fused(x, idx, w)
        elif args.with_layout:
            dc.layout_dispatch(x, idx, w)
        else:
            dc.layout(idx)
            dc.dispatch(x, idx, w)
        if ident is not dc:
            ident.layout(idx)
            ident.dispatch(x, idx, w)
        if args.cast_transpose:
            ident.cast_transpose(scale)
        dc.combine(ident.recv_x, weights)
    torch.cuda.synchronize()
    mode = ", fused" if args.fused else (", with layout" if args.with_layout else "")
    print(f"{args.workload} ({order}{mode}): T={cfg.T} H={cfg.H} E={cfg.E} k={cfg.k} W={cfg.W} R={R} "
          f"iters={args.iters} status={int(dc.status.item())}")


if __name__ == "__main__":
    main()
