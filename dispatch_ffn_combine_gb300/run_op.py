"""Run one public entry point of the library on a named synthetic workload.

    python -m dispatch_ffn_combine_gb300.run_op --op route --config large --warmup 3 --calls 1

The inputs of the chosen call are prepared by the earlier entry points (route,
then dispatch, then the expert FFN), outside the timed calls; then the call runs
``--warmup`` times untimed and ``--calls`` times bracketed by CUDA events on one
stream.  Prints one JSON line with the mean milliseconds per call.  This is the
driver for profiling a single step of the layer (ncu ``-k`` on the step's
kernel); ``bench.py`` is the one that times the whole layer.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import (MK_PATH_FUSED, MK_PATH_STEPS, alloc_dispatch_gemm_workspace, alloc_workspace, mk_moe_combine,
               mk_moe_dispatch, mk_moe_dispatch_gemm, mk_moe_expert_ffn, mk_moe_layer, mk_moe_route)
from .workloads import CONFIGS, make_inputs

OPS = ("route", "dispatch", "expert_ffn", "combine", "layer", "dispatch_gemm")


def main(argv=None) -> dict:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--op", choices=OPS, required=True)
    ap.add_argument("--config", choices=sorted(CONFIGS), default="large")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's token count")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--calls", type=int, default=1)
    ap.add_argument("--path", choices=("steps", "fused"), default="steps", help="layer path (op=layer)")
    args = ap.parse_args(argv)

    cfg = CONFIGS[args.config]
    dev = torch.device("cuda")
    need_experts = args.op in ("expert_ffn", "combine", "layer", "dispatch_gemm")
    inp = make_inputs(cfg, seed=0, device=dev, T=args.tokens, experts=need_experts)
    x, wg, bias = inp["x"], inp["wg"], inp["bias"]
    T, d = x.shape
    E, k, f = cfg.E, cfg.k, cfg.f
    ws = alloc_workspace(T, d, E, k, f, dev)
    path = MK_PATH_STEPS if args.path == "steps" else MK_PATH_FUSED

    dg_ws = alloc_dispatch_gemm_workspace(T, d, E, k, dev) if args.op == "dispatch_gemm" else None
    ids, w, _ = mk_moe_route(x, wg, bias, k, ws=ws)
    disp = mk_moe_dispatch(x, ids, w, E, ws=ws) if args.op in ("expert_ffn", "combine") else None
    h = P = None
    if args.op == "combine":
        h, P = mk_moe_expert_ffn(disp["x_perm"], disp["expert_offsets"], disp["row_weight"], inp["w1"], inp["w3"],
                                 inp["w2"], ws=ws)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)

    def call():
        if args.op == "route":
            mk_moe_route(x, wg, bias, k, topk_ids=ids, topk_w=w, ws=ws)
        elif args.op == "dispatch":
            mk_moe_dispatch(x, ids, w, E, ws=ws)
        elif args.op == "expert_ffn":
            mk_moe_expert_ffn(disp["x_perm"], disp["expert_offsets"], disp["row_weight"], inp["w1"], inp["w3"],
                              inp["w2"], ws=ws)
        elif args.op == "combine":
            mk_moe_combine(P, disp["slot_row"], y=y)
        elif args.op == "dispatch_gemm":  # the layer's gate projection W1 as the experts' weight
            mk_moe_dispatch_gemm(x, wg, bias, inp["w1"], k, ws=dg_ws)
        else:
            mk_moe_layer(x, wg, bias, inp["w1"], inp["w3"], inp["w2"], k, y=y, ws=ws, path=path)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.calls):
        call()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / max(args.calls, 1)
    out = {"op": args.op, "config": cfg.name, "T": T, "calls": args.calls, "ms_per_call": ms}
    if args.op == "layer":
        out["path"] = args.path
    print(json.dumps(out))
    return out


if __name__ == "__main__":
    main()
