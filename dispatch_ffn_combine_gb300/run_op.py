"""Run one public entry point of the library on a named synthetic workload.

    python -m dispatch_ffn_combine_gb300.run_op --op route --config large --warmup 3 --calls 1

The inputs of the chosen call are prepared by the earlier entry points (route,
then dispatch, then the expert FFN), outside the timed calls; then the call runs
``--warmup`` times untimed and ``--calls`` times bracketed by CUDA events on one
stream.  Prints one JSON line with the mean milliseconds per call.  This is the
driver for profiling a single step of the layer (ncu ``-k`` on the step's
kernel); ``bench.py`` is the one that times the whole layer.

With ``--op layer --path fused --trace`` one more call records the persistent
kernel's task trace, and a summary follows the JSON line: per task kind its
count, span and mean duration, the GEMM tiles' mean time, and the number of
blocks busy in each kind per time window.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import (MK_PATH_FUSED, MK_PATH_STEPS, MK_PATH_TILES, TRACE_KINDS, alloc_dispatch_gemm_workspace, alloc_workspace,
               mk_moe_combine, mk_moe_dispatch, mk_moe_dispatch_gemm, mk_moe_expert_ffn, mk_moe_layer,
               mk_moe_layer_trace_count, mk_moe_route)
from .workloads import CONFIGS, make_inputs

OPS = ("route", "dispatch", "expert_ffn", "combine", "layer", "dispatch_gemm")


def trace_summary(tr, n: int, windows: int = 20) -> list:
    """Text lines describing one fused call's task records (see mk_moe_opts.trace)."""
    import numpy as np

    t = tr[: min(n, tr.shape[0])].cpu().numpy().astype(np.int64)
    if len(t) == 0:
        return ["no task records"]
    start = (t[:, 4] & 0xFFFFFFFF) | (t[:, 5] << 32)
    end = (t[:, 6] & 0xFFFFFFFF) | (t[:, 7] << 32)
    t0 = start.min()
    st, en = (start - t0) / 1e3, (end - t0) / 1e3  # microseconds from the first task
    tiles = t[:, 3] & 0x7FFFFFFF
    span = float(en.max())
    lines = [f"records {len(t)}, span {span:.1f} us"]
    for kind in sorted(set(t[:, 1].tolist())):
        m = t[:, 1] == kind
        name = TRACE_KINDS.get(int(kind), str(kind))
        line = (f"  {name:8s} tasks {int(m.sum()):6d}  first start {st[m].min():9.1f} us  last end {en[m].max():9.1f} us"
                f"  mean {float((en[m] - st[m]).mean()):9.1f} us")
        if tiles[m].sum() > 0:
            line += f"  tiles {int(tiles[m].sum())}, {float((en[m] - st[m]).sum() / tiles[m].sum()):.1f} us per tile"
        lines.append(line)
    kinds = sorted(set(t[:, 1].tolist()))
    w = span / windows
    occ = np.zeros((windows, len(kinds)))
    for i in range(len(t)):
        a, b = st[i], en[i]
        for j in range(int(a // w), min(int(b // w), windows - 1) + 1):
            lo, hi = max(a, j * w), min(b, (j + 1) * w)
            if hi > lo:
                occ[j, kinds.index(t[i, 1])] += (hi - lo) / w
    lines.append("  window start (us)  " + "  ".join(f"{TRACE_KINDS.get(int(k), str(k)):>8s}" for k in kinds)
                 + "   (blocks busy)")
    for j in range(windows):
        lines.append(f"  {j * w:17.0f}  " + "  ".join(f"{occ[j, c]:8.1f}" for c in range(len(kinds))))
    return lines


def main(argv=None) -> dict:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--op", choices=OPS, required=True)
    ap.add_argument("--config", choices=sorted(CONFIGS), default="large")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's token count")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--calls", type=int, default=1)
    ap.add_argument("--path", choices=("steps", "fused", "tiles"), default="steps", help="layer path (op=layer)")
    ap.add_argument("--trace", action="store_true", help="op=layer, path=fused: summarise one traced call")
    args = ap.parse_args(argv)
    if args.trace and (args.op != "layer" or args.path != "fused"):
        ap.error("--trace needs --op layer --path fused")

    cfg = CONFIGS[args.config]
    dev = torch.device("cuda")
    need_experts = args.op in ("expert_ffn", "combine", "layer", "dispatch_gemm")
    inp = make_inputs(cfg, seed=0, device=dev, T=args.tokens, experts=need_experts)
    x, wg, bias = inp["x"], inp["wg"], inp["bias"]
    T, d = x.shape
    E, k, f = cfg.E, cfg.k, cfg.f
    ws = alloc_workspace(T, d, E, k, f, dev)
    path = {"steps": MK_PATH_STEPS, "fused": MK_PATH_FUSED, "tiles": MK_PATH_TILES}[args.path]

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
    if args.trace:
        tr = torch.zeros((1 << 18, 8), dtype=torch.int32, device=dev)
        mk_moe_layer(x, wg, bias, inp["w1"], inp["w3"], inp["w2"], k, y=y, ws=ws, path=path, trace=tr)
        n = mk_moe_layer_trace_count(ws, T, d, E, k, f)
        print("\n".join(trace_summary(tr, n)))
    return out


if __name__ == "__main__":
    main()
