"""Token-count sweep of MoE Dispatch + GEMM and of the whole layer.

    python -m dispatch_ffn_combine_gb300.sweep --tokens 8192,16384,32768,65536,131072

The paper's section 5.3 measures its Dispatch + GEMM kernel at 8K to 128K
total tokens (throughput in TFLOP/s per GPU, Figures 3-6).  This runs the same
token counts on one GPU with the large layer's dimensions (d = 7168, E = 256,
k = 8) and, as the Dispatch + GEMM weight, the layer's gate projection W1
[E, 2048, d]; the layer itself runs beside it on the same tokens.  Inputs are
seeded and synthetic (the layer's recipe); the token rows of a smaller count
are the first rows of the largest.  Every call is timed alone with CUDA events
on its stream, after an L2 flush (a 256 MiB write) outside the timed span; the
median of the timed calls is reported.  One JSON line per token count.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import (alloc_dispatch_gemm_workspace, alloc_workspace, mk_moe_dispatch_gemm, mk_moe_last_device_error,
               mk_moe_layer, MK_OK)
from .workloads import CONFIGS, make_inputs


def _time(fn, calls: int, warmup: int, flush: torch.Tensor) -> float:
    for _ in range(warmup):
        fn()
    times = []
    for _ in range(calls):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def main(argv=None) -> list:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--tokens", default="8192,16384,32768,65536,131072")
    ap.add_argument("--calls", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--no-layer", action="store_true", help="time only Dispatch + GEMM")
    args = ap.parse_args(argv)

    sizes = sorted(int(t) for t in args.tokens.split(","))
    cfg = CONFIGS["large"]
    dev = torch.device("cuda")
    inp = make_inputs(cfg, seed=0, device=dev, T=sizes[-1], experts=True)
    d, E, k, f = cfg.d, cfg.E, cfg.k, cfg.f
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    lines = []
    for T in sizes:
        x = inp["x"][:T]
        ws = alloc_dispatch_gemm_workspace(T, d, E, k, dev)
        out = {"out": torch.empty((T * k, f), dtype=torch.bfloat16, device=dev),
               "expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
               "row_token": torch.empty(T * k, dtype=torch.int32, device=dev),
               "row_weight": torch.empty(T * k, dtype=torch.float32, device=dev)}

        def dg():
            mk_moe_dispatch_gemm(x, inp["wg"], inp["bias"], inp["w1"], k, out=out, ws=ws)

        ms = _time(dg, args.calls, args.warmup, flush)
        assert mk_moe_last_device_error(ws)[0] == MK_OK
        flops = 2.0 * T * k * d * f
        rec = {"op": "dispatch_gemm", "T": T, "d": d, "E": E, "k": k, "n": f, "ms": ms,
               "tflops": flops / ms / 1e9, "tokens_per_s": T / ms * 1e3}
        del ws, out
        if not args.no_layer:
            lws = alloc_workspace(T, d, E, k, f, dev)
            y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)

            def layer():
                mk_moe_layer(x, inp["wg"], inp["bias"], inp["w1"], inp["w3"], inp["w2"], k, y=y, ws=lws)

            lms = _time(layer, args.calls, args.warmup, flush)
            assert mk_moe_last_device_error(lws)[0] == MK_OK
            rec.update({"layer_ms": lms, "layer_tflops": 3 * flops / lms / 1e9, "layer_tokens_per_s": T / lms * 1e3})
            del lws, y
        torch.cuda.empty_cache()
        print(json.dumps(rec), flush=True)
        lines.append(rec)
    return lines


if __name__ == "__main__":
    main()
