"""Benchmark of the fused MoE layer on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config large] [--impl ours|reference]

One step = one pass of the whole layer (route -> dispatch -> expert FFN ->
combine) over one batch of synthetic tokens, inputs resident in HBM.  The
default workload is the large prefill layer (T=32768, d=7168, E=256, k=8,
ffn=2048), the largest configuration that fits one GPU; every input is larger
than L2 (22.5 GB of expert weights, 470 MB of tokens), so no L2 flush is
needed between steps.  Smaller configurations (--config) flush L2 between
steps when their inputs fit in it.

Multi-GPU (torchrun): every rank runs an independent replica of the layer on
its own token batch (weak scaling, no data-path collective); the timed region
is bracketed by barriers and the slowest rank's time is reported.

--impl reference times the CPU oracle (the plain, slow restatement of the
layer) on a bounded token sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dispatch_ffn_combine_gb300.workloads import CONFIGS, bf16_bits, make_inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        p["source"] = "measured"
        return p
    p = dict(FALLBACK_PEAKS)
    p["source"] = "fallback"
    return p


def token_seed(rank: int) -> int:
    """Seed of a rank's token batch: rank 0 uses the workload seed (0), so its
    batch is the one the parity tests check; other ranks draw their own."""
    return 0 if rank == 0 else 1000 + rank


def max_over_ranks(value: float, device, dist_on: bool) -> float:
    """Slowest rank's value (all-reduce MAX); the value itself on one rank."""
    if not dist_on:
        return float(value)
    import torch.distributed as tdist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms; the samples whose
    timestamps fall inside the timed region (host clock, marked by begin/end)
    are the ones reported (the nearest one if the region is shorter than the
    interval)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t_begin = None
        self.t_end = None

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"mkmoe_clocks_gpu{self.gpu}_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []  # (time, sm, sm_max, power, reasons)
        with open(self.path) as fh:
            for ln in fh:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    row = (ts, float(parts[2]), float(parts[3]), float(parts[4]),
                           {nm for nm, v in zip(names, parts[6:10]) if v.lower() == "active"})
                except ValueError:
                    continue
                rows.append(row)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = rows
        if self.t_begin is not None and self.t_end is not None:
            inside = [r for r in rows if self.t_begin <= r[0] <= self.t_end]
            if not inside:
                mid = 0.5 * (self.t_begin + self.t_end)
                inside = [min(rows, key=lambda r: abs(r[0] - mid))]
        reasons = set().union(*(r[4] for r in inside))
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max(r[3] for r in inside)}


def launches_per_step(cfg, path) -> int:
    """Kernels one mk_moe_layer call launches.  The kernel-per-step path runs
    route (plain: logits + top-k; with the tensor-core candidate filter, which
    the library picks when T >= 2048, T*d*E >= 2^32 and the token row fits its
    staging: prep + approximate logits + select), count, scan, scatter, gemm1,
    gemm2, combine.  The fused path is one persistent kernel, preceded, where
    the candidate filter applies, by the filter's three kernels, count and scan."""
    import dispatch_ffn_combine_gb300 as mk
    filt = (cfg.T >= 2048 and cfg.T * cfg.d * cfg.E >= 2 ** 32 and 2 * cfg.d + 8 * cfg.E <= 160 * 1024)
    if path == mk.MK_PATH_FUSED:
        return 1 + (5 if filt else 0)
    return (3 if filt else 2) + 6  # the tile-synchronised path launches the same kernels


def flops_bytes(cfg, offsets):
    """Algorithmic work per layer call and per phase."""
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    S = T * k
    counts = np.diff(offsets)
    touched = int(np.count_nonzero(counts))
    w13 = 2 * touched * f * d * 2
    w2 = touched * d * f * 2
    return {
        "gemm1": {"flops": 4 * S * d * f, "bytes": w13 + S * d * 2 + S * f * 2},
        "gemm2": {"flops": 2 * S * d * f, "bytes": w2 + S * f * 2 + S * d * 2},
        "combine": {"flops": 0, "bytes": S * d * 2 + T * d * 2},
        "scatter": {"flops": 0, "bytes": T * d * 2 + S * d * 2},
        "route_logits": {"flops": 2 * T * d * E, "bytes": T * d * 2 + E * d * 4 + T * E * 4},
        "layer": {"flops": 6 * S * d * f, "bytes": w13 + w2 + 2 * T * d * 2 + E * d * 4},
        "touched_experts": touched,
    }


def roofline(work: dict, ms: float, peaks: dict) -> dict:
    """A kernel's algorithmic work per launch (flops, bytes) over its time:
    against the tensor roof when its arithmetic intensity is at or above the
    ridge point, else against the HBM copy rate; `other` is the same kernel
    against the other roof.  The tensor roof is the burst bf16 rate (the
    timed region is under a second, as the burst figure's matmul loop); the
    fraction of the sustained rate (a seconds-long loop under the power cap)
    is given beside it."""
    tensor_peak = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained")
    ridge = tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tfs = work["flops"] / (ms / 1e3) / 1e12
    gbs = work["bytes"] / (ms / 1e3) / 1e9
    t = {"bound": "tensor", "achieved": tfs, "peak": tensor_peak, "unit": "TFLOP/s", "frac": tfs / tensor_peak}
    if sustained:
        t["sustained"] = {"peak": sustained, "frac": tfs / sustained}
    h = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}
    src = peaks.get("source", "")
    if work["flops"] and work["flops"] / max(work["bytes"], 1) >= ridge:
        return dict(t, peak_source=src + " (bf16 burst)", other=h)
    roof = dict(h, peak_source=src + " (HBM copy)")
    if work["flops"]:
        roof["other"] = t
    return roof


def sources_digest(names) -> str:
    """First 16 hex digits of the SHA-256 over the named csrc files, in order."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "dispatch_ffn_combine_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_record(kernel: str, cfg_name: str, path: str | None = None):
    """DRAM bytes per launch from a committed ncu summary, only while every
    source file the kernel is built from is unchanged since the counters were
    taken (else None)."""
    path = path or os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(kernel, {}).get(cfg_name)
    if not rec or "sources" not in rec:
        return None
    if sources_digest(rec["sources"]) != rec["sha256_16"]:
        return None
    return rec["dram_bytes_per_launch"]


def cpu_baseline(cfg, inp_host, budget_s: float, seed: int = 0):
    """Oracle (fp64 FFN, fp32 canonical router) on a token sample, host cores."""
    import oracle

    xb = bf16_bits(inp_host["x"])
    args = (xb, inp_host["wg"].numpy(), None if inp_host["bias"] is None else inp_host["bias"].numpy(),
            bf16_bits(inp_host["w1"]), bf16_bits(inp_host["w3"]), bf16_bits(inp_host["w2"]), cfg.k)
    cores = oracle.num_threads()
    rs = np.random.RandomState(seed)
    # calibrate on one token per core, then size the sample to the budget
    n0 = min(cfg.T, cores)
    t0 = time.perf_counter()
    oracle.layer(*args, tokens=rs.choice(cfg.T, n0, replace=False))
    dt0 = time.perf_counter() - t0
    n = int(min(cfg.T, max(n0, n0 * budget_s / max(dt0, 1e-6))))
    n = max(cores, (n // cores) * cores) if n >= cores else n
    toks = rs.choice(cfg.T, n, replace=False)
    t0 = time.perf_counter()
    oracle.layer(*args, tokens=toks)
    dt = time.perf_counter() - t0
    return n / dt, n, dt, cores


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = CONFIGS[args.config]
    inp = make_inputs(cfg, seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    inp = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
    per_step_s = max(2.0, 150.0 / max(args.steps + args.warmup, 1))
    vals, total_tok, total_t, cores, n = [], 0, 0.0, 1, 0
    for i in range(args.warmup + args.steps):
        tps, n, dt, cores = cpu_baseline(cfg, inp, per_step_s, seed=i)
        if i >= args.warmup:
            vals.append(tps)
            total_tok += n
            total_t += dt
    value = total_tok / total_t
    line = {
        "impl": "reference", "metric": "MoE layer tokens/s (TFLOP/s beside it)", "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / max(args.steps, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.describe(), "sample_tokens_per_step": n},
        "tflops": value * 6 * cfg.k * cfg.d * cfg.f / 1e12,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} random tokens of the workload per step (route + k expert FFNs + "
                                   f"combine, fp64), {args.steps} timed steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_layer(mk, cfg, inp, ws, y, stream, path, mover_ctas, steps, warmup, scrub=None, clocks=None,
               dist=False, dev=None):
    """Warm-up, then `steps` timed layer calls on `stream` (CUDA events).
    With `scrub` (a buffer larger than L2) L2 is flushed before every step and
    only the steps themselves are summed; without it the steps run back to
    back between two events.  Returns (total ms over the steps, per-phase ms
    per step)."""
    x, wg, bias, w1, w3, w2 = (inp[k] for k in ("x", "wg", "bias", "w1", "w3", "w2"))
    nph = len(mk.PHASES)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(steps)]
    for row in ev:  # materialise the event handles before passing them to the library
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()

    def step(i=None):
        mk.mk_moe_layer(x, wg, bias, w1, w3, w2, cfg.k, y=y, ws=ws, phase_events=None if i is None else ev[i],
                        stream=stream, path=path, mover_ctas=mover_ctas)

    for _ in range(warmup):
        if scrub is not None:
            scrub.random_()
        step()
    st, site = mk.mk_moe_last_device_error(ws)
    if st != mk.MK_OK:
        raise RuntimeError(f"device error during warm-up: {mk.status_string(st)} site {site:#x}")
    if clocks is not None:
        clocks.start()
    if dist:
        import torch.distributed as tdist
        tdist.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.begin()
    if scrub is not None:
        for i in range(steps):
            scrub.random_()
            step(i)
        torch.cuda.synchronize()
        total_ms = sum(ev[i][0].elapsed_time(ev[i][nph]) for i in range(steps))
    else:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(steps):
            step(i)
        t_end.record(stream)
        torch.cuda.synchronize()
        total_ms = t_start.elapsed_time(t_end)
    if clocks is not None:
        clocks.end()
    if dist:
        tdist.barrier()
    st, site = mk.mk_moe_last_device_error(ws)
    if st != mk.MK_OK:
        raise RuntimeError(f"device error in the timed region: {mk.status_string(st)} site {site:#x}")
    phase_ms = {}
    if path in (mk.MK_PATH_FUSED, mk.MK_PATH_TILES):  # event 0 before the kernels, the others after them
        phase_ms[PATH_KEYS[path]] = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)) / steps
    else:
        for p, name in enumerate(mk.PHASES):
            phase_ms[name] = sum(ev[i][p].elapsed_time(ev[i][p + 1]) for i in range(steps)) / steps
    return total_ms, phase_ms


PATH_KEYS = {1: "fused_layer", 2: "tiles_layer"}
ALT_ROUNDS, ALT_STEPS = 5, 8  # the alternating comparison of the three paths
# Pinned output buffers of the end-to-end loop (a buffer is reused 2 steps later).  Four measured
# slower: the first downloads into a newly pinned buffer run at ~16 GB/s, and more buffers in
# rotation stalled downloads more often.
E2E_BUFFERS = 2
PATH_NAMES = {0: "one kernel per step", 1: "fused persistent kernel",
              2: "kernel per step, tile semaphores and programmatic dependent launch"}


def time_graph(mk, cfg, inp, ws, y, path, steps, warmup, scrub=None):
    """The layer call captured once into a CUDA graph (after an eager call has
    configured the kernels), then `steps` timed replays under the same rules
    as time_layer.  Returns the total ms over the steps."""
    x, wg, bias, w1, w3, w2 = (inp[k] for k in ("x", "wg", "bias", "w1", "w3", "w2"))
    mk.mk_moe_layer(x, wg, bias, w1, w3, w2, cfg.k, y=y, ws=ws, path=path)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        mk.mk_moe_layer(x, wg, bias, w1, w3, w2, cfg.k, y=y, ws=ws, path=path)
    for _ in range(warmup):
        if scrub is not None:
            scrub.random_()
        g.replay()
    torch.cuda.synchronize()
    total = 0.0
    if scrub is not None:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            scrub.random_()
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        total = sum(a.elapsed_time(b) for a, b in evs)
    else:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        total = a.elapsed_time(b)
    st, site = mk.mk_moe_last_device_error(ws)
    if st != mk.MK_OK:
        raise RuntimeError(f"device error in graph replays: {mk.status_string(st)} site {site:#x}")
    del g
    return total


def dominant_roofline(fb, phase_ms, path, peaks):
    """The roofline object of the step that takes the most time (the whole
    layer on the paths whose steps overlap)."""
    if path in PATH_KEYS:
        dom, work = PATH_KEYS[path], fb["layer"]
    else:
        dom = max(("gemm1", "gemm2", "combine", "scatter", "route_logits"), key=lambda n: phase_ms[n])
        work = fb[dom]
    roof = roofline(work, phase_ms[dom], peaks)
    roof.update({"kernel": dom, "kernel_ms": phase_ms[dom]})
    return roof


def phase_rooflines(fb, phase_ms, peaks):
    """Each step of the kernel-per-step path against its own roof: the two
    GEMMs (tensor), the scatter and the combine (HBM), and the router (its
    kernels together; HBM by its algorithmic intensity, x read once)."""
    out = {}
    for name in ("gemm1", "gemm2", "scatter", "combine"):
        if name in phase_ms:
            out[name] = dict(roofline(fb[name], phase_ms[name], peaks), ms=phase_ms[name])
    if "route_logits" in phase_ms and "topk" in phase_ms:
        ms = phase_ms["route_logits"] + phase_ms["topk"]
        out["route"] = dict(roofline(fb["route_logits"], ms, peaks), ms=ms)
    return out


def needs_flush(inp) -> bool:
    """Inputs that fit twice in L2 are flushed out of it between steps."""
    nbytes = sum(t.numel() * t.element_size() for k, t in inp.items() if t is not None and k != "bias")
    return nbytes < 2 * L2_BYTES


def other_configs(mk, names, dev, stream, steps, warmup, peaks):
    """Each other layer workload timed as the headline (both paths), one at a
    time, its tensors freed before the next: ms/step, tokens/s, TFLOP/s, the
    dominant kernel's roofline and the whole layer against the HBM roof."""
    out = {}
    for name in names:
        cfg = CONFIGS[name]
        inp = make_inputs(cfg, seed=0, device=dev)
        ws = mk.alloc_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, dev)
        y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
        scrub = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if needs_flush(inp) else None
        res = {"workload": cfg.describe(), "l2": "flushed between steps" if scrub is not None else
               "inputs larger than L2 (no flush)", "steps": steps}
        for path, key in ((mk.MK_PATH_STEPS, "steps_path"), (mk.MK_PATH_FUSED, "fused_path"),
                          (mk.MK_PATH_TILES, "tiles_path")):
            total, phase = time_layer(mk, cfg, inp, ws, y, stream, path, 0, steps, warmup, scrub=scrub)
            ms = total / steps
            _, _, offsets, _ = mk.mk_moe_layer_routing(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.f)
            fb = flops_bytes(cfg, offsets.cpu().numpy())
            r = {"ms_per_step": ms, "tokens_per_s": cfg.T / (ms / 1e3),
                 "tflops": fb["layer"]["flops"] / (ms / 1e3) / 1e12,
                 "layer_hbm_frac": fb["layer"]["bytes"] / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                 "roofline": dominant_roofline(fb, phase, path, peaks)}
            if path == mk.MK_PATH_STEPS:
                r["phase_ms"] = phase
                r["phase_roofline"] = phase_rooflines(fb, phase, peaks)
            res[key] = r
        # the kernel-per-step and tile-synchronised calls replayed from a CUDA graph (no host
        # work per call: what a serving loop that captures the layer gets)
        for path, key in ((mk.MK_PATH_STEPS, "steps_path_graph"), (mk.MK_PATH_TILES, "tiles_path_graph")):
            ms = time_graph(mk, cfg, inp, ws, y, path, steps, warmup, scrub=scrub) / steps
            res[key] = {"ms_per_step": ms, "tokens_per_s": cfg.T / (ms / 1e3),
                        "tflops": fb["layer"]["flops"] / (ms / 1e3) / 1e12}
        out[name] = res
        del inp, ws, y, scrub
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import dispatch_ffn_combine_gb300 as mk

    world, rank, local = dist_env()
    dist = world > 1
    if dist:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = CONFIGS[args.config]
    peaks = load_peaks()

    # Weights are shared (seed 0); each rank draws its own token batch.
    inp = make_inputs(cfg, seed=0, device=dev)
    if rank:
        inp["x"] = make_inputs(cfg, seed=token_seed(rank), device=dev, experts=False)["x"]
    x, wg, bias, w1, w3, w2 = (inp[k] for k in ("x", "wg", "bias", "w1", "w3", "w2"))
    ws = mk.alloc_workspace(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, dev)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    flush = needs_flush(inp)
    scrub = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None

    clocks = ClockSampler(local)
    total_ms, phase_ms = time_layer(mk, cfg, inp, ws, y, stream, args.path, args.mover_ctas, args.steps,
                                    args.warmup, scrub=scrub, clocks=clocks, dist=dist, dev=dev)
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, dev, dist)
    ms_per_step = total_ms / args.steps
    value = world * cfg.T / (ms_per_step / 1e3)

    # ---- end to end through the pipelined host-buffer entry point (pinned host x
    # in, y out): each step uploads its x and downloads its y; a step's download
    # runs on the copy engine while the next step computes, and a y buffer is
    # reused only after its event says the previous download into it is done.
    x_host = x.cpu().pin_memory()
    nbuf = E2E_BUFFERS
    y_hosts = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    y_evs = [torch.cuda.Event() for _ in range(nbuf)]

    def e2e_step(i):
        if i >= nbuf:
            y_evs[i % nbuf].synchronize()  # the consumer is done with this buffer's previous output
        mk.mk_moe_layer_host_async(x_host, wg, bias, w1, w3, w2, cfg.k, y_hosts[i % nbuf], ws, y_evs[i % nbuf],
                                   stream=stream, path=args.path, mover_ctas=args.mover_ctas)

    for i in range(max(args.warmup, nbuf + 1)):  # every output buffer has taken a download before timing
        e2e_step(i)
    for ev in y_evs:
        ev.synchronize()
    # the host link's copy rates into and out of these pinned buffers, for the record
    link = {}
    for name, dst, src in (("h2d", y, x_host), ("d2h", y_hosts[0], y)):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        dst.copy_(src, non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        link[name] = src.numel() * src.element_size() / (c0.elapsed_time(c1) / 1e3) / 1e9
    e2e_clocks = ClockSampler(local)
    e2e_clocks.start()
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    step_marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e2e_clocks.begin()
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
        step_marks[i].record(stream)
    stream.wait_event(y_evs[(args.steps - 1) % nbuf])  # the last step's output is in host memory
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_clocks.end()
    e2e_clk = e2e_clocks.stop()
    # per-step intervals on the caller's stream (each step's kernels, after the previous step's)
    step_ms = [e0.elapsed_time(step_marks[0])] + [step_marks[i - 1].elapsed_time(step_marks[i])
                                                    for i in range(1, args.steps)]
    step_med = statistics.median(step_ms)
    te = max_over_ranks(e0.elapsed_time(e1), dev, dist)
    if dist:
        tdist.barrier()
    e2e_value = world * cfg.T / (te / args.steps / 1e3)

    # ---- the other layer paths on the same inputs (device buffers), for comparison
    others = {}
    for other in (mk.MK_PATH_STEPS, mk.MK_PATH_FUSED, mk.MK_PATH_TILES):
        if other == args.path:
            continue
        other_total, other_phase = time_layer(mk, cfg, inp, ws, y, stream, other, 0, args.steps, args.warmup,
                                              scrub=scrub)
        others[other] = (max_over_ranks(other_total, dev, dist) / args.steps, other_phase)

    # ---- the headline path replayed from a CUDA graph (no host work per call)
    graph_ms = max_over_ranks(time_graph(mk, cfg, inp, ws, y, args.path, args.steps, args.warmup, scrub=scrub),
                              dev, dist) / args.steps

    # ---- the three paths once more, alternating in rounds so that no path is
    # measured only at a later (warmer, slower-clocked) time than another
    alt = {o: [] for o in (mk.MK_PATH_STEPS, mk.MK_PATH_FUSED, mk.MK_PATH_TILES)}
    for _ in range(ALT_ROUNDS):
        for o in alt:
            t, _ = time_layer(mk, cfg, inp, ws, y, stream, o, 0, ALT_STEPS, 1, scrub=scrub)
            alt[o].append(max_over_ranks(t, dev, dist) / ALT_STEPS)

    if rank != 0:
        if dist:
            tdist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel
    _, _, offsets, _ = mk.mk_moe_layer_routing(ws, cfg.T, cfg.d, cfg.E, cfg.k, cfg.f)
    fb = flops_bytes(cfg, offsets.cpu().numpy())
    roof = dominant_roofline(fb, phase_ms, args.path, peaks)
    roof["traffic"] = traffic_record(roof["kernel"], args.config)

    # ---- CPU baseline (oracle) on a bounded sample, rank 0 at N=1 only
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        host = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
        tps, n, dt, cores = cpu_baseline(cfg, host, args.cpu_budget)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} random tokens of the workload (route + k expert FFNs + combine in fp64), "
                         f"{dt:.1f} s"}
        del host

    # ---- the other workloads, one at a time (rank 0 at N=1 only)
    configs = None
    if world == 1 and not args.no_configs:
        del inp, x, wg, bias, w1, w3, w2, ws, y, x_host, y_hosts, scrub
        torch.cuda.empty_cache()
        names = [n for n in ("tiny", "mid", "skewed", "decode", "large") if n != args.config]
        configs = other_configs(mk, names, dev, stream, args.config_steps, args.warmup, peaks)

    layer_tflops = fb["layer"]["flops"] / (ms_per_step / 1e3) / 1e12 * world
    line = {
        "metric": "MoE layer tokens/s (TFLOP/s beside it)", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.describe(), "tokens_per_gpu": cfg.T,
                   "l2": "flushed between steps" if flush else "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tflops": layer_tflops,
        "tflops_frac_of_measured_bf16": layer_tflops / world / peaks["bf16_tflops"],
        "phase_ms": phase_ms,
        "phase_roofline": phase_rooflines(fb, phase_ms, peaks) if args.path == mk.MK_PATH_STEPS else None,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": cfg.T * cfg.d * 2,
                "d2h_bytes_per_step": cfg.T * cfg.d * 2, "entry_point": "mk_moe_layer_host_async",
                "note": f"each step's x upload and y download (small copy kernels) overlap other steps' kernels; "
                        f"every upload and download is inside "
                        f"the timed region; {E2E_BUFFERS} pinned output buffers, each reused after its event",
                "clocks": e2e_clk,
                "host_link_gbs": {k: round(v, 1) for k, v in link.items()},
                "median_step_ms": step_med,
                "steps_over_1.5x_median": sum(1 for v in step_ms if v > 1.5 * step_med)},
        "gpu_launches": launches_per_step(cfg, args.path) * args.steps,
        "path": PATH_NAMES[args.path],
        "mover_ctas": args.mover_ctas,
        "other_paths": [{"path": PATH_NAMES[o], "ms_per_step": ms, "value": world * cfg.T / (ms / 1e3),
                         "unit": "tokens/s", "roofline": dominant_roofline(fb, ph, o, peaks)}
                        for o, (ms, ph) in others.items()],
        "other_paths_note": "same inputs and timing rules, measured after the main run; not the headline",
        "graph": {"path": PATH_NAMES[args.path] + ", replayed from a CUDA graph", "ms_per_step": graph_ms,
                  "value": world * cfg.T / (graph_ms / 1e3), "unit": "tokens/s"},
        "paths_alternating": {
            "rounds": ALT_ROUNDS, "steps_per_round": ALT_STEPS,
            "median_ms_per_step": {PATH_NAMES[o]: statistics.median(v) for o, v in alt.items()},
            "note": "each round times the three paths back to back on the same inputs, one warm-up step each"},
        "configs": configs,
        "clocks": clk,
        "peaks": {k: peaks.get(k) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "source")},
    }
    print(json.dumps(line), flush=True)
    if dist:
        tdist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="large", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' entries")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps per path for each other workload")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2],
                    help="0: one kernel per step (default), 1: one persistent kernel, "
                         "2: kernel per step with tile semaphores and programmatic dependent launch")
    ap.add_argument("--mover-ctas", type=int, default=0,
                    help="fused path: 0 adaptive SM split, n > 0 fixed split with n mover blocks, -1 none")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
