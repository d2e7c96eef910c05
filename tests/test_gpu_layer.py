"""GPU parity of the whole layer (mk_moe_layer) against the CPU oracle.

Small shapes are checked on every token; the full-size workloads run in the
launch configuration the benchmark times, with routing and dispatch checked on
every token (bit-exact) and the output on a fixed token sample."""
import gc

import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
import oracle
from _support import Workload, check_output, sample_tokens

pytestmark = pytest.mark.gpu


def _run_layer(wl, **kw):
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    y = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, ws=ws, **kw)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_OK, (st, hex(site))
    return y, ws


def _check_routing(wl, ws, ids_ref, w_ref):
    c = wl.cfg
    ids, w, offsets, slot = mk.mk_moe_layer_routing(ws, wl.T, c.d, c.E, c.k, c.f)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=1e-7)
    _, off_ref, _, slot_ref = oracle.dispatch(ids_ref, c.E)
    np.testing.assert_array_equal(offsets.cpu().numpy(), off_ref)
    np.testing.assert_array_equal(slot.cpu().numpy(), slot_ref)


@pytest.mark.parametrize("name", ["tiny", "ragged", "ragged_skew", "single", "ragged_pair", "edge_min", "many_experts"])
def test_layer_small_all_tokens(name):
    wl = Workload(name)
    y, ws = _run_layer(wl)
    y_ref, ids_ref, w_ref = wl.oracle_layer()
    _check_routing(wl, ws, ids_ref, w_ref)
    check_output(y.cpu(), y_ref, name)


@pytest.mark.parametrize("T", [1, 2, 129])
def test_layer_few_tokens(T):
    wl = Workload("ragged", T=T)
    y, ws = _run_layer(wl)
    y_ref, ids_ref, w_ref = wl.oracle_layer()
    _check_routing(wl, ws, ids_ref, w_ref)
    check_output(y.cpu(), y_ref, f"ragged T={T}")


def test_layer_zero_tokens_is_noop():
    wl = Workload("tiny", T=0)
    c = wl.cfg
    ws = mk.alloc_workspace(0, c.d, c.E, c.k, c.f, wl.dev)
    y = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, ws=ws)
    assert y.shape == (0, c.d)


def test_layer_mid_sampled():
    wl = Workload("mid")
    y, ws = _run_layer(wl)
    _, ids_ref, w_ref = wl.oracle_routing()
    _check_routing(wl, ws, ids_ref, w_ref)
    toks = sample_tokens(wl.T, 256)
    y_ref, _, _ = wl.oracle_layer(tokens=toks)
    check_output(y.cpu()[torch.from_numpy(toks)], y_ref, "mid")


def test_layer_deterministic():
    wl = Workload("ragged_skew")
    y1, ws = _run_layer(wl)
    y2, _ = _run_layer(wl)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_layer_host_buffers_match_device_call():
    wl = Workload("ragged")
    c = wl.cfg
    y_dev, ws = _run_layer(wl)
    x_host = wl.g["x"].cpu().pin_memory()
    y_host = torch.empty((wl.T, c.d), dtype=torch.bfloat16).pin_memory()
    mk.mk_moe_layer_host(x_host, wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, y_host, ws)
    torch.cuda.synchronize()
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))


@pytest.mark.parametrize("T", [7, 1000])
def test_layer_host_calls_back_to_back(T):
    """Host-buffer calls issued back to back on one workspace (their copies
    overlap the previous call's kernels), alternating paths, inputs and
    pinned / pageable inputs and outputs: every y_host equals the
    device-buffer result for its own input."""
    wl = Workload("ragged", T=T)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    g = torch.Generator().manual_seed(7)
    xs = [wl.g["x"].cpu()] + [torch.randn((wl.T, c.d), generator=g).to(torch.bfloat16) for _ in range(3)]
    # pinned inputs take the upload kernel, the pageable one (call 1) the copy engine
    xs_host = [x.clone() if i == 1 else x.pin_memory() for i, x in enumerate(xs)]
    # pinned outputs take the direct write, pageable ones the chunked downloads
    ys_host = [torch.empty((wl.T, c.d), dtype=torch.bfloat16) for _ in xs]
    ys_host = [y.pin_memory() if i % 2 == 0 else y for i, y in enumerate(ys_host)]
    paths = [mk.MK_PATH_STEPS, mk.MK_PATH_STEPS, mk.MK_PATH_FUSED, mk.MK_PATH_STEPS]
    args = (wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    for xh, yh, path in zip(xs_host, ys_host, paths):
        mk.mk_moe_layer_host(xh, *args, yh, ws, path=path)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    ws2 = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    for x, yh in zip(xs, ys_host):
        y_dev = mk.mk_moe_layer(x.to(wl.dev), *args, ws=ws2)
        torch.cuda.synchronize()
        assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))


def test_layer_host_calls_gathering_rows_back_to_back():
    """With gemm1 gathering its rows from the staged x (gather_rows), back-to-back
    host-buffer calls (blocking and pipelined, pinned inputs uploaded beside the
    previous call's kernels) keep each call's x until its gemm1 has read it:
    every y_host equals the device-buffer result for its own input."""
    wl = Workload("ragged", T=1000)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    g = torch.Generator().manual_seed(13)
    xs = [torch.randn((wl.T, c.d), generator=g).to(torch.bfloat16) for _ in range(4)]
    xs_host = [x.pin_memory() for x in xs]
    ys_host = [torch.full((wl.T, c.d), -1.0, dtype=torch.bfloat16).pin_memory() for _ in xs]
    args = (wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    events = []
    for i, (xh, yh) in enumerate(zip(xs_host, ys_host)):
        if i % 2 == 0:
            ev = torch.cuda.Event()
            mk.mk_moe_layer_host_async(xh, *args, yh, ws, ev, gather_rows=True)
            events.append(ev)
        else:
            mk.mk_moe_layer_host(xh, *args, yh, ws, gather_rows=True)
    for ev in events:
        ev.synchronize()
    torch.cuda.synchronize()
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    ws2 = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    for x, yh in zip(xs, ys_host):
        y_dev = mk.mk_moe_layer(x.to(wl.dev), *args, ws=ws2)
        torch.cuda.synchronize()
        assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))


def test_layer_host_async_more_workspaces_than_pipes():
    """Pipelined host-buffer calls rotating over more workspaces than the
    library keeps copy pipes for (each workspace's pipe is evicted and made
    again while its last call may still run), without synchronising between
    calls: every y_host equals the device-buffer result for its own input."""
    wl = Workload("ragged", T=256)
    c = wl.cfg
    n_ws = 10  # more than the library's pipe cache
    wss = [mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev) for _ in range(n_ws)]
    g = torch.Generator().manual_seed(17)
    xs = [torch.randn((wl.T, c.d), generator=g).to(torch.bfloat16) for _ in range(2 * n_ws)]
    xs_host = [x.pin_memory() for x in xs]
    ys_host = [torch.full((wl.T, c.d), -1.0, dtype=torch.bfloat16).pin_memory() for _ in xs]
    args = (wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    events = []
    for i, (xh, yh) in enumerate(zip(xs_host, ys_host)):
        ev = torch.cuda.Event()
        mk.mk_moe_layer_host_async(xh, *args, yh, wss[i % n_ws], ev)
        events.append(ev)
    for ev in events:
        ev.synchronize()
    torch.cuda.synchronize()
    for ws in wss:
        assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    ws2 = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    for x, yh in zip(xs, ys_host):
        y_dev = mk.mk_moe_layer(x.to(wl.dev), *args, ws=ws2)
        torch.cuda.synchronize()
        assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))


@pytest.mark.parametrize("T", [7, 1000])
def test_layer_host_async_back_to_back(T):
    """The pipelined host entry point issued back to back on one workspace,
    interleaved with the blocking one and the fused path, each output its
    own y_host and event, one input pageable: once its event has completed,
    every y_host equals the device-buffer result for its own input; the
    stream never waited for the downloads of the async calls."""
    wl = Workload("ragged", T=T)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    g = torch.Generator().manual_seed(11)
    xs = [wl.g["x"].cpu()] + [torch.randn((wl.T, c.d), generator=g).to(torch.bfloat16) for _ in range(4)]
    # pinned inputs take the upload kernel, the pageable one (call 1) the copy engine
    xs_host = [x.clone() if i == 1 else x.pin_memory() for i, x in enumerate(xs)]
    # pinned outputs, and one pageable one (its download still completes before the event)
    ys_host = [torch.full((wl.T, c.d), -1.0, dtype=torch.bfloat16) for _ in xs]
    ys_host = [y if i == 4 else y.pin_memory() for i, y in enumerate(ys_host)]
    kinds = ["async", "async", "blocking", "async_fused", "async"]
    args = (wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    events = []
    for xh, yh, kind in zip(xs_host, ys_host, kinds):
        if kind == "blocking":
            mk.mk_moe_layer_host(xh, *args, yh, ws)
            events.append(None)
        else:
            ev = torch.cuda.Event()
            path = mk.MK_PATH_FUSED if kind == "async_fused" else mk.MK_PATH_STEPS
            mk.mk_moe_layer_host_async(xh, *args, yh, ws, ev, path=path)
            events.append(ev)
    for ev in events:
        if ev is not None:
            ev.synchronize()
    torch.cuda.synchronize()
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    ws2 = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    for x, yh in zip(xs, ys_host):
        y_dev = mk.mk_moe_layer(x.to(wl.dev), *args, ws=ws2)
        torch.cuda.synchronize()
        assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))


def test_layer_host_async_needs_an_event():
    wl = Workload("tiny")
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    x_host = wl.g["x"].cpu().pin_memory()
    y_host = torch.empty((wl.T, c.d), dtype=torch.bfloat16).pin_memory()
    lib = mk.load_library()
    import ctypes
    st = lib.mk_moe_layer_host_async(mk._p(x_host), mk._p(wl.g["wg"]), None, mk._p(wl.g["w1"]), mk._p(wl.g["w3"]),
                                     mk._p(wl.g["w2"]), wl.T, c.d, c.E, c.k, c.f, mk._p(y_host), mk._p(ws),
                                     ws.numel(), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), None)
    assert st == mk.MK_ERR_INVALID_ARG


def test_layer_route_fallback_path_is_exact():
    """With the candidate filter's bound forced to zero, (almost) every token
    takes the exact fallback (all E logits in the fixed order): the layer's
    output is bit-identical to the normal call."""
    wl = Workload("ragged_skew")
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    args = (wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    y0 = mk.mk_moe_layer(*args, ws=ws).clone()
    assert mk.mk_moe_route_fallbacks(ws) == 0
    y1 = mk.mk_moe_layer(*args, ws=ws, inject=mk.MK_INJECT_ROUTE_ZERO_BOUND)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    assert mk.mk_moe_route_fallbacks(ws) > wl.T // 2
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("name", ["ragged", "ragged_pair"])
def test_layer_bounded_wait_times_out_cleanly(name):
    """A grouped-GEMM stage that is announced but never filled: the waits on it
    run out after the given limit, the call reports MK_ERR_TIMEOUT, nothing
    faults or hangs, and the next call on the same context is correct."""
    wl = Workload(name)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    args = (wl.g["x"], wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    mk.mk_moe_layer(*args, ws=ws, inject=mk.MK_INJECT_STALL_GEMM1, timeout_ns=20_000_000)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_ERR_TIMEOUT, (st, hex(site))
    y = mk.mk_moe_layer(*args, ws=ws)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    y_ref, _, _ = wl.oracle_layer()
    check_output(y.cpu(), y_ref, "after timeout")


def _check_experts_every_row(wl, ws, name):
    """Every row of a few experts of the layer just run, through the oracle's
    per-expert FFN: P[r] = row_weight[r] * FFN_e(x[row_token[r]]).  The experts
    are the one with the most rows, the one with the fewest, and the ones whose
    last 256-row block is the shortest and the longest short of a full block,
    so the CTA-pair GEMMs' swap tiles (an expert's partial last block) and the
    tile tables at full size are covered.  Returns the experts checked."""
    c = wl.cfg
    view = lambda r: mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, r)
    offsets = view("offsets").cpu().numpy().astype(np.int64)
    row_token = view("row_token").cpu().numpy().astype(np.int64)
    row_weight = view("row_weight").cpu().numpy().astype(np.float64)
    counts = np.diff(offsets)
    live = np.nonzero(counts)[0]
    tail = counts % 256
    has_tail = live[tail[live] > 0]
    picks = [int(live[np.argmax(counts[live])]), int(live[np.argmin(counts[live])])]
    if has_tail.size:
        picks += [int(has_tail[np.argmin(tail[has_tail])]), int(has_tail[np.argmax(tail[has_tail])])]
    picks = sorted(set(picks))
    P = view("P")
    for e in picks:
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        toks = row_token[r0:r1]
        ref = oracle.expert_ffn(wl.bits("x"), wl.bits("w1"), wl.bits("w3"), wl.bits("w2"), toks,
                                np.full(toks.size, e, dtype=np.int64))
        ref = ref * row_weight[r0:r1, None]
        check_output(P[r0:r1].cpu(), ref, f"{name} expert {e} ({r1 - r0} rows, tail {tail[e]})")
    return picks, counts


def chunk_spread_tokens(T, n, seed=0):
    """The first, middle and last 128-token chunks whole, plus a seeded random
    spread of the other tokens: n tokens in all (n >= 384)."""
    chunks = [np.arange(0, 128), np.arange(T // 2 - 64, T // 2 + 64), np.arange(T - 128, T)]
    fixed = np.unique(np.concatenate(chunks))
    rest = np.setdiff1d(np.arange(T), fixed)
    rs = np.random.RandomState(seed)
    extra = rs.choice(rest, size=max(0, n - fixed.size), replace=False)
    return np.sort(np.concatenate([fixed, extra])).astype(np.int64)


@pytest.mark.parametrize("name,n_sample", [("skewed", 512), ("decode", 128), ("large", 1024)])
def test_layer_full_size(name, n_sample):
    """Full-size workload in the benchmark's launch configuration: routing and
    dispatch tables of every token bit-exact, the dispatched rows bitwise
    copies of their tokens, every row of a few experts through the oracle's
    expert FFN, and the output on a token sample that covers the first,
    middle and last chunks."""
    wl = Workload(name)
    c = wl.cfg
    y, ws = _run_layer(wl)
    _, ids_ref, w_ref = wl.oracle_routing()
    _check_routing(wl, ws, ids_ref, w_ref)
    _, _, row_token_ref, _ = oracle.dispatch(ids_ref, c.E)
    row_token = mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "row_token")
    np.testing.assert_array_equal(row_token.cpu().numpy(), row_token_ref)
    xp = mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "x_perm").view(torch.int16)
    rt = torch.from_numpy(row_token_ref.astype(np.int64)).to(wl.dev)
    for r0 in range(0, rt.numel(), 1 << 16):
        assert torch.equal(xp[r0:r0 + (1 << 16)], wl.g["x"].view(torch.int16).index_select(0, rt[r0:r0 + (1 << 16)]))
    _check_experts_every_row(wl, ws, name)
    toks = chunk_spread_tokens(wl.T, n_sample) if wl.T > 384 else np.arange(wl.T, dtype=np.int64)
    y_ref, _, _ = wl.oracle_layer(tokens=toks)
    check_output(y.cpu()[torch.from_numpy(toks)], y_ref, name)
    # the persistent-kernel path on the same workspace: the same bits
    y_f = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], wl.cfg.k, ws=ws,
                          path=mk.MK_PATH_FUSED)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    assert torch.equal(y_f.view(torch.int16), y.view(torch.int16))
    del wl, y, y_f, ws, xp, rt
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["ragged", "ragged_pair", "many_experts", "mid", "large"])
def test_layer_gemm1_gathering_from_x_is_bitwise(name):
    """gemm1 reading its rows straight from x by their source tokens (TMA
    gather4, no dispatched copy of x) gives the same h, P and y bits as the
    kernel-per-step path: the MMA sees the same rows."""
    wl = Workload(name)
    c = wl.cfg
    y, ws = _run_layer(wl)
    h = mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "h").clone()
    y_g = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, ws=ws,
                          gather_rows=True)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    assert torch.equal(mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "h").view(torch.int16), h.view(torch.int16))
    assert torch.equal(y_g.view(torch.int16), y.view(torch.int16))
    del wl, ws, y, y_g, h
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", ["steps", "tiles", "fused"])
def test_layer_replays_from_a_cuda_graph(path):
    """The layer call captured into a CUDA graph (after one eager call on the
    workspace has configured the kernels) and replayed twice, with new input
    values copied in between: every replay is bit-identical to an eager call
    on the same input.  The library allocates nothing per call, so the graph
    holds only its memsets and kernel launches."""
    wl = Workload("ragged_skew")
    c = wl.cfg
    p = {"steps": mk.MK_PATH_STEPS, "tiles": mk.MK_PATH_TILES, "fused": mk.MK_PATH_FUSED}[path]
    args = (wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    x = wl.g["x"].clone()
    y = torch.empty((wl.T, c.d), dtype=torch.bfloat16, device=wl.dev)
    mk.mk_moe_layer(x, *args, y=y, ws=ws, path=p)  # configures the kernels outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        mk.mk_moe_layer(x, *args, y=y, ws=ws, path=p)
    gen = torch.Generator(device="cpu").manual_seed(5)
    ws2 = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    for _ in range(2):
        x.copy_(torch.randn((wl.T, c.d), generator=gen).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
        y_ref = mk.mk_moe_layer(x, *args, ws=ws2, path=mk.MK_PATH_STEPS)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
