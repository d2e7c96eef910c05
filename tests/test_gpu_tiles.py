"""GPU parity of the tile-synchronised path (MK_PATH_TILES): one kernel per
step, each launched as a programmatic dependent of the one before, the
dispatch, both GEMMs and the combine synchronised per 128-row M-tile by
data-tile semaphores (the MegaOps page's kernel-per-operator design, with
in/out semaphores on data tiles).

Its arithmetic is the kernel-per-step path's, so its output must equal that
path's bit for bit, and the oracle within the layer tolerance; a dropped tile
signal must end in MK_ERR_TIMEOUT from bounded waits, with the next call
correct."""
import gc

import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
from _support import Workload, check_output

pytestmark = pytest.mark.gpu


def _layer(wl, ws, path, **kw):
    c = wl.cfg
    y = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, ws=ws,
                        path=path, **kw)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_OK, (st, hex(site))
    return y


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("name", ["tiny", "ragged", "ragged_skew", "single", "ragged_pair", "edge_min", "many_experts"])
def test_tiles_small_bitwise_and_oracle(name):
    """Single-CTA GEMMs (ragged, many_experts, ...) and CTA pairs with swap
    tiles (ragged_pair): same bits as the kernel-per-step path, and the
    oracle's output within tolerance on every token."""
    wl = Workload(name)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    y_steps = _layer(wl, ws, mk.MK_PATH_STEPS).clone()
    h_steps = mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "h").clone()
    y_tiles = _layer(wl, ws, mk.MK_PATH_TILES)
    assert torch.equal(_bits(y_tiles), _bits(y_steps))
    assert torch.equal(_bits(mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "h")), _bits(h_steps))
    y_ref, _, _ = wl.oracle_layer()
    check_output(y_tiles.cpu(), y_ref, f"{name} tiles")


@pytest.mark.parametrize("T", [1, 2, 129, 3000])
def test_tiles_token_counts(T):
    wl = Workload("ragged_pair", T=T)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    y_steps = _layer(wl, ws, mk.MK_PATH_STEPS).clone()
    y_tiles = _layer(wl, ws, mk.MK_PATH_TILES)
    assert torch.equal(_bits(y_tiles), _bits(y_steps))


def test_tiles_back_to_back_calls_on_one_workspace():
    """Calls issued back to back on one stream and workspace, alternating
    inputs and paths: every output equals a separate kernel-per-step call (the
    semaphores are re-zeroed per call, nothing leaks between calls)."""
    wl = Workload("ragged_pair")
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    g = torch.Generator().manual_seed(9)
    xs = [wl.g["x"]] + [torch.randn((wl.T, c.d), generator=g).to(torch.bfloat16).to(wl.dev) for _ in range(3)]
    args = (wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    paths = [mk.MK_PATH_TILES, mk.MK_PATH_TILES, mk.MK_PATH_STEPS, mk.MK_PATH_TILES]
    ys = [mk.mk_moe_layer(x, *args, ws=ws, path=p).clone() for x, p in zip(xs, paths)]
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    ws2 = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    for x, y in zip(xs, ys):
        assert torch.equal(_bits(y), _bits(mk.mk_moe_layer(x, *args, ws=ws2)))


def test_tiles_host_buffers_match_device_call():
    wl = Workload("ragged_pair")
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    y_dev = _layer(wl, ws, mk.MK_PATH_STEPS).clone()
    x_host = wl.g["x"].cpu().pin_memory()
    y_host = torch.empty((wl.T, c.d), dtype=torch.bfloat16)  # pageable: chunked downloads
    mk.mk_moe_layer_host(x_host, wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, y_host, ws,
                         path=mk.MK_PATH_TILES)
    torch.cuda.synchronize()
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    assert torch.equal(_bits(y_host), _bits(y_dev.cpu()))


@pytest.mark.parametrize("name", ["ragged", "ragged_pair"])
def test_tiles_dropped_signal_times_out_cleanly(name):
    """The dispatch never publishes token 0's rows: the GEMM tiles and the
    combine that wait on their M-tiles give up after the given limit, the call
    reports MK_ERR_TIMEOUT, nothing faults or hangs, and the next call on the
    same workspace is bit-identical to the kernel-per-step path."""
    wl = Workload(name)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    args = (wl.g["x"], wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    mk.mk_moe_layer(*args, ws=ws, path=mk.MK_PATH_TILES, inject=mk.MK_INJECT_DROP_TILE_SIGNAL,
                    timeout_ns=20_000_000)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_ERR_TIMEOUT, (st, hex(site))
    y = mk.mk_moe_layer(*args, ws=ws, path=mk.MK_PATH_TILES)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    y_steps = mk.mk_moe_layer(*args, ws=ws)
    assert torch.equal(_bits(y), _bits(y_steps))


def test_tiles_rejects_other_hooks():
    wl = Workload("tiny")
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    args = (wl.g["x"], wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    for path, inject in ((mk.MK_PATH_TILES, mk.MK_INJECT_STALL_GEMM1), (mk.MK_PATH_STEPS, mk.MK_INJECT_DROP_TILE_SIGNAL)):
        with pytest.raises(mk.MoEError) as err:
            mk.mk_moe_layer(*args, ws=ws, path=path, inject=inject)
        assert err.value.status == mk.MK_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["mid", "skewed", "decode", "large"])
def test_tiles_full_size_bitwise(name):
    """Full-size workloads in the benchmark's launch configuration: the tile-
    synchronised path writes the same h, P and y bits as the kernel-per-step
    path (whose output the full-size oracle tests check)."""
    wl = Workload(name)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    y_steps = _layer(wl, ws, mk.MK_PATH_STEPS).clone()
    P_steps = mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "P").clone()
    y_tiles = _layer(wl, ws, mk.MK_PATH_TILES)
    assert torch.equal(_bits(y_tiles), _bits(y_steps))
    assert torch.equal(_bits(mk.workspace_view(ws, wl.T, c.d, c.E, c.k, c.f, "P")), _bits(P_steps))
    del wl, ws, y_steps, P_steps, y_tiles
    gc.collect()
    torch.cuda.empty_cache()
