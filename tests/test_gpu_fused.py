"""The fused persistent kernel (one launch, blocks in mover / compute roles).

Every step runs the same arithmetic in the same order as the kernel-per-step
path, so the two paths must agree bit for bit, and so must every split of the
blocks between roles (adaptive controller or fixed); the oracle checks the
output itself."""
import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
from _support import Workload, check_output

pytestmark = pytest.mark.gpu


def _layer(wl, **kw):
    c = wl.cfg
    kw.setdefault("path", mk.MK_PATH_FUSED)
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    y = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, ws=ws, **kw)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_OK, (st, hex(site))
    return y


@pytest.mark.parametrize("name", ["tiny", "ragged", "ragged_skew", "single", "ragged_pair", "edge_min", "many_experts", "mid", "skewed"])
def test_fused_equals_steps_bitwise(name):
    wl = Workload(name)
    y_f = _layer(wl, path=mk.MK_PATH_FUSED, timeout_ns=500_000_000)
    y_s = _layer(wl, path=mk.MK_PATH_STEPS)
    assert torch.equal(y_f.view(torch.int16), y_s.view(torch.int16))


def test_fused_chunk_dispatch_tasks_bitwise():
    """20000 tokens make 157 counting chunks, at least one per SM, so the
    persistent kernel dispatches whole 128-token chunks (smaller layers take
    quarter chunks); the result must equal the kernel-per-step path's."""
    wl = Workload("ragged", T=20000)
    y_f = _layer(wl, path=mk.MK_PATH_FUSED)
    y_s = _layer(wl, path=mk.MK_PATH_STEPS)
    assert torch.equal(y_f.view(torch.int16), y_s.view(torch.int16))


@pytest.mark.parametrize("movers", [1, 16, 75, 151, -1])
def test_fused_any_split_bitwise(movers):
    wl = Workload("ragged_skew")
    y0 = _layer(wl)
    y1 = _layer(wl, mover_ctas=movers)
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("T", [1, 37, 128, 129])
def test_fused_few_tokens(T):
    wl = Workload("ragged", T=T)
    y = _layer(wl)
    y_ref, _, _ = wl.oracle_layer()
    check_output(y.cpu(), y_ref, f"fused T={T}")


def test_fused_repeated_calls_same_workspace():
    """Counters and flags are cleared per call: back-to-back calls on one
    workspace give identical results."""
    wl = Workload("ragged")
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    args = (wl.g["x"], wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    ys = [mk.mk_moe_layer(*args, ws=ws, path=mk.MK_PATH_FUSED).clone() for _ in range(3)]
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    assert all(torch.equal(ys[0].view(torch.int16), y.view(torch.int16)) for y in ys[1:])


@pytest.mark.parametrize("movers", [8, -1])
def test_fused_prerouted_any_split_bitwise(movers):
    """Skewed is large enough for the candidate-filter router, so the fused path
    takes its routing, counts and scans from kernels launched before the
    persistent kernel; every split still gives the kernel-per-step bits."""
    wl = Workload("skewed")
    y_s = _layer(wl, path=mk.MK_PATH_STEPS)
    y_f = _layer(wl, mover_ctas=movers)
    assert torch.equal(y_f.view(torch.int16), y_s.view(torch.int16))
