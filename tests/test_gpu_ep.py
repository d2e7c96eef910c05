"""GPU checks of the expert-parallel layer's pieces: the row regroup kernel
(mk_moe_ep_regroup) against its definition, G ranks of the expert-parallel
layer run in one process on one GPU (ep_layer_virtual) against the one-GPU
layer bit for bit, and ep_layer over a one-rank NCCL group.  (More than one
GPU per run is not available here; the exchange logic across processes is
covered by world-size-2 gloo ranks in tests/test_ep_cpu.py.)"""
import os
import socket

import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
from _support import Workload
from dispatch_ffn_combine_gb300 import ep

pytestmark = pytest.mark.gpu


def _regroup_ref(rows, counts, to_expert_major):
    c = counts.astype(np.int64)
    G, El = c.shape
    src = np.concatenate([[0], np.cumsum(c.reshape(-1))])
    dst = np.zeros((G, El), dtype=np.int64)
    s = 0
    for e in range(El):
        for q in range(G):
            dst[q, e] = s
            s += c[q, e]
    out = np.empty_like(rows)
    for q in range(G):
        for e in range(El):
            a, b, n = src[q * El + e], dst[q, e], c[q, e]
            if to_expert_major:
                out[b:b + n] = rows[a:a + n]
            else:
                out[a:a + n] = rows[b:b + n]
    return out, np.concatenate([dst[0], [s]]).astype(np.int32)


@pytest.mark.parametrize("G,El,d,dtype", [(4, 3, 128, torch.bfloat16), (2, 5, 1, torch.float32),
                                          (8, 32, 64, torch.bfloat16), (1, 4, 256, torch.bfloat16)])
def test_regroup_matches_definition_both_ways(G, El, d, dtype):
    rs = np.random.RandomState(G * 100 + El)
    counts = rs.randint(0, 40, size=(G, El)).astype(np.int32)
    counts[0, El - 1] = 0  # an empty group
    R = int(counts.sum())
    dev = torch.device("cuda:0")
    rows = torch.randn((R, d), generator=torch.Generator().manual_seed(3)).to(dtype)
    c_dev = torch.from_numpy(counts).to(dev)
    off = torch.full((El + 1,), -1, dtype=torch.int32, device=dev)
    em = mk.mk_moe_ep_regroup(rows.to(dev), c_dev, True, expert_offsets=off)
    ref, off_ref = _regroup_ref(rows.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy(), counts,
                                True)
    got = em.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy()
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(off.cpu().numpy(), off_ref)
    back = mk.mk_moe_ep_regroup(em, c_dev, False)
    assert torch.equal(back.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       rows.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))


def test_regroup_rejects_inconsistent_counts_on_device():
    dev = torch.device("cuda:0")
    counts = torch.tensor([[3, -1], [2, 2]], dtype=torch.int32, device=dev)
    rows = torch.arange(6 * 4, dtype=torch.float32, device=dev).reshape(6, 4)
    n = int(mk.load_library().mk_moe_ep_regroup_workspace_size(2, 2))
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    out = mk.mk_moe_ep_regroup(rows, counts, True, ws=ws)
    st, _ = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_ERR_BOUNDS
    assert torch.equal(out, rows)  # copied unmoved
    good = torch.tensor([[3, 0], [2, 1]], dtype=torch.int32, device=dev)
    mk.mk_moe_ep_regroup(rows, good, True, ws=ws)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK


@pytest.mark.parametrize("name,G", [("tiny", 2), ("tiny", 8), ("ragged_pair", 3), ("mid", 4), ("large", 8)])
def test_virtual_ranks_equal_one_gpu_layer(name, G):
    """Every token's output through G expert-parallel ranks equals the one-GPU
    layer's bit for bit: each row meets the same expert weights in the same
    GEMM arithmetic, and the combine adds the same rows in the same order."""
    wl = Workload(name)
    c = wl.cfg
    y_one = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    T = wl.T
    cuts = np.linspace(0, T, G + 1).astype(int)
    cuts[1] = max(cuts[1] - T // (3 * G), 0)  # uneven token counts across ranks
    xs = [wl.g["x"][cuts[r]:cuts[r + 1]].contiguous() for r in range(G)]
    ys = ep.ep_layer_virtual(xs, wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
    torch.cuda.synchronize()
    y_ep = torch.cat(ys, dim=0)
    assert torch.equal(y_ep.view(torch.int16), y_one.view(torch.int16))


def test_ep_layer_over_a_one_rank_nccl_group():
    import torch.distributed as dist

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        wl = Workload("ragged_pair")
        c = wl.cfg
        y_one = mk.mk_moe_layer(wl.g["x"], wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k)
        y = ep.ep_layer(wl.g["x"], wl.g["wg"], None, wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, c.E, ep.DistExchange())
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_one.view(torch.int16))
    finally:
        dist.destroy_process_group()
