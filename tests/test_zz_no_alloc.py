"""The router entry point that allocates nothing (mk_moe_route_noalloc).

It exists for callers that cannot allocate device memory for a workspace: a
runtime whose memory is planned up front, a path that must not call cudaMalloc,
a plug-in that is only handed its inputs and outputs.  Its logits live in a
static device array inside the library instead.  This file checks, through
the C ABI, that two calls in a row give the same routing as mk_moe_route
(ids bit for bit, weights within the routing tolerance of the other tests),
and that sizes beyond the static array are refused.  It is collected last so a
run that stops at the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
from dispatch_ffn_combine_gb300.workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _route_both(cfg, seed):
    dev = torch.device("cuda:0")
    inp = make_inputs(cfg, seed=seed, device=dev, experts=False)
    x, wg, bias = inp["x"], inp["wg"], inp["bias"]
    T, E, k = x.shape[0], cfg.E, cfg.k
    ids_ref, w_ref, cnt_ref = mk.mk_moe_route(x, wg, bias, k)
    ids = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    w = torch.full((T, k), -7.0, dtype=torch.float32, device=dev)
    cnt = torch.full((E,), -7, dtype=torch.int32, device=dev)
    mk.mk_moe_route_noalloc(x, wg, bias, k, ids, w, cnt)
    torch.cuda.synchronize()
    return (ids, w, cnt), (ids_ref, w_ref, cnt_ref)


def test_noalloc_router_matches_workspace_router_two_calls():
    # Two calls in a row with different shapes (E = 64 with a skew bias, then
    # E = 256): the second must not see anything the first left in the array.
    for name, seed in (("skewed", 3), ("decode", 4)):
        cfg = CONFIGS[name]
        T = 8192 if name == "skewed" else cfg.T
        cfg = type(cfg)(cfg.name, T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.zipf_s)
        (ids, w, cnt), (ids_ref, w_ref, cnt_ref) = _route_both(cfg, seed)
        np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy())
        np.testing.assert_allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=1e-6, atol=1e-7)
        np.testing.assert_array_equal(cnt.cpu().numpy(), cnt_ref.cpu().numpy())


def test_noalloc_router_refuses_more_logits_than_its_array():
    dev = torch.device("cuda:0")
    T, d, E, k = 8193, 64, 256, 2  # T * E = 2,097,408 > 2,097,152
    x = torch.zeros((T, d), dtype=torch.bfloat16, device=dev)
    wg = torch.zeros((E, d), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    with pytest.raises(mk.MoEError) as err:
        mk.mk_moe_route_noalloc(x, wg, None, k, ids, w)
    assert err.value.status == mk.MK_ERR_UNSUPPORTED
