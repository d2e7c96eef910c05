"""The router entry point that allocates nothing (mk_moe_route_noalloc).

It exists for callers that cannot allocate device memory for a workspace: a
runtime whose memory is planned up front, a path that must not call cudaMalloc,
a plug-in that is only handed its inputs and outputs.  Its logits live in a
static device array inside the library instead.  This file checks, through
the C ABI, on two calls in a row with different shapes:

  - against the CPU oracle: ids and counts bit for bit, weights within the
    routing tolerance of the other tests (1e-6 relative);
  - against mk_moe_route (the workspace router, which takes the tensor-core
    candidate filter on these shapes): ids, weights and counts bit for bit,
    since both compute the same fixed-order fp32 logits and the same softmax.

It also checks that sizes beyond the static array are refused and that the
largest size it holds is accepted.  It is collected last so a run that stops
at the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
import oracle
from dispatch_ffn_combine_gb300.workloads import CONFIGS, bf16_bits, make_inputs

pytestmark = pytest.mark.gpu


def _route_both(cfg, seed):
    dev = torch.device("cuda:0")
    inp = make_inputs(cfg, seed=seed, device=dev, experts=False)
    x, wg, bias = inp["x"], inp["wg"], inp["bias"]
    T, E, k = x.shape[0], cfg.E, cfg.k
    ids_ws, w_ws, cnt_ws = mk.mk_moe_route(x, wg, bias, k)
    ids = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    w = torch.full((T, k), -7.0, dtype=torch.float32, device=dev)
    cnt = torch.full((E,), -7, dtype=torch.int32, device=dev)
    mk.mk_moe_route_noalloc(x, wg, bias, k, ids, w, cnt)
    torch.cuda.synchronize()
    logits = oracle.router_logits(bf16_bits(x.cpu()), wg.cpu().numpy(), None if bias is None else bias.cpu().numpy())
    ids_ref, w_ref = oracle.topk(logits, k)
    return (ids, w, cnt), (ids_ws, w_ws, cnt_ws), (ids_ref, w_ref)


def test_noalloc_router_matches_oracle_and_workspace_router_two_calls():
    # Two calls in a row with different shapes (E = 64 with a skew bias, then
    # E = 256): the second must not see anything the first left in the array.
    for name, seed in (("skewed", 3), ("decode", 4)):
        cfg = CONFIGS[name]
        T = 8192 if name == "skewed" else cfg.T
        cfg = type(cfg)(cfg.name, T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.zipf_s)
        (ids, w, cnt), (ids_ws, w_ws, cnt_ws), (ids_ref, w_ref) = _route_both(cfg, seed)
        ids_np = ids.cpu().numpy()
        np.testing.assert_array_equal(ids_np, ids_ref)
        np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=1e-7)
        np.testing.assert_array_equal(cnt.cpu().numpy(), np.bincount(ids_ref.ravel(), minlength=cfg.E))
        np.testing.assert_array_equal(ids_np, ids_ws.cpu().numpy())
        assert torch.equal(w.view(torch.int32), w_ws.view(torch.int32)), "weights differ in their bits"
        np.testing.assert_array_equal(cnt.cpu().numpy(), cnt_ws.cpu().numpy())


def _zeros(T, d, E, k):
    dev = torch.device("cuda:0")
    x = torch.zeros((T, d), dtype=torch.bfloat16, device=dev)
    wg = torch.zeros((E, d), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    return x, wg, ids, w


def test_noalloc_router_refuses_more_logits_than_its_array():
    T, d, E, k = 8193, 64, 256, 2  # T * E = 2,097,408 > 2,097,152
    x, wg, ids, w = _zeros(T, d, E, k)
    with pytest.raises(mk.MoEError) as err:
        mk.mk_moe_route_noalloc(x, wg, None, k, ids, w)
    assert err.value.status == mk.MK_ERR_UNSUPPORTED


def test_noalloc_router_accepts_a_full_array():
    # T * E = 2,097,152 exactly: every logit equal (zero rows), so the k
    # lowest ids win and the weights are 1/k each
    T, d, E, k = 8192, 64, 256, 2
    x, wg, ids, w = _zeros(T, d, E, k)
    cnt = torch.empty(E, dtype=torch.int32, device=x.device)
    mk.mk_moe_route_noalloc(x, wg, None, k, ids, w, cnt)
    torch.cuda.synchronize()
    assert torch.equal(ids.cpu(), torch.tensor([[0, 1]], dtype=torch.int32).expand(T, k))
    assert torch.equal(w.cpu(), torch.full((T, k), 0.5))
    assert cnt[:2].tolist() == [T, T] and int(cnt[2:].abs().sum()) == 0
