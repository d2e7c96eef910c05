"""GPU parity: router and dispatch against the CPU oracle, through the C ABI.

Routing decides integers, so ids, counts, offsets, row order and slot rows
must match the oracle bit for bit; the fp32 routing weights (GPU expf vs the
oracle's fp64 exp of the same fp32 logits) must agree to 1e-6 relative."""
import math

import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
import oracle
from _support import Workload, sample_tokens
from dispatch_ffn_combine_gb300.workloads import bits_to_float

pytestmark = pytest.mark.gpu

ROUTE_CONFIGS = ["tiny", "ragged", "ragged_skew", "single", "edge_min", "many_experts", "mid", "skewed", "decode", "large"]


@pytest.mark.parametrize("name", ROUTE_CONFIGS)
def test_route_bit_exact(name):
    wl = Workload(name, experts=False)
    E, k = wl.cfg.E, wl.cfg.k
    ws = mk.alloc_workspace(wl.T, wl.cfg.d, E, k, 64, wl.dev)
    ids, w, counts = mk.mk_moe_route(wl.g["x"], wl.g["wg"], wl.g["bias"], k, ws=ws)
    # the candidate filter's error bound held for every logit it was checked on
    assert mk.mk_moe_route_fallbacks(ws) == 0
    _, ids_ref, w_ref = wl.oracle_routing()
    ids_g = ids.cpu().numpy()
    mismatch = np.nonzero(np.any(ids_g != ids_ref, axis=1))[0]
    assert mismatch.size == 0, f"{mismatch.size} tokens routed differently (first {mismatch[:5]}); " \
                               f"near-ties in fp64: {wl.near_ties(ids_ref)}"
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=1e-7)
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(ids_ref.ravel(), minlength=E))


def _route_vs_oracle(x, wg, bias, k, expect_fallbacks=0):
    dev = torch.device("cuda:0")
    T, d = x.shape
    E = wg.shape[0]
    ws = mk.alloc_workspace(T, d, E, k, 64, dev)
    ids, w, counts = mk.mk_moe_route(x.to(dev), wg.to(dev), None if bias is None else bias.to(dev), k, ws=ws)
    assert mk.mk_moe_route_fallbacks(ws) == expect_fallbacks
    from dispatch_ffn_combine_gb300.workloads import bf16_bits
    logits = oracle.router_logits(bf16_bits(x), wg.numpy(), None if bias is None else bias.numpy())
    ids_ref, w_ref = oracle.topk(logits, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=1e-7)
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(ids_ref.ravel(), minlength=E))
    return ids_ref


def test_route_exact_and_near_ties():
    """Gate rows that tie exactly (duplicates: the lower id must win) or differ
    by one ulp in one element, scaled up so that they compete for the top
    slots: the tensor-core filter cannot separate them, every one is a
    candidate, and the fixed-order logits decide as in the oracle."""
    T, d, E, k = 512, 512, 64, 8
    g = torch.Generator().manual_seed(11)
    x = torch.randn((T, d), generator=g).to(torch.bfloat16)
    wg = torch.randn((E, d), generator=g) * d ** -0.5
    wg[5] *= 3.0
    wg[6] = wg[5]                                   # exact duplicate of 5
    wg[8] = wg[5]
    wg[8, 17] = torch.nextafter(wg[8, 17], torch.tensor(10.0))   # one ulp away in one element
    wg[9] = wg[8]
    wg[40] = wg[5] * (1.0 + 2.0 ** -23)             # a relative hair above 5
    wg[41] = wg[40]
    ids_ref = _route_vs_oracle(x, wg, None, k)
    # the tied rows really did compete: 5 beats its duplicates 6 in every token choosing both
    both = (ids_ref == 5).any(1) & (ids_ref == 6).any(1)
    assert both.sum() > T // 4
    pos5 = np.argmax(ids_ref == 5, axis=1)[both]
    pos6 = np.argmax(ids_ref == 6, axis=1)[both]
    assert np.all(pos5 < pos6)


def test_route_wide_dynamic_range_and_cancellation():
    """Token rows with a few huge entries of both signs and gate rows spanning
    many binades: large cancellation inside each logit, and a bias."""
    T, d, E, k = 300, 1024, 32, 4
    g = torch.Generator().manual_seed(12)
    x = torch.randn((T, d), generator=g)
    x[:, ::97] *= 512.0
    x = x.to(torch.bfloat16)
    scale = torch.pow(2.0, torch.randint(-20, 6, (E, d), generator=g).float())
    wg = torch.randn((E, d), generator=g) * scale * d ** -0.5
    wg[:, 1::97] = -wg[:, ::97][:, : wg[:, 1::97].shape[1]]
    bias = torch.randn(E, generator=g)
    _route_vs_oracle(x, wg, bias, k)


def test_route_fixed_order_decides_weights():
    """Hand-worked order case on the GPU: token 0's expert 0 row is the
    'tree_not_chain' vector (R1 logit 2^24+2; a single sequential chain gives
    2^24, exact-then-round 2^24+4); expert 1's logit is exactly 2^24.  The
    routing weights are then 1/(1+e^-2) and e^-2/(1+e^-2) only under R1."""
    d, E, k = 64, 2, 2
    dev = torch.device("cuda:0")
    x = torch.zeros((1, d), dtype=torch.float32)
    x[0, :4] = 1.0
    wg = torch.zeros((E, d), dtype=torch.float32)
    wg[0, 0] = 16777216.0
    wg[0, 1:4] = 1.0
    wg[1, 0] = 16777216.0
    xb = x.to(torch.bfloat16).to(dev)
    ids, w, _ = mk.mk_moe_route(xb, wg.to(dev), None, k)
    torch.cuda.synchronize()
    assert ids.cpu().tolist() == [[0, 1]]
    e2 = math.exp(-2.0)
    np.testing.assert_allclose(w.cpu().numpy()[0], [1 / (1 + e2), e2 / (1 + e2)], rtol=1e-6)


@pytest.mark.parametrize("name", ["tiny", "ragged", "ragged_skew", "single", "edge_min", "many_experts", "mid", "skewed",
                                  "decode", "large"])
def test_dispatch_bit_exact(name):
    """GPU dispatch of the oracle's routing equals the oracle's dispatch."""
    wl = Workload(name, experts=False)
    E, k, T, d = wl.cfg.E, wl.cfg.k, wl.T, wl.cfg.d
    _, ids_ref, w_ref = wl.oracle_routing()
    ids_dev = torch.from_numpy(ids_ref).to(wl.dev)
    w_dev = torch.from_numpy(w_ref.astype(np.float32)).to(wl.dev)
    ws = mk.alloc_workspace(T, d, E, k, 64, wl.dev)
    res = mk.mk_moe_dispatch(wl.g["x"], ids_dev, w_dev, E, ws=ws)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_OK, (st, hex(site))
    counts, offsets, row_token, slot_row = oracle.dispatch(ids_ref, E)
    np.testing.assert_array_equal(res["expert_offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(res["row_token"].cpu().numpy(), row_token)
    np.testing.assert_array_equal(res["slot_row"].cpu().numpy(), slot_row)
    rw = res["row_weight"].cpu().numpy()
    np.testing.assert_array_equal(rw[slot_row.ravel()], w_ref.astype(np.float32).ravel())
    # x_perm rows are bitwise copies of the token rows
    xp = res["x_perm"].view(torch.int16)
    xs = wl.g["x"].view(torch.int16)
    rt = torch.from_numpy(row_token.astype(np.int64)).to(wl.dev)
    assert torch.equal(xp, xs.index_select(0, rt))


def test_dispatch_random_routing_and_edge_counts():
    """Routing not produced by the router: every expert count from 0 upward,
    including experts nobody picks."""
    T, d, E, k = 531, 128, 16, 4
    rs = np.random.RandomState(5)
    ids = np.stack([rs.choice(np.arange(E - 3), size=k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[::7, k - 1] = E - 1  # a rarely used expert; experts E-3 and E-2 stay empty
    for r in ids:
        assert len(set(r.tolist())) == k
    dev = torch.device("cuda:0")
    x = (torch.randn((T, d), generator=torch.Generator().manual_seed(3))).to(torch.bfloat16).to(dev)
    res = mk.mk_moe_dispatch(x, torch.from_numpy(ids).to(dev), None, E)
    torch.cuda.synchronize()
    counts, offsets, row_token, slot_row = oracle.dispatch(ids, E)
    assert counts[E - 3] == 0 and counts[E - 2] == 0
    np.testing.assert_array_equal(res["expert_offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(res["row_token"].cpu().numpy(), row_token)
    np.testing.assert_array_equal(res["slot_row"].cpu().numpy(), slot_row)
    np.testing.assert_array_equal(res["row_weight"].cpu().numpy(), 1.0)


def test_dispatch_rejects_bad_ids_on_device():
    """Out-of-range and repeated expert ids are caught by the kernel's own
    checks (MK_ERR_BOUNDS), every access stays in bounds, and the next call on
    the same workspace works."""
    T, d, E, k = 300, 128, 8, 2
    dev = torch.device("cuda:0")
    x = torch.zeros((T, d), dtype=torch.bfloat16, device=dev)
    ws = mk.alloc_workspace(T, d, E, k, 64, dev)
    good = np.stack([np.array([t % E, (t + 1) % E]) for t in range(T)]).astype(np.int32)
    for bad_fill in ("range", "repeat"):
        ids = good.copy()
        if bad_fill == "range":
            ids[17, 1] = E + 3
            ids[200, 0] = -1
        else:
            ids[42, 1] = ids[42, 0]
        mk.mk_moe_dispatch(x, torch.from_numpy(ids).to(dev), None, E, ws=ws)
        st, site = mk.mk_moe_last_device_error(ws)
        assert st == mk.MK_ERR_BOUNDS, (bad_fill, st, hex(site))
    res = mk.mk_moe_dispatch(x, torch.from_numpy(good).to(dev), None, E, ws=ws)
    st, _ = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_OK
    np.testing.assert_array_equal(res["slot_row"].cpu().numpy(), oracle.dispatch(good, E)[3])


@pytest.mark.parametrize("name", ["tiny", "ragged", "edge_min", "mid", "skewed", "decode", "large"])
def test_approx_logit_error_within_model(name):
    """The candidate filter's bound takes each tensor-core MMA step to err by at
    most 2^-18 of its magnitudes.  The whole approximate logit (bf16 split of the
    gate rows, tensor-core accumulation, fp32 chunk sums, bias) must stay within
    2^-19 ||x_t|| ||w_e|| of the fixed-order logit on every (token, expert) of a
    token sample -- measured 2^-20.6 at d = 256 and 2^-22.6 at d = 7168."""
    wl = Workload(name, experts=False)
    c = wl.cfg
    ws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, 64, wl.dev)
    mk.mk_moe_route(wl.g["x"], wl.g["wg"], wl.g["bias"], c.k, ws=ws)
    A = mk.mk_moe_route_approx_logits(ws, wl.T, c.d, c.E, c.k).cpu().numpy().astype(np.float64)
    toks = sample_tokens(wl.T, 512)
    xb = wl.bits("x")[toks]
    exact = oracle.router_logits(xb, wl.wg, wl.bias).astype(np.float64)
    x = bits_to_float(xb).astype(np.float64)
    nx = np.sqrt((x ** 2).sum(1))
    nw = np.sqrt((wl.wg.astype(np.float64) ** 2).sum(1))
    ratio = np.abs(A[toks] - exact) / (nx[:, None] * nw[None, :])
    assert ratio.max() <= 2.0 ** -19, f"{name}: approximate logit error 2^{np.log2(ratio.max()):.2f} ||x|| ||w||"
    assert mk.mk_moe_route_fallbacks(ws) == 0


def test_tensor_core_step_error_within_eta():
    """The router's candidate filter assumes that one tcgen05 MMA step (16 bf16
    products added to the fp32 accumulator) errs by at most
    eta * (|acc| + sum |products|), eta = 2^-18.  This test measures that on
    inputs built to make the step error as large as the accumulator allows:
    d = 64, so the approximate logit is one accumulation of four steps over the
    gate rows' high parts (then four steps of exactly zero products, the gate
    rows being bf16 values), with no bias and one chunk, so the logit the
    library returns is the accumulator itself.  Column 0 holds a large product
    2^(a_t + b_e) (a_t in [0, 20], b_e in [-8, 23]); the other 63 columns hold
    products of mixed sign with exponents spread over [-8, 10), so across the
    (token, expert) pairs the small products fall above, across and below the
    accumulator's last bit.  Every product is exact in fp64 and the exact sum
    comes from math.fsum, so |A - exact| is the hardware's accumulation error;
    it must stay under eta times sum over the four steps of (|exact partial sum
    before the step| + sum |products of the step|)."""
    import math

    T, d, E, k = 2048, 64, 64, 2
    rs = np.random.RandomState(21)
    mx = rs.randint(0, 128, size=(T, d))
    ex = rs.randint(-4, 5, size=(T, d))
    sx = rs.choice([-1.0, 1.0], size=(T, d))
    x = sx * (1.0 + mx / 128.0) * np.exp2(ex)
    x[:, 0] = np.exp2(rs.randint(0, 21, size=T))
    mw = rs.randint(0, 128, size=(E, d))
    ew = rs.randint(-4, 5, size=(E, d))
    sw = rs.choice([-1.0, 1.0], size=(E, d))
    w = sw * (1.0 + mw / 128.0) * np.exp2(ew)
    w[:, 0] = np.exp2((np.arange(E) % 32) - 8)
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(xb.float(), torch.from_numpy(x.astype(np.float32)))  # every value exact in bf16
    wg = torch.from_numpy(w.astype(np.float32))
    assert torch.equal(wg.to(torch.bfloat16).float(), wg)  # the gate rows' low parts are zero
    dev = torch.device("cuda:0")
    ws = mk.alloc_workspace(T, d, E, k, 64, dev)
    mk.mk_moe_route(xb.to(dev), wg.to(dev), None, k, ws=ws)
    A = mk.mk_moe_route_approx_logits(ws, T, d, E, k).cpu().numpy().astype(np.float64)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK

    prods = x[:, None, :] * w[None, :, :]  # [T, E, d], exact in fp64 (8-bit x 8-bit significands)
    exact = np.array([[math.fsum(prods[t, e]) for e in range(E)] for t in range(T)])
    steps = prods.reshape(T, E, 4, 16)
    step_abs = np.abs(steps).sum(axis=3)
    before = np.zeros((T, E, 4))
    for s in range(1, 4):
        before[:, :, s] = np.array([[math.fsum(steps[t, e, :s].ravel()) for e in range(E)] for t in range(T)])
    M = (np.abs(before) + step_abs).sum(axis=2)
    ratio = np.abs(A - exact) / M
    eta = 2.0 ** -18
    worst = float(ratio.max())
    assert worst <= eta, f"tensor-core accumulation error 2^{math.log2(worst):.2f} of its magnitudes > 2^-18"
    # the construction does reach the accumulator's last bit: some pairs lose low-order product bits
    assert np.count_nonzero(ratio) > T * E // 100
