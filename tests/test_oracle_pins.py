"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test compares the oracle with a closed form, a library routine on a
special case, a brute-force definition on tiny inputs, an invariant, or a
hand-worked value (tests/golden/).  Together they are chosen so that a
plausible slip (a dropped term, a wrong sign or index, a transposed operand,
gate and up swapped, a different summation order, a wrong tie-break) fails at
least one of them; test_oracle_mutants.py plants such slips and checks that.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dispatch_ffn_combine_gb300.workloads import bf16_bits, bits_to_float

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_seed = 1234


def _bf16(a):
    """float array -> bf16 bit patterns (round to nearest even, via torch)."""
    return bf16_bits(torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


# ---------------------------------------------------------------- router logits

def test_logits_exact_on_integers():
    """Small integers: every product and partial sum is exact in fp32, so any
    order must give the exact integer dot product (catches dropped terms,
    wrong strides and a transposed gate matrix; T != E != d)."""
    rs = np.random.RandomState(0)
    T, d, E = 7, 96, 5
    x = rs.randint(-8, 9, size=(T, d)).astype(np.float32)
    wg = rs.randint(-8, 9, size=(E, d)).astype(np.float32)
    bias = rs.randint(-50, 51, size=E).astype(np.float32)
    got = oracle.router_logits(_bf16(x), wg, bias)
    want = x.astype(np.int64) @ wg.astype(np.int64).T + bias.astype(np.int64)
    np.testing.assert_array_equal(got, want.astype(np.float32))
    got_nb = oracle.router_logits(_bf16(x), wg, None)
    np.testing.assert_array_equal(got_nb, (x.astype(np.int64) @ wg.astype(np.int64).T).astype(np.float32))


def test_logits_hand_worked_order():
    """Hand-derived values for the R1 order (golden fixture)."""
    spec = json.load(open(os.path.join(GOLDEN, "router_r1_order.json")))
    for case in spec["cases"]:
        d = case["d"]
        x = np.zeros((1, d), np.float32)
        wg = np.zeros((1, d), np.float32)
        for i, v in case["x"]:
            x[0, i] = v
        for i, v in case["wg"]:
            wg[0, i] = v
        xb = _bf16(x)
        assert np.array_equal(bits_to_float(xb), x), case["name"] + ": x not bf16-exact"
        assert np.array_equal(wg.astype(np.float64), np.array(wg, np.float64))
        bias = None if case["bias"] is None else np.array([case["bias"]], np.float32)
        got = oracle.router_logits(xb, wg, bias)[0, 0]
        assert got == np.float32(case["expected"]), (case["name"], float(got), case["expected"])


def test_logits_error_bound_vs_fp64():
    """Random inputs: the fp32 R1 logit lies within the standard forward error
    bound of the exact (fp64) dot product: |err| <= gamma_n * sum|x_i w_i|,
    n = d/32 + 5 (+1 for the bias)."""
    rs = np.random.RandomState(1)
    T, d, E = 16, 512, 12
    x = _bf16(rs.randn(T, d))
    wg = (rs.randn(E, d) / math.sqrt(d)).astype(np.float32)
    bias = rs.randn(E).astype(np.float32)
    got = oracle.router_logits(x, wg, bias).astype(np.float64)
    xf = bits_to_float(x).astype(np.float64)
    exact = xf @ wg.astype(np.float64).T + bias
    absdot = np.abs(xf) @ np.abs(wg.astype(np.float64)).T + np.abs(bias)
    u = 2.0 ** -24
    n = d // 32 + 5 + 1
    gamma = n * u / (1 - n * u)
    assert np.all(np.abs(got - exact) <= gamma * absdot)
    # and the fp64 diagnostic path is the exact value up to fp64 rounding
    f64 = oracle.router_logits_f64(x, wg, bias)
    assert np.allclose(f64, exact, rtol=0, atol=1e-12 * absdot.max())


# ---------------------------------------------------------------- top-k + weights

def _brute_topk(l, k):
    """Brute force from the definition: expert e's rank is the number of
    experts that beat it (larger logit, or equal logit and lower id); the
    expert of rank j sits in slot j, for j < k."""
    E = len(l)
    rank = [sum(1 for e2 in range(E) if l[e2] > l[e] or (l[e2] == l[e] and e2 < e)) for e in range(E)]
    slots = [None] * k
    for e in range(E):
        if rank[e] < k:
            slots[rank[e]] = e
    return slots


@pytest.mark.parametrize("E,k", [(8, 2), (6, 6), (13, 4), (32, 8), (5, 1)])
def test_topk_matches_brute_force_with_ties(E, k):
    rs = np.random.RandomState(E * 100 + k)
    T = 200
    # integer-valued logits from a small range: many exact ties
    logits = rs.randint(-3, 4, size=(T, E)).astype(np.float32)
    ids, w = oracle.topk(logits, k)
    for t in range(T):
        assert list(ids[t]) == _brute_topk(list(logits[t]), k)


def test_topk_signed_zero_tie():
    logits = np.array([[0.0, -0.0, -1.0], [-0.0, 0.0, -1.0]], np.float32)
    ids, w = oracle.topk(logits, 1)
    assert list(ids[:, 0]) == [0, 0]
    ids2, w2 = oracle.topk(logits, 2)
    assert [list(r) for r in ids2] == [[0, 1], [0, 1]]
    np.testing.assert_array_equal(w2, 0.5)


def test_topk_weights_k1_is_one():
    rs = np.random.RandomState(3)
    ids, w = oracle.topk(rs.randn(50, 16).astype(np.float32), 1)
    np.testing.assert_array_equal(w, 1.0)


def test_topk_weights_are_softmax_of_chosen():
    """Weights equal torch.softmax (fp64) over the chosen logits, sum to one,
    and with k = E equal the full softmax over all experts."""
    rs = np.random.RandomState(4)
    T, E, k = 64, 16, 5
    logits = (3 * rs.randn(T, E)).astype(np.float32)
    ids, w = oracle.topk(logits, k)
    chosen = np.take_along_axis(logits, ids, axis=1).astype(np.float64)
    ref = torch.softmax(torch.from_numpy(chosen), dim=1).numpy()
    np.testing.assert_allclose(w, ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-13)
    assert np.all(np.diff(chosen, axis=1) <= 0)  # slot order: descending logit
    idsE, wE = oracle.topk(logits, E)
    full = torch.softmax(torch.from_numpy(logits.astype(np.float64)), dim=1).numpy()
    np.testing.assert_allclose(wE, np.take_along_axis(full, idsE, axis=1), rtol=1e-13, atol=1e-16)


def test_topk_closed_form_two_experts():
    """Logits 0 and -ln 3 (to fp32): weights 1/(1+e^l) in closed form ~ (3/4, 1/4)."""
    l1 = np.float32(-math.log(3.0))
    ids, w = oracle.topk(np.array([[l1, 0.0]], np.float32), 2)
    assert list(ids[0]) == [1, 0]
    assert abs(w[0, 0] - 0.75) < 1e-7 and abs(w[0, 1] - 0.25) < 1e-7


# ---------------------------------------------------------------- dispatch

def _brute_dispatch(ids, E):
    T, k = ids.shape
    flat = [(t, j, int(ids[t, j])) for t in range(T) for j in range(k)]
    off = [sum(1 for (_, _, e2) in flat if e2 < e) for e in range(E + 1)]
    slot = np.empty((T, k), np.int64)
    for (t, j, e) in flat:
        earlier = sum(1 for t2 in range(t) if e in ids[t2])
        slot[t, j] = off[e] + earlier
    return np.array(off), slot


@pytest.mark.parametrize("T,E,k", [(40, 6, 2), (33, 9, 3), (17, 4, 4), (25, 1, 1)])
def test_dispatch_brute_force(T, E, k):
    rs = np.random.RandomState(T + E + k)
    ids = np.stack([rs.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, row_token, slot_row = oracle.dispatch(ids, E)
    off_bf, slot_bf = _brute_dispatch(ids, E)
    np.testing.assert_array_equal(offsets, off_bf)
    np.testing.assert_array_equal(slot_row, slot_bf)
    np.testing.assert_array_equal(counts, np.diff(off_bf))


def test_dispatch_invariants():
    rs = np.random.RandomState(7)
    T, E, k = 500, 24, 6
    ids = np.stack([rs.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, row_token, slot_row = oracle.dispatch(ids, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) == counts)
    assert sorted(slot_row.ravel().tolist()) == list(range(T * k))  # bijection
    for t in range(T):
        for j in range(k):
            r = slot_row[t, j]
            assert row_token[r] == t
            assert offsets[ids[t, j]] <= r < offsets[ids[t, j] + 1]
    for e in range(E):
        blk = row_token[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(blk) > 0)  # ascending token order inside an expert
    # each token appears exactly k times
    np.testing.assert_array_equal(np.bincount(row_token, minlength=T), k)


# ---------------------------------------------------------------- FFN / layer

def _weights(rs, E, d, f, same=False):
    def mk(shape, std):
        return _bf16(rs.randn(*shape) * std)
    if same:
        w1, w3, w2 = mk((1, f, d), d ** -0.5), mk((1, f, d), d ** -0.5), mk((1, d, f), f ** -0.5)
        return np.repeat(w1, E, 0), np.repeat(w3, E, 0), np.repeat(w2, E, 0)
    return mk((E, f, d), d ** -0.5), mk((E, f, d), d ** -0.5), mk((E, d, f), f ** -0.5)


def _torch_ffn(xb, w1b, w3b, w2b):
    """Dense SwiGLU FFN in fp64 with torch: W2 (silu(W1 x) * (W3 x))."""
    x = torch.from_numpy(bits_to_float(xb).astype(np.float64))
    w1 = torch.from_numpy(bits_to_float(w1b).astype(np.float64))
    w3 = torch.from_numpy(bits_to_float(w3b).astype(np.float64))
    w2 = torch.from_numpy(bits_to_float(w2b).astype(np.float64))
    h = torch.nn.functional.silu(x @ w1.T) * (x @ w3.T)
    return (h @ w2.T).numpy()


def test_layer_single_expert_is_dense_swiglu():
    """E = 1, k = 1: the layer is a dense SwiGLU FFN (torch fp64)."""
    rs = np.random.RandomState(11)
    T, d, f = 24, 96, 160
    xb = _bf16(rs.randn(T, d))
    wg = rs.randn(1, d).astype(np.float32)
    w1, w3, w2 = _weights(rs, 1, d, f)
    y, ids, w = oracle.layer(xb, wg, None, w1, w3, w2, k=1)
    assert np.all(ids == 0) and np.all(w == 1.0)
    ref = _torch_ffn(xb, w1[0], w3[0], w2[0])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_layer_identical_experts_is_dense():
    """All experts equal: whatever the routing, the weights sum to one, so y = FFN(x)."""
    rs = np.random.RandomState(12)
    T, d, E, k, f = 20, 64, 7, 3, 128
    xb = _bf16(rs.randn(T, d))
    wg = rs.randn(E, d).astype(np.float32)
    w1, w3, w2 = _weights(rs, E, d, f, same=True)
    y, _, _ = oracle.layer(xb, wg, None, w1, w3, w2, k=k)
    ref = _torch_ffn(xb, w1[0], w3[0], w2[0])
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


def test_layer_k_equals_E_is_full_mixture():
    """k = E: y = sum_e softmax(l)_e * FFN_e(x), every expert (torch fp64 einsum)."""
    rs = np.random.RandomState(13)
    T, d, E, f = 12, 64, 4, 96
    xb = _bf16(rs.randn(T, d))
    wg = (rs.randn(E, d) / 8).astype(np.float32)
    bias = rs.randn(E).astype(np.float32)
    w1, w3, w2 = _weights(rs, E, d, f)
    y, ids, w = oracle.layer(xb, wg, bias, w1, w3, w2, k=E)
    logits = oracle.router_logits(xb, wg, bias).astype(np.float64)
    p = torch.softmax(torch.from_numpy(logits), dim=1)
    outs = torch.stack([torch.from_numpy(_torch_ffn(xb, w1[e], w3[e], w2[e])) for e in range(E)], 1)
    ref = torch.einsum("te,ted->td", p, outs).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


def test_layer_power_of_two_scaling_is_exact():
    """Doubling W2 (exact in bf16) doubles y bit for bit."""
    rs = np.random.RandomState(14)
    T, d, E, k, f = 16, 64, 5, 2, 64
    xb = _bf16(rs.randn(T, d))
    wg = rs.randn(E, d).astype(np.float32)
    w1, w3, w2 = _weights(rs, E, d, f)
    w2x2 = _bf16(bits_to_float(w2) * 2)
    assert np.array_equal(bits_to_float(w2x2), bits_to_float(w2) * 2)
    y1, _, _ = oracle.layer(xb, wg, None, w1, w3, w2, k=k)
    y2, _, _ = oracle.layer(xb, wg, None, w1, w3, w2x2, k=k)
    np.testing.assert_array_equal(y2, 2 * y1)


def test_layer_consistent_with_pieces_and_sample():
    """The layer's routing equals router_logits+topk; its per-token outputs equal
    sum_j w_j * expert_ffn; a token sample gives the same rows as the full run."""
    rs = np.random.RandomState(15)
    T, d, E, k, f = 30, 64, 6, 2, 64
    xb = _bf16(rs.randn(T, d))
    wg = rs.randn(E, d).astype(np.float32)
    w1, w3, w2 = _weights(rs, E, d, f)
    y, ids, w = oracle.layer(xb, wg, None, w1, w3, w2, k=k)
    ids2, w2_ = oracle.topk(oracle.router_logits(xb, wg, None), k)
    np.testing.assert_array_equal(ids, ids2)
    np.testing.assert_array_equal(w, w2_)
    toks = np.repeat(np.arange(T), k)
    outs = oracle.expert_ffn(xb, w1, w3, w2, toks, ids.ravel()).reshape(T, k, d)
    np.testing.assert_allclose(y, np.einsum("tk,tkd->td", w, outs), rtol=1e-13, atol=1e-14)
    sample = np.array([29, 3, 3, 0])
    ys, _, _ = oracle.layer(xb, wg, None, w1, w3, w2, k=k, tokens=sample)
    np.testing.assert_array_equal(ys, y[sample])


# ---------------------------------------------------------------- expert linear (Dispatch + GEMM)

def test_expert_linear_matches_torch_matmul():
    """W_e x_t for listed pairs equals torch's fp64 matmul of the same bf16 values."""
    rs = np.random.RandomState(21)
    T, d, E, n = 9, 96, 4, 80
    xb = _bf16(rs.randn(T, d))
    wb = _bf16(rs.randn(E, n, d) * d ** -0.5)
    toks = np.array([0, 8, 3, 3, 5, 1, 7])
    exps = np.array([2, 0, 3, 1, 2, 0, 3])
    out = oracle.expert_linear(xb, wb, toks, exps)
    x = torch.from_numpy(bits_to_float(xb).astype(np.float64))
    w = torch.from_numpy(bits_to_float(wb).astype(np.float64))
    ref = torch.stack([w[e] @ x[t] for t, e in zip(toks, exps)]).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())


def test_expert_linear_permutation_and_scale_experts():
    """Expert e = 2^e times a permutation matrix: out row = 2^e * x permuted, exactly
    (a transposed weight index would apply the inverse permutation)."""
    rs = np.random.RandomState(22)
    T, d, E = 5, 64, 3
    xb = _bf16(rs.randn(T, d))
    perms = [rs.permutation(d) for _ in range(E)]
    w = np.zeros((E, d, d), dtype=np.float32)
    for e, pi in enumerate(perms):
        w[e, np.arange(d), pi] = 2.0 ** e          # row c picks input pi[c]
    wb = _bf16(w)
    toks = np.array([4, 0, 2, 2, 1])
    exps = np.array([0, 1, 2, 0, 1])
    out = oracle.expert_linear(xb, wb, toks, exps)
    x = bits_to_float(xb).astype(np.float64)
    for p, (t, e) in enumerate(zip(toks, exps)):
        np.testing.assert_array_equal(out[p], (2.0 ** e) * x[t][perms[e]])


def test_dispatch_gemm_composes_route_dispatch_linear():
    """Dispatch + GEMM = the router's choice, the dispatch row order, and each row's
    expert map: row r of expert e holds W_e x_{row_token[r]}; row weights are the
    routing weights of (token, slot)."""
    rs = np.random.RandomState(23)
    T, d, E, k, n = 21, 64, 5, 2, 64
    xb = _bf16(rs.randn(T, d))
    wg = rs.randn(E, d).astype(np.float32)
    wb = _bf16(rs.randn(E, n, d) * d ** -0.5)
    out, off, row_token, row_weight = oracle.dispatch_gemm(xb, wg, None, wb, k)
    ids, w = oracle.topk(oracle.router_logits(xb, wg, None), k)
    x = bits_to_float(xb).astype(np.float64)
    wf = bits_to_float(wb).astype(np.float64)
    assert off[0] == 0 and off[-1] == T * k
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            t = row_token[r]
            j = list(ids[t]).index(e)
            assert row_weight[r] == w[t, j]
            np.testing.assert_allclose(out[r], wf[e] @ x[t], rtol=1e-13, atol=1e-13)
