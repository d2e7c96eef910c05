"""GPU parity: MoE Dispatch + GEMM (route -> dispatch -> one grouped GEMM).

The README's "MoE Dispatch + GEMM" row computes, for every token and each of
its k experts, that expert's linear map of the token's row, with the rows
grouped by expert.  Here the weight of each workload's experts is the layer's
gate projection W1 [E, ffn, d] (n = ffn).  The routing tables are compared
bit for bit with the oracle's, the routing weights to 1e-6, and the GEMM rows
with the oracle's fp64 per-expert linear map within the layer tolerance."""
import gc

import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
import oracle
from _support import Workload, check_output, sample_tokens
from dispatch_ffn_combine_gb300.workloads import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _rand_bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _check_grouped(counts, d, n, seed, weights):
    E = len(counts)
    S = int(sum(counts))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x_perm = _rand_bf16((S, d), 1.0, seed)
    w = _rand_bf16((E, n, d), d ** -0.5, seed + 1)
    rw = torch.rand(S, generator=torch.Generator().manual_seed(seed + 2)) if weights else None
    out = mk.mk_moe_grouped_gemm(x_perm.to(DEV), torch.from_numpy(offsets).to(DEV), w.to(DEV),
                                 row_weight=None if rw is None else rw.to(DEV))
    torch.cuda.synchronize()
    rows = np.arange(S)
    expert_of_row = (np.searchsorted(offsets, rows, side="right") - 1).astype(np.int32)
    ref = oracle.expert_linear(bf16_bits(x_perm), bf16_bits(w), rows, expert_of_row)
    if rw is not None:
        ref = ref * rw.numpy().astype(np.float64)[:, None]
    check_output(out.cpu(), ref, f"grouped GEMM counts={counts}")


def test_grouped_gemm_tile_edges_single_cta():
    """Experts of 0, 1, 127, 128, 129, 255, 256, 300 rows (single-CTA tiles: the
    experts average fewer than 256 rows); K = 320 and N = 192 ragged against the
    64-wide k-blocks and 256-wide N tiles."""
    _check_grouped([0, 1, 127, 128, 129, 0, 255, 256, 300], d=320, n=192, seed=70, weights=True)


def test_grouped_gemm_tile_edges_pairs():
    """Experts of 0 ... 600 rows averaging over 256 (CTA-pair tiles, half tiles for
    odd 128-row block counts); N = 384 leaves half of the last N tile outside."""
    _check_grouped([0, 1, 255, 256, 257, 600, 511, 513, 129], d=256, n=384, seed=71, weights=False)


def test_grouped_gemm_long_k():
    """K = 2048 (32 k-blocks: several trips round the pipeline ring)."""
    _check_grouped([300, 40, 700], d=2048, n=256, seed=72, weights=True)


def test_grouped_gemm_rejects_bad_offsets():
    """Offsets that do not end at S: MK_ERR_BOUNDS on the device, no tile runs,
    the output is left untouched, and the next call on the workspace works."""
    S, d, n, E = 30, 128, 128, 2
    x_perm = _rand_bf16((S, d), 1.0, 73).to(DEV)
    w = _rand_bf16((E, n, d), d ** -0.5, 74).to(DEV)
    ws = torch.zeros(512, dtype=torch.uint8, device=DEV)
    out = torch.full((S, n), 7.0, dtype=torch.bfloat16, device=DEV)
    bad = torch.tensor([0, 25, 40], dtype=torch.int32, device=DEV)
    mk.mk_moe_grouped_gemm(x_perm, bad, w, out=out, ws=ws)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_ERR_BOUNDS, (st, hex(site))
    assert bool((out == 7.0).all())
    good = torch.tensor([0, 10, 30], dtype=torch.int32, device=DEV)
    mk.mk_moe_grouped_gemm(x_perm, good, w, out=out, ws=ws)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK


def _run(wl, ws=None):
    c = wl.cfg
    ws = mk.alloc_dispatch_gemm_workspace(wl.T, c.d, c.E, c.k, wl.dev) if ws is None else ws
    res = mk.mk_moe_dispatch_gemm(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], c.k, ws=ws)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK
    return res, ws


def _check_tables(wl, res):
    c = wl.cfg
    ids, w = oracle.topk(oracle.router_logits(wl.bits("x"), wl.wg, wl.bias), c.k)
    _, off_ref, row_token_ref, slot_ref = oracle.dispatch(ids, c.E)
    np.testing.assert_array_equal(res["expert_offsets"].cpu().numpy(), off_ref)
    np.testing.assert_array_equal(res["row_token"].cpu().numpy(), row_token_ref)
    rw_ref = np.empty(wl.T * c.k)
    rw_ref[slot_ref.ravel()] = w.ravel()
    np.testing.assert_allclose(res["row_weight"].cpu().numpy(), rw_ref, rtol=1e-6, atol=1e-7)
    row_expert = np.empty(wl.T * c.k, dtype=np.int32)
    row_expert[slot_ref.ravel()] = ids.ravel()
    return row_token_ref, row_expert


@pytest.mark.parametrize("name", ["tiny", "ragged", "ragged_skew", "single", "ragged_pair", "edge_min", "many_experts"])
def test_dispatch_gemm_small_all_rows(name):
    wl = Workload(name)
    res, _ = _run(wl)
    out_ref, off_ref, row_token_ref, rw_ref = oracle.dispatch_gemm(wl.bits("x"), wl.wg, wl.bias, wl.bits("w1"),
                                                                   wl.cfg.k)
    _check_tables(wl, res)
    np.testing.assert_array_equal(res["row_token"].cpu().numpy(), row_token_ref)
    check_output(res["out"].cpu(), out_ref, name)


@pytest.mark.parametrize("T", [1, 2, 129])
def test_dispatch_gemm_few_tokens(T):
    wl = Workload("ragged", T=T)
    res, _ = _run(wl)
    out_ref, _, _, _ = oracle.dispatch_gemm(wl.bits("x"), wl.wg, wl.bias, wl.bits("w1"), wl.cfg.k)
    _check_tables(wl, res)
    check_output(res["out"].cpu(), out_ref, f"ragged T={T}")


def test_dispatch_gemm_zero_tokens_and_bad_sizes():
    wl = Workload("tiny", T=0)
    c = wl.cfg
    ws = mk.alloc_dispatch_gemm_workspace(0, c.d, c.E, c.k, wl.dev)
    res = mk.mk_moe_dispatch_gemm(wl.g["x"], wl.g["wg"], None, wl.g["w1"], c.k, ws=ws)
    assert res["out"].shape == (0, c.f)
    assert int(res["expert_offsets"].abs().sum()) == 0
    w_bad = torch.zeros((c.E, 96, c.d), dtype=torch.bfloat16, device=wl.dev)  # n not a multiple of 64
    with pytest.raises(mk.MoEError) as exc:
        mk.mk_moe_dispatch_gemm(wl.g["x"], wl.g["wg"], None, w_bad, c.k, ws=ws)
    assert exc.value.status == mk.MK_ERR_INVALID_ARG


def test_dispatch_gemm_deterministic_and_matches_layer_steps():
    """Two calls give the same bits; the dispatched rows and offsets equal the
    layer's own routing tables on the same inputs."""
    wl = Workload("ragged_pair")
    c = wl.cfg
    a, ws = _run(wl)
    b, _ = _run(wl, ws)
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))
    assert torch.equal(a["row_token"], b["row_token"])
    lws = mk.alloc_workspace(wl.T, c.d, c.E, c.k, c.f, wl.dev)
    mk.mk_moe_layer(wl.g["x"], wl.g["wg"], wl.g["bias"], wl.g["w1"], wl.g["w3"], wl.g["w2"], c.k, ws=lws)
    _, _, offsets, _ = mk.mk_moe_layer_routing(lws, wl.T, c.d, c.E, c.k, c.f)
    assert torch.equal(offsets, a["expert_offsets"])


@pytest.mark.parametrize("name,T,n_sample", [("large", 8192, 64), ("large", None, 48), ("skewed", None, 64)])
def test_dispatch_gemm_full_size(name, T, n_sample):
    """Full-size dimensions in the sweep's and the benchmark's launch configuration:
    routing tables bit-exact on all tokens, GEMM rows on a token sample (all k
    rows of each sampled token)."""
    wl = Workload(name, T=T)
    res, _ = _run(wl)
    row_token, row_expert = _check_tables(wl, res)
    toks = sample_tokens(wl.T, n_sample)
    rows = np.flatnonzero(np.isin(row_token, toks))
    ref = oracle.expert_linear(wl.bits("x"), wl.bits("w1"), row_token[rows], row_expert[rows])
    check_output(res["out"].cpu()[torch.from_numpy(rows)], ref, f"{name} T={wl.T}")
    del wl, res
    gc.collect()
    torch.cuda.empty_cache()
