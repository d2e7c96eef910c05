"""GPU parity: the grouped expert FFN (tcgen05 GEMMs) and the combine.

The FFN is checked against the oracle's fp64 expert FFN on rows dispatched by
the oracle; the combine against its plain definition in its own precision
(fp32 sum in ascending slot order, rounded once to bf16): bit-exact."""
import numpy as np
import pytest
import torch

import dispatch_ffn_combine_gb300 as mk
import oracle
from _support import check_output
from dispatch_ffn_combine_gb300.workloads import bf16_bits, bits_to_float

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _rand_bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _ffn_case(counts, d, f, seed=0, weights=True):
    """Expert-contiguous rows with the given per-expert counts."""
    E = len(counts)
    S = int(sum(counts))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x_perm = _rand_bf16((S, d), 1.0, seed)
    w1 = _rand_bf16((E, f, d), d ** -0.5, seed + 1)
    w3 = _rand_bf16((E, f, d), d ** -0.5, seed + 2)
    w2 = _rand_bf16((E, d, f), f ** -0.5, seed + 3)
    rw = torch.rand(S, generator=torch.Generator().manual_seed(seed + 4)) if weights else None
    return offsets, x_perm, w1, w3, w2, rw


def _check_ffn(counts, d, f, seed=0, weights=True, sample=None):
    offsets, x_perm, w1, w3, w2, rw = _ffn_case(counts, d, f, seed, weights)
    E = len(counts)
    S = x_perm.shape[0]
    h, P = mk.mk_moe_expert_ffn(x_perm.to(DEV), torch.from_numpy(offsets).to(DEV),
                                None if rw is None else rw.to(DEV), w1.to(DEV), w3.to(DEV), w2.to(DEV))
    torch.cuda.synchronize()
    rows = np.arange(S) if sample is None else sample
    expert_of_row = np.searchsorted(offsets, rows, side="right") - 1
    ref = oracle.expert_ffn(bf16_bits(x_perm), bf16_bits(w1), bf16_bits(w3), bf16_bits(w2), rows,
                            expert_of_row.astype(np.int32))
    if rw is not None:
        ref = ref * rw.numpy().astype(np.float64)[rows, None]
    check_output(P.cpu()[torch.from_numpy(rows)], ref, f"P counts={counts}")
    # h against its definition in fp64 (torch), per expert
    xf = bits_to_float(bf16_bits(x_perm)).astype(np.float64)
    hg = bits_to_float(bf16_bits(h.cpu())).astype(np.float64)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        xe = torch.from_numpy(xf[a:b])
        g = xe @ torch.from_numpy(bits_to_float(bf16_bits(w1[e])).astype(np.float64)).T
        u = xe @ torch.from_numpy(bits_to_float(bf16_bits(w3[e])).astype(np.float64)).T
        check_output(hg[a:b], (torch.nn.functional.silu(g) * u).numpy(), f"h expert {e}")


def test_ffn_tile_edges():
    """Experts with 0, 1, 127, 128, 129, 255, 256, 300 rows; K and N ragged
    against the 64 / 128 / 256 tile sizes (d = 320, ffn = 192)."""
    _check_ffn([0, 1, 127, 128, 129, 0, 255, 256, 300], d=320, f=192, seed=10)


def test_ffn_tile_edges_many_rows():
    """Experts with 0, 1, 255, 256, 257, 511, 513, 600 rows (tiles claimed in
    expert-local N groups; groups with one, several and a partial last row
    block); d = 384 leaves half of the last 256-column gemm2 tile outside the
    output."""
    _check_ffn([0, 1, 255, 256, 257, 600, 511, 513, 129], d=384, f=320, seed=60)


@pytest.mark.parametrize("d,f", [(256, 384), (384, 320)])
def test_ffn_swap_tile_sizes(d, f):
    """Every expert has one full 256-row block and a partial one of 1..255
    rows, which runs with the operands exchanged: the tails cross each
    activation box (16 / 32 / 64 / 128 rows per CTA) and N step (16); with
    d = 384 and ffn = 320 the last output tile of each GEMM is partly outside
    the output."""
    tails = [1, 8, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 240, 255]
    _check_ffn([256 + t for t in tails], d=d, f=f, seed=70 + d)


def test_ffn_swap_tile_sizes_long_k():
    """K = 4096 (64 k-blocks): gemm1 also runs tails of 129..255 rows as swap
    tiles (shorter K keeps them as full tiles); the tail rows are checked."""
    tails = [1, 17, 100, 129, 200, 255]
    counts = [256 + t for t in tails]
    offs = np.cumsum([0] + counts)
    sample = np.concatenate([np.arange(offs[i] + 250, offs[i + 1]) for i in range(len(counts))])
    _check_ffn(counts, d=4096, f=256, seed=95, sample=sample)


@pytest.mark.parametrize("d,tail", [(256, 100), (4096, 200)])
def test_ffn_swap_tiles_bitwise_equal_full_tiles(d, tail):
    """The same rows through a full tile and through a swap tile give the same
    bits: expert 1 repeats expert 0's weights, and its rows after the first
    256 repeat rows of expert 0 (the first 256 of them make a full tile)."""
    f = 384
    offsets, x_perm, w1, w3, w2, rw = _ffn_case([512, 256 + tail], d, f, seed=90)
    for w in (w1, w3, w2):
        w[1] = w[0]
    x_perm[512 + 256:] = x_perm[:tail]
    rw[512 + 256:] = rw[:tail]
    h, P = mk.mk_moe_expert_ffn(x_perm.to(DEV), torch.from_numpy(offsets).to(DEV), rw.to(DEV), w1.to(DEV),
                                w3.to(DEV), w2.to(DEV))
    torch.cuda.synchronize()
    h, P = h.cpu().view(torch.int16), P.cpu().view(torch.int16)
    assert torch.equal(h[512 + 256:], h[:tail])
    assert torch.equal(P[512 + 256:], P[:tail])


def test_ffn_single_expert_many_tiles():
    _check_ffn([1000], d=512, f=640, seed=20)


def test_ffn_no_row_weight():
    _check_ffn([5, 64, 200], d=256, f=256, seed=30, weights=False)


def test_ffn_large_k_extent():
    """Long K loop (d = 4096: 64 k-blocks, many trips round the 4-stage ring)."""
    counts = [130, 7, 260]
    _check_ffn(counts, d=4096, f=256, seed=40, sample=np.r_[0:10, 125:140, 390:397])


def test_ffn_rejects_bad_offsets():
    """Offsets that do not run from 0 to S are caught on the device (MK_ERR_BOUNDS)
    and no tile runs; the next call on the workspace works."""
    offsets, x_perm, w1, w3, w2, rw = _ffn_case([10, 20], 128, 128, seed=50)
    ws = torch.zeros(512, dtype=torch.uint8, device=DEV)
    bad = torch.tensor([0, 25, 40], dtype=torch.int32, device=DEV)  # ends past S = 30
    args = (x_perm.to(DEV), bad, rw.to(DEV), w1.to(DEV), w3.to(DEV), w2.to(DEV))
    mk.mk_moe_expert_ffn(*args, ws=ws)
    st, site = mk.mk_moe_last_device_error(ws)
    assert st == mk.MK_ERR_BOUNDS, (st, hex(site))
    mk.mk_moe_expert_ffn(x_perm.to(DEV), torch.from_numpy(offsets).to(DEV), *args[2:], ws=ws)
    assert mk.mk_moe_last_device_error(ws)[0] == mk.MK_OK


@pytest.mark.parametrize("T,d,k", [(1, 64, 1), (37, 192, 3), (300, 1024, 8)])
def test_combine_bit_exact(T, d, k):
    S = T * k
    P = _rand_bf16((S, d), 0.3, T + d + k)
    rs = np.random.RandomState(T)
    slot_row = rs.permutation(S).reshape(T, k).astype(np.int32)
    y = mk.mk_moe_combine(P.to(DEV), torch.from_numpy(slot_row).to(DEV))
    torch.cuda.synchronize()
    pf = bits_to_float(bf16_bits(P))
    acc = np.zeros((T, d), np.float32)
    for j in range(k):
        acc = (acc + pf[slot_row[:, j]]).astype(np.float32)
    want = bf16_bits(torch.from_numpy(acc).to(torch.bfloat16))
    np.testing.assert_array_equal(bf16_bits(y.cpu()), want)
