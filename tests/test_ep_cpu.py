"""Expert-parallel layer (dispatch_ffn_combine_gb300.ep) on world-size-2 gloo
ranks on the CPU: the exchange plan (count matrices, split sizes, the
source-major / expert-major regroup and its inverse, the return exchange)
with the five steps taken from the CPU oracle.  Each rank's outputs must equal
the oracle's single-process layer on that rank's tokens, and every rank's
received counts must equal the brute-force count from all ranks' routing.

The steps here are test infrastructure (the oracle, plus a regroup written
from its definition); the library's own steps run on the GPU
(tests/test_gpu_ep.py)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from dispatch_ffn_combine_gb300 import ep
from dispatch_ffn_combine_gb300.workloads import CONFIGS, bf16_bits, make_inputs


class OracleSteps:
    """The five steps on host tensors, from the CPU oracle (fp64 outputs)."""

    def route(self, x, wg, bias, k):
        logits = oracle.router_logits(bf16_bits(x), wg.numpy(), None if bias is None else bias.numpy())
        ids, w = oracle.topk(logits, k)
        counts = np.bincount(ids.ravel(), minlength=wg.shape[0]).astype(np.int32)
        return torch.from_numpy(ids), torch.from_numpy(w), torch.from_numpy(counts)

    def dispatch(self, x, ids, w, E):
        _, offsets, row_token, slot_row = oracle.dispatch(ids.numpy(), E)
        row_weight = np.zeros(row_token.size, dtype=np.float64)
        row_weight[slot_row.ravel()] = w.numpy().ravel()
        return {"expert_offsets": torch.from_numpy(offsets), "row_token": torch.from_numpy(row_token),
                "row_weight": torch.from_numpy(row_weight), "slot_row": torch.from_numpy(slot_row),
                "x_perm": x[torch.from_numpy(row_token.astype(np.int64))]}

    def regroup(self, rows, counts, to_expert_major, expert_offsets=None):
        # definition: a row keeps its place inside its (source q, expert e) group;
        # source-major groups run (q, e), expert-major groups (e, q)
        c = counts.numpy().astype(np.int64)
        G, El = c.shape
        src = np.concatenate([[0], np.cumsum(c.reshape(-1))])
        dst = np.zeros((G, El), dtype=np.int64)
        s = 0
        for e in range(El):
            for q in range(G):
                dst[q, e] = s
                s += c[q, e]
        out = torch.empty_like(rows)
        for q in range(G):
            for e in range(El):
                a, b, n = src[q * El + e], dst[q, e], c[q, e]
                if to_expert_major:
                    out[b:b + n] = rows[a:a + n]
                else:
                    out[a:a + n] = rows[b:b + n]
        if expert_offsets is not None:
            expert_offsets[:El] = torch.from_numpy(dst[0].astype(np.int32))
            expert_offsets[El] = int(c.sum())
        return out

    def expert_ffn(self, rows, offsets, row_weight, w1, w3, w2):
        off = offsets.numpy().astype(np.int64)
        experts = np.repeat(np.arange(len(off) - 1), np.diff(off))
        if rows.shape[0] == 0:
            return torch.zeros((0, w2.shape[1]), dtype=torch.float64)
        out = oracle.expert_ffn(bf16_bits(rows), bf16_bits(w1), bf16_bits(w3), bf16_bits(w2),
                                np.arange(rows.shape[0], dtype=np.int64), experts)
        return torch.from_numpy(out * row_weight.numpy().astype(np.float64)[:, None])

    def combine(self, P, slot_row):
        return P[slot_row.long()].sum(dim=1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, splits, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = CONFIGS["tiny"]
        inp = make_inputs(cfg, seed=0, device="cpu", T=sum(splits))
        x_all = inp["x"]
        t0 = sum(splits[:rank])
        x = x_all[t0:t0 + splits[rank]]
        shard = ep.Shard(rank, world, cfg.E)
        lo, hi = shard.first, shard.first + shard.local
        steps = OracleSteps()
        ex = ep.DistExchange()
        y = ep.ep_layer(x, inp["wg"], inp["bias"], inp["w1"][lo:hi], inp["w3"][lo:hi], inp["w2"][lo:hi], cfg.k, cfg.E,
                        ex, steps=steps)
        # the oracle's layer on this rank's tokens
        y_ref, ids_ref, _ = oracle.layer(bf16_bits(x_all), inp["wg"].numpy(), None, bf16_bits(inp["w1"]),
                                         bf16_bits(inp["w3"]), bf16_bits(inp["w2"]), cfg.k,
                                         tokens=np.arange(t0, t0 + splits[rank]))
        err = float(np.abs(y.numpy() - y_ref).max()) if y.numel() else 0.0
        # brute-force received counts: rows from every rank's tokens for my experts
        ids_all = oracle.topk(oracle.router_logits(bf16_bits(x_all), inp["wg"].numpy(), None), cfg.k)[0]
        recv_bf = []
        for src in range(world):
            s0 = sum(splits[:src])
            ids_src = ids_all[s0:s0 + splits[src]].ravel()
            recv_bf.append([int((ids_src == e).sum()) for e in range(lo, hi)])
        st = ep.phase_route_dispatch(steps, shard, x, inp["wg"], inp["bias"], cfg.k)
        flat = torch.tensor(st.send_counts, dtype=torch.int32).reshape(-1)
        recv = ex.all_to_all(flat, [shard.local] * world, [shard.local] * world).reshape(world, shard.local).tolist()
        q.put((rank, err, float(np.abs(y_ref).max()) if y_ref.size else 0.0, recv == recv_bf, recv))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("splits", [(128, 128), (100, 37), (0, 60)])
def test_ep_layer_two_gloo_ranks_matches_oracle(splits):
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_rank_main, args=(2, _free_port(), list(splits), q), nprocs=2, join=True,
                       start_method="spawn")
    res = sorted(q.get() for _ in range(2))
    for rank, err, scale, counts_ok, recv in res:
        assert counts_ok, (rank, recv)
        assert err <= 1e-12 * max(scale, 1.0), (rank, err, scale)


def test_exchange_plan_and_virtual_all_to_all():
    """The split sizes are the row sums of the count matrices, and the virtual
    all-to-all hands rank q, in source order, the piece of each sender meant
    for q."""
    send = [[1, 2], [0, 3]]
    recv = [[4, 0], [2, 2]]
    assert ep.exchange_plan(send, recv) == ([3, 3], [4, 4])
    a = torch.arange(5).reshape(5, 1)
    b = torch.arange(10, 13).reshape(3, 1)
    out = ep._virtual_all_to_all([a, b], [[2, 3], [1, 2]])
    assert out[0].ravel().tolist() == [0, 1, 10]
    assert out[1].ravel().tolist() == [2, 3, 4, 11, 12]
    with pytest.raises(ValueError):
        ep.Shard(0, 3, 8)
