"""Expert-parallel MoE layer over G ranks (one GPU per rank).

The mKernel README's "MoE Dispatch + FFN + Combine" row is the expert-parallel
layer: tokens are routed "to their expert ranks", each rank runs the FFN of the
experts it owns, and the weighted outputs are combined "back to each token's
source rank" (the paper's section 3.1 and Table 3 describe the dispatch
exchange).  Here rank r owns experts [r E/G, (r + 1) E/G) and holds their
W1, W3, W2; the gate is replicated.  One layer call on rank r:

  1. route and dispatch its own tokens over all E experts (mk_moe_route,
     mk_moe_dispatch): the rows are expert-contiguous, so the rows for rank q
     are one contiguous range;
  2. exchange the per-(rank, local expert) row counts, then the rows and their
     routing weights (all-to-all); rank r receives, from every source q, the
     rows of its experts in source-major order [q][e][rows];
  3. regroup them expert-major (mk_moe_ep_regroup, which also gives the local
     expert offsets) and run the grouped expert FFN of the local experts
     (mk_moe_expert_ffn: gemm1 -> SwiGLU -> gemm2 with the routing weight);
  4. regroup the weighted outputs back to source-major order and return them
     (all-to-all with the splits reversed): every source gets its rows back in
     the order it sent them, i.e. in its own dispatch order;
  5. combine them into its tokens' outputs (mk_moe_combine).

The arithmetic runs in the library's kernels; this module marshals tensors and
sizes the exchanges (a few host integers per call).  The exchange is pluggable:
`DistExchange` uses torch.distributed all-to-all (NCCL between GPUs; gloo for
host tensors), and `ep_layer_virtual` runs G ranks in one process on one device,
moving the exchanged rows with tensor copies, to check the expert-parallel
arithmetic on one GPU.  The steps are pluggable too (`steps=`), so the
exchange logic can be exercised with other implementations of the five steps.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass
class Shard:
    """Rank `rank` of `world` owns experts [first, first + local) of E."""

    rank: int
    world: int
    E: int

    def __post_init__(self):
        if self.world < 1 or self.E % self.world != 0:
            raise ValueError(f"E={self.E} experts do not split evenly over {self.world} ranks")
        if not 0 <= self.rank < self.world:
            raise ValueError(f"rank {self.rank} outside [0, {self.world})")

    @property
    def local(self) -> int:
        return self.E // self.world

    @property
    def first(self) -> int:
        return self.rank * self.local


def exchange_plan(send_counts_host, recv_counts_host):
    """Split sizes of the row exchanges from the count matrices (host ints).

    send_counts_host[q][e]: rows this rank sends to rank q for q's local expert e;
    recv_counts_host[q][e]: rows this rank receives from source q for its expert e.
    Returns (send_splits, recv_splits), one entry per rank."""
    send = [int(sum(row)) for row in send_counts_host]
    recv = [int(sum(row)) for row in recv_counts_host]
    return send, recv


class CudaSteps:
    """The five steps on the library's kernels (device tensors)."""

    def __init__(self):
        from . import (mk_moe_combine, mk_moe_dispatch, mk_moe_ep_regroup, mk_moe_expert_ffn,  # noqa: F401
                       mk_moe_route)

        self._route = mk_moe_route
        self._dispatch = mk_moe_dispatch
        self._regroup = mk_moe_ep_regroup
        self._ffn = mk_moe_expert_ffn
        self._combine = mk_moe_combine

    def route(self, x, wg, bias, k):
        """(ids [T,k], weights [T,k], counts [E]) over all E experts."""
        return self._route(x, wg, bias, k)

    def dispatch(self, x, ids, w, E):
        """dict(expert_offsets, row_token, row_weight, slot_row, x_perm): rows expert-contiguous."""
        return self._dispatch(x, ids, w, E)

    def regroup(self, rows, counts, to_expert_major, expert_offsets=None):
        return self._regroup(rows, counts, to_expert_major, expert_offsets=expert_offsets)

    def expert_ffn(self, rows, offsets, row_weight, w1, w3, w2):
        return self._ffn(rows, offsets, row_weight, w1, w3, w2)[1]

    def combine(self, P, slot_row):
        return self._combine(P, slot_row)


class DistExchange:
    """All-to-all over a torch.distributed process group."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_to_all(self, send, send_splits, recv_splits):
        out = torch.empty((int(sum(recv_splits)),) + tuple(send.shape[1:]), dtype=send.dtype, device=send.device)
        self.dist.all_to_all_single(out, send.contiguous(), list(recv_splits), list(send_splits), group=self.group)
        return out


@dataclasses.dataclass
class RankState:
    """One rank's tensors between the phases of a layer call."""

    T: int
    counts: torch.Tensor = None      # [E] rows per expert from this rank's tokens
    disp: dict = None                # dispatch outputs (own rows, expert-contiguous)
    send_counts: list = None         # host [G][E_local]
    recv_counts: list = None         # host [G][E_local]
    send_splits: list = None
    recv_splits: list = None
    recv_rows: torch.Tensor = None
    recv_w: torch.Tensor = None
    P_src: torch.Tensor = None       # this rank's experts' outputs, source-major


def phase_route_dispatch(steps, shard, x, wg, bias, k):
    st = RankState(T=x.shape[0])
    ids, w, counts = steps.route(x, wg, bias, k)
    st.counts = counts
    st.disp = steps.dispatch(x, ids, w, shard.E)
    cnt = counts.reshape(shard.world, shard.local).cpu()
    st.send_counts = cnt.tolist()
    return st


def phase_experts(steps, shard, st, w1, w3, w2):
    """Regroup the received rows expert-major, run the local experts' FFN, and
    regroup the outputs back to source-major order."""
    dev = st.recv_rows.device
    counts = torch.tensor(st.recv_counts, dtype=torch.int32).to(dev)
    offsets = torch.empty(shard.local + 1, dtype=torch.int32, device=dev)
    rows_em = steps.regroup(st.recv_rows, counts, True, expert_offsets=offsets)
    w_em = steps.regroup(st.recv_w, counts, True)
    P_em = steps.expert_ffn(rows_em, offsets, w_em.reshape(-1), w1, w3, w2)
    st.P_src = steps.regroup(P_em, counts, False)
    return st


def ep_layer(x, wg, bias, w1_local, w3_local, w2_local, k, E, exchange, steps=None):
    """The expert-parallel layer on one rank: this rank's tokens x [T, d] in,
    their outputs y [T, d] out.  w1_local, w3_local [E/G, ffn, d] and
    w2_local [E/G, d, ffn] are the weights of the experts this rank owns."""
    steps = steps or CudaSteps()
    shard = Shard(exchange.rank, exchange.world, E)
    st = phase_route_dispatch(steps, shard, x, wg, bias, k)
    G, El = shard.world, shard.local
    flat = torch.tensor(st.send_counts, dtype=torch.int32).reshape(-1).to(x.device)
    st.recv_counts = exchange.all_to_all(flat, [El] * G, [El] * G).reshape(G, El).tolist()
    st.send_splits, st.recv_splits = exchange_plan(st.send_counts, st.recv_counts)
    st.recv_rows = exchange.all_to_all(st.disp["x_perm"], st.send_splits, st.recv_splits)
    st.recv_w = exchange.all_to_all(st.disp["row_weight"].reshape(-1, 1), st.send_splits, st.recv_splits)
    phase_experts(steps, shard, st, w1_local, w3_local, w2_local)
    P_back = exchange.all_to_all(st.P_src, st.recv_splits, st.send_splits)
    return steps.combine(P_back, st.disp["slot_row"])


def _virtual_all_to_all(sends, send_splits):
    """What G ranks' all-to-all delivers, with every rank's data in this process:
    rank q receives, in source order, the piece of every sender's rows meant for q."""
    G = len(sends)
    pieces = [list(torch.split(sends[r], send_splits[r], dim=0)) for r in range(G)]
    return [torch.cat([pieces[r][q] for r in range(G)], dim=0) for q in range(G)]


def ep_layer_virtual(xs, wg, bias, w1, w3, w2, k, steps=None):
    """G ranks of the expert-parallel layer in one process on one device: xs is
    the list of the ranks' token batches; w1, w3, w2 hold all E experts and rank
    r uses its slice.  Returns the list of the ranks' outputs.  The exchanges
    are tensor copies; every step of each rank runs as ep_layer would run it."""
    steps = steps or CudaSteps()
    G = len(xs)
    E = w1.shape[0]
    shards = [Shard(r, G, E) for r in range(G)]
    El = shards[0].local
    sts = [phase_route_dispatch(steps, shards[r], xs[r], wg, bias, k) for r in range(G)]
    for q in range(G):  # counts: rank q receives row q of every sender's matrix
        sts[q].recv_counts = [sts[r].send_counts[q] for r in range(G)]
    for st in sts:
        st.send_splits, st.recv_splits = exchange_plan(st.send_counts, st.recv_counts)
    recv_rows = _virtual_all_to_all([st.disp["x_perm"] for st in sts], [st.send_splits for st in sts])
    recv_w = _virtual_all_to_all([st.disp["row_weight"].reshape(-1, 1) for st in sts], [st.send_splits for st in sts])
    for r in range(G):
        sts[r].recv_rows, sts[r].recv_w = recv_rows[r], recv_w[r]
        lo, hi = r * El, (r + 1) * El
        phase_experts(steps, shards[r], sts[r], w1[lo:hi], w3[lo:hi], w2[lo:hi])
    backs = _virtual_all_to_all([st.P_src for st in sts], [st.recv_splits for st in sts])
    return [steps.combine(backs[r], sts[r].disp["slot_row"]) for r in range(G)]
