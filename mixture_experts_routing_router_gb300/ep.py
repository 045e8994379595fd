"""Expert parallelism: the count-first exchange across ranks around the one-GPU
kernels.

afdEP-comm count-first validation record (.change, .setup, and the fault
patches P3 "count puts" / P4 "FFN publishes prefix sums"): the experts of a
layer are split over the ranks of a node; a token's rows travel to the ranks
that own its experts and the expert outputs travel back.  Counts go first:

  1. every rank routes and dispatches its own tokens (moe_route, moe_dispatch:
     x_perm is expert-contiguous, hence already grouped by owner rank);
  2. the per-expert counts are all-gathered (E int32 per rank);
  3. moe_ep_plan turns them into every segment's place: where rank s's rows of
     expert e start in s's x_perm, and where they land in the owner's receive
     buffer -- expert-contiguous, sources in rank order -- plus the capacity
     verdict, which every rank reaches alike;
  4. each (source, expert) segment moves once, point to point, straight into
     its slot (no staging copy on the receiver);
  5. the owner runs the grouped expert FFN on its local experts (moe_expert_ffn
     with the received bucket bounds);
  6. the outputs go back along the same segments into each source's own
     dispatch order, and the source combines (moe_combine).

Experts are owned in contiguous balanced blocks: rank g holds experts
[g*E//G, (g+1)*E//G).  Shared experts are not part of this layer.

The transport is pluggable: TorchDistTransport moves tensors with
torch.distributed point-to-point operations (NCCL between GPUs, gloo between
CPU processes); a segment of a rank to itself is a local copy.  Moving the rows
is plumbing: every number of the layer comes from the library's kernels, and
the plan from its host code (moe_ep_plan).
"""
from __future__ import annotations

import numpy as np
import torch

from . import native as N


def owned_experts(experts: int, world: int, rank: int) -> range:
    """The experts rank `rank` owns when `experts` are split over `world` ranks."""
    return range(rank * experts // world, (rank + 1) * experts // world)


class TorchDistTransport:
    """Collectives and ordered point-to-point segments over torch.distributed."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        """[world, *t.shape]: every rank's t, in rank order."""
        parts = [torch.empty_like(t) for _ in range(self.world)]
        self.dist.all_gather(parts, t.contiguous(), group=self.group)
        return torch.stack(parts)

    def exchange(self, sends, recvs):
        """Move segments: sends and recvs are lists of (peer, tensor, tag), each
        list in the order both sides agree on (ascending expert per peer)."""
        ops = [self.dist.P2POp(self.dist.isend, t, self._global(p), self.group, tag) for p, t, tag in sends]
        ops += [self.dist.P2POp(self.dist.irecv, t, self._global(p), self.group, tag) for p, t, tag in recvs]
        if ops:
            for req in self.dist.batch_isend_irecv(ops):
                req.wait()

    def _global(self, peer: int) -> int:
        if self.group is None:
            return peer
        return self.dist.get_global_rank(self.group, peer)


class ExchangePlan:
    """The plan of one layer call: every rank's counts and this rank's segments."""

    def __init__(self, experts, world, rank, capacity, counts_all):
        self.experts, self.world, self.rank = experts, world, rank
        self.counts_all = np.ascontiguousarray(counts_all, dtype=np.int32)
        self.status, p = N.moe_ep_plan(experts, world, rank, capacity, self.counts_all)
        self.send_offsets = p["send_offsets"]
        self.recv_offsets = p["recv_offsets"]
        self.recv_slot = p["recv_slot"]
        self.peer_send = p["peer_send"]
        self.peer_recv = p["peer_recv"]
        self.local = owned_experts(experts, world, rank)

    @property
    def recv_rows(self) -> int:
        return int(self.recv_offsets[-1])

    def segments_out(self):
        """(peer, first row in this rank's x_perm, rows, expert) of every
        non-empty segment this rank sends, ascending expert per peer."""
        for h in range(self.world):
            for e in owned_experts(self.experts, self.world, h):
                c = int(self.counts_all[self.rank, e])
                if c:
                    yield h, int(self.send_offsets[e]), c, e

    def segments_in(self):
        """(source, first row in the receive buffer, rows, expert) of every
        non-empty segment this rank receives, ascending expert per source."""
        e0 = self.local.start
        for s in range(self.world):
            for j in range(len(self.local)):
                c = int(self.counts_all[s, e0 + j])
                if c:
                    yield s, int(self.recv_slot[s, j]), c, e0 + j


def exchange_counts(transport, counts: torch.Tensor, experts: int, capacity: int) -> ExchangePlan:
    """Steps 2-3: all-gather the per-expert counts and plan the segments."""
    counts_all = transport.all_gather(counts.to(torch.int32)).cpu().numpy()
    return ExchangePlan(experts, transport.world, transport.rank, capacity, counts_all)


def exchange_dispatch(transport, plan: ExchangePlan, x_perm: torch.Tensor) -> torch.Tensor:
    """Step 4: every segment of this rank's x_perm to its owner; returns the
    receive buffer [recv_rows, H], expert-contiguous for the local experts."""
    if plan.status != N.MOE_OK:
        raise N.MoEError(plan.status, "exchange_dispatch")
    x_recv = torch.empty((plan.recv_rows,) + tuple(x_perm.shape[1:]), dtype=x_perm.dtype, device=x_perm.device)
    slot = {(s, e): r for s, r, c, e in plan.segments_in()}
    sends, recvs = [], []
    for h, r, c, e in plan.segments_out():
        if h == plan.rank:
            d = slot[(h, e)]
            x_recv[d:d + c].copy_(x_perm[r:r + c])
        else:
            sends.append((h, x_perm[r:r + c], e))
    for s, r, c, e in plan.segments_in():
        if s != plan.rank:
            recvs.append((s, x_recv[r:r + c], e))
    transport.exchange(sends, recvs)
    return x_recv


def exchange_combine(transport, plan: ExchangePlan, y_recv: torch.Tensor) -> torch.Tensor:
    """Step 6: the mirror image -- the local experts' outputs back to their
    sources; returns this rank's y_perm [its dispatched rows, H], in its own
    dispatch order (the order moe_combine reads through dest)."""
    if plan.status != N.MOE_OK:
        raise N.MoEError(plan.status, "exchange_combine")
    rows = int(plan.send_offsets[-1])
    y_perm = torch.empty((rows,) + tuple(y_recv.shape[1:]), dtype=y_recv.dtype, device=y_recv.device)
    src = {(h, e): r for h, r, c, e in plan.segments_out()}
    sends, recvs = [], []
    for s, r, c, e in plan.segments_in():
        if s == plan.rank:
            d = src[(s, e)]
            y_perm[d:d + c].copy_(y_recv[r:r + c])
        else:
            sends.append((s, y_recv[r:r + c], e))
    for h, r, c, e in plan.segments_out():
        if h != plan.rank:
            recvs.append((h, y_perm[r:r + c], e))
    transport.exchange(sends, recvs)
    return y_perm


class ExpertParallelLayer:
    """One MoE layer whose routed experts are split over the ranks of a transport.

    w13_local [el, up, H] and w2_local [el, H, I] are this rank's experts
    (owned_experts(E, world, rank)), BF16 on this rank's GPU.  A call takes this
    rank's tokens (x [T, H] BF16, router logits [T, E] FP32) and returns their
    layer output [T, H]: route, dispatch, exchange, local expert FFN, exchange
    back, combine.  capacity bounds the rows any one expert receives from all
    ranks together (0: the global token count)."""

    def __init__(self, transport, hidden, experts, top_k, inter, w13_local, w2_local, act=N.MOE_ACT_SWIGLU,
                 capacity=0):
        self.t = transport
        self.H, self.E, self.k, self.I, self.act = hidden, experts, top_k, inter, act
        self.capacity = capacity
        self.local = owned_experts(experts, transport.world, transport.rank)
        assert w13_local.shape[0] == len(self.local) and w2_local.shape[0] == len(self.local)
        self.w13, self.w2 = w13_local, w2_local

    def __call__(self, x: torch.Tensor, logits: torch.Tensor, stream=None) -> torch.Tensor:
        dev = x.device
        T = x.shape[0]
        tokens = self.t.all_gather(torch.tensor([T], dtype=torch.int32, device=dev)).sum().item()
        cap = self.capacity if self.capacity > 0 else max(int(tokens), 1)
        shape = N.make_shape(T, self.H, self.E, self.k, self.I, self.act, capacity=cap)
        ws = N.workspace(shape, dev)
        R = T * self.k
        ids = torch.empty(T, self.k, dtype=torch.int32, device=dev)
        w = torch.empty(T, self.k, dtype=torch.float32, device=dev)
        counts = torch.empty(self.E, dtype=torch.int32, device=dev)
        offsets = torch.empty(self.E + 1, dtype=torch.int32, device=dev)
        dest = torch.empty(R, dtype=torch.int32, device=dev)
        sp = torch.empty(R, dtype=torch.int32, device=dev)
        x_perm = torch.empty(R, self.H, dtype=torch.bfloat16, device=dev)
        N.moe_route(shape, logits, ids, w, ws, stream)
        N.moe_dispatch(shape, x, ids, counts, offsets, dest, sp, x_perm, ws, stream)
        st = N.moe_status_read(ws, stream)
        if st != N.MOE_OK:
            raise N.MoEError(st, "ExpertParallelLayer: route / dispatch")
        plan = exchange_counts(self.t, counts, self.E, cap)
        if plan.status != N.MOE_OK:
            raise N.MoEError(plan.status, "ExpertParallelLayer: exchange plan")
        x_recv = exchange_dispatch(self.t, plan, x_perm)
        y_recv = torch.empty_like(x_recv)
        rows = plan.recv_rows
        if rows > 0:
            lshape = N.make_shape(rows, self.H, len(self.local), 1, self.I, self.act, capacity=rows)
            lws = N.workspace(lshape, dev)
            h = torch.empty(rows, self.I, dtype=torch.bfloat16, device=dev)
            roff = torch.from_numpy(plan.recv_offsets).to(dev)
            N.moe_expert_ffn(lshape, x_recv, roff, self.w13, self.w2, None, None, None, h, y_recv, None, lws, stream)
            st = N.moe_status_read(lws, stream)
            if st != N.MOE_OK:
                raise N.MoEError(st, "ExpertParallelLayer: expert FFN")
        y_perm = exchange_combine(self.t, plan, y_recv)
        out = torch.empty(T, self.H, dtype=torch.bfloat16, device=dev)
        N.moe_combine(shape, y_perm, dest, w, None, out, ws, stream)
        st = N.moe_status_read(ws, stream)
        if st != N.MOE_OK:
            raise N.MoEError(st, "ExpertParallelLayer: combine")
        return out
