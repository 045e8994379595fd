"""The expert-parallel count-first exchange on CPU ranks (gloo; world sizes 2
and 4), checked against the one-process layer of the concatenated batch.

Each rank routes and dispatches its own tokens with the oracle (the GPU kernels
are not available here), then the product's exchange -- count all-gather,
moe_ep_plan, point-to-point segments -- moves the rows.  The receive buffer
must equal, bit for bit, the slice of the one-process x_perm that holds the
rank's experts, with the same bucket bounds; the oracle's expert FFN on the
local experts, sent back and combined, must give the one-process layer output
bit for bit; a capacity overflow must stop the payload on every rank at once.
(afdEP-comm count-first validation record, .change / .setup.)
"""
import multiprocessing as mp
import os
import socket
import sys
import traceback

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs(case):
    """The concatenated batch, identical on every rank (seeded)."""
    import torch

    from mixture_experts_routing_router_gb300 import synth
    T = sum(case["tokens"])
    E, H, I, act = case["experts"], case["hidden"], case["inter"], case["act"]
    wl = synth.Workload("ep", T, H, E, case["top_k"], I, act=act)
    logits = synth.normal((T, E), 1.0, 5, "logits", "cpu", torch.float32).numpy()
    x = synth.bf16_bits(synth.normal((T, H), 1.0, 5, "x", "cpu"))
    w13 = np.stack([synth.bf16_bits(synth.expert_weights(wl, e, 5, "cpu", True)[0]) for e in range(E)])
    w2 = np.stack([synth.bf16_bits(synth.expert_weights(wl, e, 5, "cpu", True)[1]) for e in range(E)])
    return logits, x, w13, w2


def _rank(rank, world, port, case, q):
    try:
        os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        import torch
        import torch.distributed as dist

        import oracle
        from mixture_experts_routing_router_gb300 import ep
        from mixture_experts_routing_router_gb300 import native as N
        dist.init_process_group("gloo", rank=rank, world_size=world)
        E, k, act = case["experts"], case["top_k"], case["act"]
        logits, x, w13, w2 = _inputs(case)
        T = logits.shape[0]
        lo = sum(case["tokens"][:rank])
        hi = lo + case["tokens"][rank]
        # this rank's routing and dispatch (the oracle stands in for the kernels)
        _, ids, w = oracle.route(logits[lo:hi], k)
        _, counts, offsets, dest, sp, x_perm = oracle.dispatch(ids, x[lo:hi], E, hi - lo)
        t = ep.TorchDistTransport()
        plan = ep.exchange_counts(t, torch.from_numpy(counts), E, case["capacity"])
        if plan.status != N.MOE_OK:
            with pytest.raises(N.MoEError):
                ep.exchange_dispatch(t, plan, torch.from_numpy(x_perm.view(np.int16)))
            q.put((rank, "status", int(plan.status)))
            dist.destroy_process_group()
            return
        assert np.array_equal(plan.send_offsets, offsets)
        x_recv = ep.exchange_dispatch(t, plan, torch.from_numpy(x_perm.view(np.int16)))
        # the one-process dispatch of the concatenated batch
        _, ids_g, w_g = oracle.route(logits, k)
        _, counts_g, off_g, _, _, xp_g = oracle.dispatch(ids_g, x, E, T)
        e0, e1 = plan.local.start, plan.local.stop
        assert np.array_equal(x_recv.numpy().view(np.uint16), xp_g[off_g[e0]:off_g[e1]])
        assert np.array_equal(plan.recv_offsets, off_g[e0:e1 + 1] - off_g[e0])
        # the round trip returns this rank's x_perm
        back = ep.exchange_combine(t, plan, x_recv)
        assert np.array_equal(back.numpy().view(np.uint16), x_perm[:offsets[-1]])
        # the local experts' FFN (oracle), back to the sources, combined
        _, y_recv, _, _ = oracle.expert_ffn(x_recv.numpy().view(np.uint16), plan.recv_offsets, w13[e0:e1],
                                            w2[e0:e1], act)
        y_perm = ep.exchange_combine(t, plan, torch.from_numpy(y_recv.view(np.int16)))
        out = oracle.combine(y_perm.numpy().view(np.uint16), dest, w)
        ref = oracle.layer(x, w13, w2, act, k, T, logits=logits)
        assert np.array_equal(out, ref["out"][lo:hi])
        q.put((rank, "ok", int(plan.recv_rows)))
        dist.destroy_process_group()
    except Exception:
        q.put((rank, "error", traceback.format_exc()))


def _run(world, case):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
    errs = [r for r in res if r[1] == "error"]
    assert not errs, errs[0][2]
    return sorted(res)


CASES = {
    "w2_swiglu": (2, dict(tokens=[13, 20], experts=8, top_k=2, hidden=64, inter=48, act=0, capacity=1000)),
    "w4_uneven_experts": (4, dict(tokens=[5, 11, 1, 9], experts=10, top_k=3, hidden=32, inter=40, act=1,
                                  capacity=1000)),
    "w4_k_eq_e": (4, dict(tokens=[3, 4, 2, 6], experts=4, top_k=4, hidden=16, inter=16, act=0, capacity=1000)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_exchange_matches_one_process_layer(name):
    world, case = CASES[name]
    res = _run(world, case)
    assert all(r[1] == "ok" for r in res)
    # every routed pair lands on exactly one rank
    assert sum(r[2] for r in res) == sum(case["tokens"]) * case["top_k"]


def test_capacity_overflow_stops_every_rank():
    # 40 tokens top-2 of 4 experts: some expert receives more than 12 rows
    case = dict(tokens=[10, 10, 10, 10], experts=4, top_k=2, hidden=16, inter=16, act=0, capacity=12)
    res = _run(4, case)
    from mixture_experts_routing_router_gb300 import native as N
    assert all(r[1] == "status" and r[2] == N.MOE_ERR_CAPACITY for r in res)


def test_plan_host_arithmetic():
    """moe_ep_plan on a hand-made count matrix (two ranks, five experts:
    rank 0 owns experts 0-1, rank 1 owns 2-4)."""
    from mixture_experts_routing_router_gb300 import build as B
    from mixture_experts_routing_router_gb300 import native as N
    B.build()
    c = np.array([[1, 2, 0, 3, 4], [0, 1, 1, 1, 0]], np.int32)
    st, p = N.moe_ep_plan(5, 2, 0, 100, c)
    assert st == N.MOE_OK
    assert p["send_offsets"].tolist() == [0, 1, 3, 3, 6, 10]
    assert p["recv_offsets"].tolist() == [0, 1, 4]
    assert p["recv_slot"].tolist() == [[0, 1], [1, 3]]
    assert p["peer_send"].tolist() == [3, 7] and p["peer_recv"].tolist() == [3, 1]
    st, p = N.moe_ep_plan(5, 2, 1, 100, c)
    assert p["recv_offsets"].tolist() == [0, 1, 5, 9]
    assert p["recv_slot"].tolist() == [[0, 1, 5], [0, 4, 9]]
    assert N.moe_ep_plan(5, 2, 1, 3, c)[0] == N.MOE_ERR_CAPACITY      # expert 3 gets 4 > 3
    with pytest.raises(N.MoEError):
        N.moe_ep_plan(5, 2, 2, 100, c)
    with pytest.raises(N.MoEError):
        N.moe_ep_plan(5, 2, 0, 100, np.array([[1, -2, 0, 3, 4], [0, 1, 1, 1, 0]], np.int32))
