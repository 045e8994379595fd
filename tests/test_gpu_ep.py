"""The expert-parallel layer on one GPU: virtual ranks as threads of one
process, each with its own CUDA stream, exchanging rows through device copies
(a transport of the test; the layer's own transport is torch.distributed).

Every rank's output must equal, bit for bit, the one-process moe_layer of the
concatenated batch (each routed row goes through the same kernels' FP32 sums
in either case), and the oracle within the tolerance.  The kernels of
different virtual ranks never wait on one another: every exchange is a host
barrier between complete stream synchronisations.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routing_router_gb300 import ep
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

from gpu_util import assert_close, bits, dev, inputs, run_layer

pytestmark = pytest.mark.gpu


class Hub:
    def __init__(self, world):
        self.world = world
        self.barrier = threading.Barrier(world, timeout=120)
        self.slots = [None] * world
        self.mail = {}
        self.lock = threading.Lock()


class ThreadTransport:
    def __init__(self, hub, rank):
        self.hub, self.rank, self.world = hub, rank, hub.world

    def all_gather(self, t):
        torch.cuda.current_stream().synchronize()
        self.hub.slots[self.rank] = t.clone()
        self.hub.barrier.wait()
        out = torch.stack([s.to(t.device) for s in self.hub.slots])
        torch.cuda.current_stream().synchronize()
        self.hub.barrier.wait()
        return out

    def exchange(self, sends, recvs):
        torch.cuda.current_stream().synchronize()
        with self.hub.lock:
            for peer, t, tag in sends:
                self.hub.mail.setdefault((self.rank, peer, tag), []).append(t)
        self.hub.barrier.wait()
        for peer, t, tag in recvs:
            with self.hub.lock:
                src = self.hub.mail[(peer, self.rank, tag)].pop(0)
            t.copy_(src)
        torch.cuda.current_stream().synchronize()
        self.hub.barrier.wait()


def run_ep(wl, g, tokens):
    world = len(tokens)
    hub = Hub(world)
    cuts = np.cumsum([0] + tokens)
    outs, errs = [None] * world, []

    def body(r):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                el = ep.owned_experts(wl.experts, world, r)
                layer = ep.ExpertParallelLayer(ThreadTransport(hub, r), wl.hidden, wl.experts, wl.top_k, wl.inter,
                                               g["w13"][el.start:el.stop].contiguous(),
                                               g["w2"][el.start:el.stop].contiguous(), wl.act)
                lo, hi = cuts[r], cuts[r + 1]
                # copies: a row slice of x or logits need not start on a 16-byte boundary
                outs[r] = layer(g["x"][lo:hi].clone(), g["logits"][lo:hi].clone())
                s.synchronize()
        except Exception as e:          # surface the first failure, release the others
            errs.append(e)
            hub.barrier.abort()

    th = [threading.Thread(target=body, args=(r,)) for r in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    if errs:
        raise errs[0]
    return outs


CASES = {
    # small buckets (small-row kernel in both layers)
    "w4_decode_sized": (synth.Workload("ep_a", 41, 256, 16, 2, 128), [12, 9, 1, 19]),
    # uneven expert blocks, ReLU^2, single-CTA tile kernels
    "w4_relu2": (synth.Workload("ep_b", 500, 128, 10, 3, 136, act=synth.ACT_RELU2), [150, 7, 200, 143]),
    # 256+ rows per expert (the CTA-pair kernel in the one-process layer)
    "w2_pair_rows": (synth.Workload("ep_c", 1200, 256, 4, 2, 200), [700, 500]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_expert_parallel_layer_equals_one_process_layer(name):
    wl, tokens = CASES[name]
    assert sum(tokens) == wl.tokens
    g = inputs(wl, unit_scale=True, seed=17)
    outs = run_ep(wl, g, tokens)
    full, st = run_layer(wl, g)
    assert st == N.MOE_OK
    got = torch.cat(outs)
    assert torch.equal(got.view(torch.int16), full.view(torch.int16))
    ref = oracle.layer(bits(g["x"]), bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, wl.cap,
                       logits=g["logits"].cpu().numpy())
    assert_close(bits(got), ref["out"], f"{name} expert-parallel out")
