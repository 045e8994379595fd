"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (no cudaMalloc available to them, so no workspace).
Its scratch is a static device array inside libmoe.so.

The GPU test calls it twice in a row, on different inputs, through the C ABI
and compares each result with moe_dispatch (the workspace entry point) on the
same inputs: counts, offsets, dest, sorted_pair and x_perm must be identical
(integer and copy outputs: bit-exact is the tolerance).  The second call also
shows that the array's left-over contents from the first call do not leak.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_routing_router_gb300 import build as B
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth


def _route_ids(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    logits[:, : max(1, E // 16)] += 1.5          # a few hot experts: uneven buckets
    return torch.topk(logits, k, dim=1).indices.to(torch.int32)


def _both(T, H, E, k, seed):
    dev = torch.device("cuda:0")
    shape = N.make_shape(T, H, E, k, 64)
    x = synth.normal((T, H), 1.0, seed, "x", dev)
    ids = _route_ids(T, E, k, seed).to(dev)
    R = T * k

    def outs():
        return dict(counts=torch.full((E,), -9, dtype=torch.int32, device=dev),
                    offsets=torch.full((E + 1,), -9, dtype=torch.int32, device=dev),
                    dest=torch.full((R,), -9, dtype=torch.int32, device=dev),
                    sorted_pair=torch.full((R,), -9, dtype=torch.int32, device=dev),
                    x_perm=torch.zeros(R, H, dtype=torch.bfloat16, device=dev))

    ref = outs()
    ws = N.workspace(shape, dev)
    N.moe_dispatch(shape, x, ids, ref["counts"], ref["offsets"], ref["dest"], ref["sorted_pair"], ref["x_perm"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    got = outs()
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    N.moe_dispatch_noalloc(shape, x, ids, got["counts"], got["offsets"], got["dest"], got["sorted_pair"],
                           got["x_perm"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == N.MOE_OK
    for key in ("counts", "offsets", "dest", "sorted_pair"):
        assert torch.equal(got[key], ref[key]), key
    assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))
    return got


@pytest.mark.gpu
def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    torch.cuda.set_device(0)
    # first call: many count tiles, 128 experts
    a = _both(T=2048, H=256, E=128, k=8, seed=1)
    # second call right after: different sizes and expert count, fewer tiles,
    # so stale look-back state from the first call would show
    b = _both(T=700, H=136, E=37, k=5, seed=2)
    assert a["offsets"][-1].item() == 2048 * 8 and b["offsets"][-1].item() == 700 * 5


def test_noalloc_rejects_sizes_beyond_its_limit():
    B.build()
    L = N.lib()
    shape = N.make_shape(16385, 256, 256, 8, 64)      # 131080 pairs > 131072
    p = ctypes.c_void_p(1 << 20)                      # never dereferenced: rejected first
    st = L.moe_dispatch_noalloc(ctypes.byref(shape), p, p, p, p, p, p, p, None, None)
    assert st == N.MOE_ERR_UNSUPPORTED
    assert "exceed" in N.last_error_message()
