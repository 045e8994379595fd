"""The bounded-wait give-up path and the capacity gate of moe_layer, on the GPU.

Failure is made on the host, never by faulting the GPU: the count kernel's
look-back wait is shortened for the test (moe_workspace_set_wait) and the
count kernel is told to hand out tile ids from 1, so tile 0's counts are never
published and the look-back of tile 1 waits for a flag nothing sets (the
afdEP-comm count-first record's bounded timeout_while spins and its must-fail
case of counts that never arrive, .faults_shipped).  The wait must give up
within its limit with MOE_ERR_TIMEOUT at the look-back site, every kernel must
return, and the same workspace must then dispatch to parity again.  The GEMM
roles' bounded waits are not forced here: they hold tensor-core work and bulk
copies in flight, and their give-up paths are reviewed by reading.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

from gpu_util import alloc_stage_outputs, assert_close, bits, dev, i32_dev, inputs

pytestmark = pytest.mark.gpu

SITE_LOOKBACK = 1


def _ids(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int().numpy()


def _dispatch(shape, wl, x_dev, ids_np, ws):
    o = alloc_stage_outputs(wl)
    N.moe_dispatch(shape, x_dev, i32_dev(ids_np), o["counts"], o["offsets"], o["dest"], o["sorted_pair"],
                   o["x_perm"], ws)
    return o


def _check_dispatch(o, x_dev, ids_np, E, cap):
    st, counts, offsets, dest, sp, xp = oracle.dispatch(ids_np, bits(x_dev), E, cap)
    assert st == 0
    assert np.array_equal(o["counts"].cpu().numpy(), counts)
    assert np.array_equal(o["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(o["dest"].cpu().numpy(), dest)
    assert np.array_equal(o["sorted_pair"].cpu().numpy(), sp)
    assert torch.equal(o["x_perm"].view(torch.int16), torch.from_numpy(xp.view(np.int16)).to(dev()))


@pytest.mark.parametrize("E,k", [(16, 4), (300, 8)])
def test_lookback_wait_gives_up_and_the_workspace_recovers(E, k):
    wl = synth.Workload("lookback", 1500, 64, E, k, 64)    # 6000 / 12000 pairs: 6 / 12 count tiles
    ids = _ids(wl.tokens, E, k, seed=E)
    x_dev = synth.normal((wl.tokens, wl.hidden), 1.0, 8, "x", dev())
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())

    # must pass: a short limit on a normal dispatch still gives parity
    N.moe_workspace_set_wait(ws, 5_000_000, 0)
    o = _dispatch(shape, wl, x_dev, ids, ws)
    assert N.moe_timeout_site_read(ws) == 0
    assert N.moe_status_read(ws) == N.MOE_OK
    _check_dispatch(o, x_dev, ids, E, wl.cap)

    # must fail: tile 0 never publishes; the wait runs out after 1 ms
    N.moe_workspace_set_wait(ws, 1_000_000, 1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _dispatch(shape, wl, x_dev, ids, ws)
    site = N.moe_timeout_site_read(ws)          # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert site == SITE_LOOKBACK
    assert N.moe_status_read(ws) == N.MOE_ERR_TIMEOUT
    # (E / 256) columns per thread, each giving up after 1 ms; the default
    # 2 s limit would take far longer
    assert elapsed < 0.5, elapsed

    # the status and site were cleared by the read, and the workspace works again
    N.moe_workspace_set_wait(ws, 0, 0)
    o = _dispatch(shape, wl, x_dev, ids, ws)
    assert N.moe_timeout_site_read(ws) == 0
    assert N.moe_status_read(ws) == N.MOE_OK
    _check_dispatch(o, x_dev, ids, E, wl.cap)


def test_lookback_timeout_inside_the_layer():
    """A layer whose dispatch timed out still runs every kernel to its end
    (the GEMMs and the combine on the partial placement, all in bounds), and
    the next call on the same workspace matches the oracle."""
    wl = synth.Workload("lookback_layer", 600, 128, 16, 4, 64)     # 2400 pairs: 3 count tiles
    g = inputs(wl, unit_scale=True, seed=9)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_workspace_set_wait(ws, 1_000_000, 1)
    N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_timeout_site_read(ws) == SITE_LOOKBACK
    assert N.moe_status_read(ws) == N.MOE_ERR_TIMEOUT
    N.moe_workspace_set_wait(ws, 0, 0)
    N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    ref = oracle.layer(bits(g["x"]), bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, wl.cap,
                       logits=g["logits"].cpu().numpy())
    assert_close(bits(out), ref["out"], "layer after a timeout")


def test_set_wait_rejects_bad_arguments():
    wl = synth.Workload("args", 8, 64, 4, 2, 64)
    ws = N.workspace(N.shape_of(wl), dev())
    for skip in (-1, 2):
        with pytest.raises(N.MoEError) as e:
            N.moe_workspace_set_wait(ws, 0, skip)
        assert e.value.status == N.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("tokens", [8, 300])     # the fused small-batch dispatch, and the count kernel
def test_layer_over_capacity_leaves_out_and_residual_untouched(tokens):
    """MOE_ERR_CAPACITY moves no payload, and inside moe_layer the expert GEMMs
    and the combine then do nothing: an output that aliases the residual keeps
    the residual, bit for bit."""
    wl = synth.Workload("cap_layer", tokens, 64, 8, 2, 64, shared=1, shared_inter=32)
    g = inputs(wl, unit_scale=True, seed=13)
    ids = torch.zeros(tokens, 2, dtype=torch.int32, device=dev())
    ids[:, 1] = 1
    w = torch.full((tokens, 2), 0.5, device=dev())
    shape = N.shape_of(wl)
    shape.capacity = tokens // 2                     # every token on experts 0 and 1
    ws = N.workspace(shape, dev())
    res = synth.normal((tokens, wl.hidden), 1.0, 13, "residual", dev())
    keep = res.clone()
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], g["ws13"], g["ws2"], res, ws, residual=res)
    assert N.moe_status_read(ws) == N.MOE_ERR_CAPACITY
    assert torch.equal(res.view(torch.int16), keep.view(torch.int16))
    # logits routed through the layer with too small a capacity: same verdict
    N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], g["ws13"], g["ws2"], res, ws,
                residual=res)
    st = N.moe_status_read(ws)
    if st == N.MOE_ERR_CAPACITY:
        assert torch.equal(res.view(torch.int16), keep.view(torch.int16))
    else:
        assert st == N.MOE_OK
    # within capacity the same workspace gives the oracle's output again
    shape.capacity = tokens
    out = torch.empty_like(res)
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], g["ws13"], g["ws2"], out, ws, residual=keep)
    assert N.moe_status_read(ws) == N.MOE_OK
    ref = oracle.layer(bits(g["x"]), bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, tokens,
                       ids_in=ids.cpu().numpy(), w_in=w.cpu().numpy(), ws13=bits(g["ws13"]), ws2=bits(g["ws2"]),
                       residual=bits(keep))
    assert_close(bits(out), ref["out"], "layer within capacity")


def test_fused_decode_layer_over_capacity_leaves_out_and_residual_untouched():
    """The same at 8 tokens without shared experts, where the expert FFN and
    the combine run as one kernel after the fused dispatch."""
    wl = synth.Workload("cap_fused", 8, 128, 8, 2, 64)
    g = inputs(wl, unit_scale=True, seed=14)
    ids = torch.zeros(8, 2, dtype=torch.int32, device=dev())
    ids[:, 1] = 1
    w = torch.full((8, 2), 0.5, device=dev())
    shape = N.shape_of(wl)
    shape.capacity = 4
    ws = N.workspace(shape, dev())
    res = synth.normal((8, wl.hidden), 1.0, 14, "residual", dev())
    keep = res.clone()
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], None, None, res, ws, residual=res)
    assert N.moe_status_read(ws) == N.MOE_ERR_CAPACITY
    assert torch.equal(res.view(torch.int16), keep.view(torch.int16))
    # and the workspace runs a valid call afterwards
    shape.capacity = 8
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], None, None, res, ws, residual=res)
    assert N.moe_status_read(ws) == N.MOE_OK
