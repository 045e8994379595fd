"""Guard bands: no kernel writes outside the buffers it is given.

Every output buffer (and the workspace) is carved out of a larger allocation
with 4 KiB canary bands before and after it, filled with a byte pattern.  The
calls then run on the error and edge paths -- the four invalid-route kinds
(ONNX Runtime PR #33963, Description: malformed-route isolation; afdEP-comm
runner: negative / wide / duplicate / dummy routes), a capacity overflow,
ragged hidden and intermediate sizes, k = E, the largest E and k, one token,
the fused small-batch dispatch, quantized weights -- and every band must be
intact afterwards.  This is the out-of-bounds check that stands in for a
memory checker.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

from gpu_util import assert_close, bits, dev, inputs

pytestmark = pytest.mark.gpu

BAND = 4096
CANARY = 0xA5


class Guarded:
    """A tensor of the given shape and dtype, with canary bands around it."""

    def __init__(self, shape, dtype, fill=None):
        itemsize = torch.empty(0, dtype=dtype).element_size()
        n = math.prod(shape) * itemsize
        self.buf = torch.full((BAND + n + BAND,), CANARY, dtype=torch.uint8, device=dev())
        self.t = self.buf[BAND:BAND + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        return bool(torch.all(self.buf[:BAND] == CANARY)) and bool(torch.all(self.buf[-BAND:] == CANARY))


def guarded_workspace(shape):
    n = N.moe_workspace_size(shape)
    g = Guarded((n,), torch.uint8)
    g.t.zero_()
    return g


def stage_buffers(wl):
    T, H, E, k, I = wl.tokens, wl.hidden, wl.experts, wl.top_k, wl.inter
    R = T * k
    return dict(ids=Guarded((T, k), torch.int32), w=Guarded((T, k), torch.float32),
                counts=Guarded((E,), torch.int32), offsets=Guarded((E + 1,), torch.int32),
                dest=Guarded((R,), torch.int32), sorted_pair=Guarded((R,), torch.int32),
                x_perm=Guarded((R, H), torch.bfloat16), h=Guarded((R, I), torch.bfloat16),
                y_perm=Guarded((R, H), torch.bfloat16),
                y_shared=Guarded((T, H), torch.bfloat16) if wl.shared else None,
                out=Guarded((T, H), torch.bfloat16))


def all_intact(bufs, what):
    bad = [name for name, b in bufs.items() if b is not None and not b.intact()]
    assert not bad, f"{what}: canary bands overwritten around {bad}"


def run_stages(wl, g, ids_dev=None, w_dev=None, capacity=None):
    """route (unless ids are given), dispatch, expert FFN and combine, every
    output guarded; -> (buffers, the device status after each stage)."""
    shape = N.shape_of(wl)
    if capacity is not None:
        shape.capacity = capacity
    b = stage_buffers(wl)
    wsg = guarded_workspace(shape)
    ws = wsg.t
    sts = []
    if ids_dev is None:
        N.moe_route(shape, g["logits"], b["ids"].t, b["w"].t, ws)
        sts.append(N.moe_status_read(ws))
    else:
        b["ids"].t.copy_(ids_dev)
        b["w"].t.copy_(w_dev)
    N.moe_dispatch(shape, g["x"], b["ids"].t, b["counts"].t, b["offsets"].t, b["dest"].t, b["sorted_pair"].t,
                   b["x_perm"].t, ws)
    sts.append(N.moe_status_read(ws))
    N.moe_expert_ffn(shape, b["x_perm"].t, b["offsets"].t, g["w13"], g["w2"], g["x"], g.get("ws13"), g.get("ws2"),
                     b["h"].t, b["y_perm"].t, None if b["y_shared"] is None else b["y_shared"].t, ws)
    sts.append(N.moe_status_read(ws))
    N.moe_combine(shape, b["y_perm"].t, b["dest"].t, b["w"].t, None if b["y_shared"] is None else b["y_shared"].t,
                  b["out"].t, ws)
    sts.append(N.moe_status_read(ws))
    b["workspace"] = wsg
    return b, sts


def run_layer_guarded(wl, g, ids_dev=None, w_dev=None, capacity=None, residual=None):
    shape = N.shape_of(wl)
    if capacity is not None:
        shape.capacity = capacity
    wsg = guarded_workspace(shape)
    out = Guarded((wl.tokens, wl.hidden), torch.bfloat16)
    if ids_dev is None:
        N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], g.get("ws13"), g.get("ws2"), out.t,
                    wsg.t, residual=residual)
    else:
        N.moe_layer(shape, None, ids_dev, w_dev, g["x"], g["w13"], g["w2"], g.get("ws13"), g.get("ws2"), out.t,
                    wsg.t, residual=residual)
    st = N.moe_status_read(wsg.t)
    return dict(out=out, workspace=wsg), st


def bad_routes(T, E, k, kind, seed=9):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    t = T // 2
    if kind == "negative":
        ids[t, k - 1] = -5
    elif kind == "wide":
        ids[t, k - 1] = E + 3
    elif kind == "duplicate":
        ids[t, k - 1] = ids[t, 0]
    else:                              # dummy: the -1 placeholder of an unused slot
        ids[t, k - 1] = -1
    ids[T - 1, 0] = 1 << 20            # and a very wide id in the last token
    w = torch.full((T, k), 1.0 / k)
    return ids.to(dev()), w.to(dev())


@pytest.mark.parametrize("kind", ["negative", "wide", "duplicate", "dummy"])
@pytest.mark.parametrize("tokens", [8, 1500])       # fused small-batch dispatch / count kernel
def test_invalid_routes_stay_in_bounds(kind, tokens):
    wl = synth.Workload("bad", tokens, 64, 16, 4, 64)
    g = inputs(wl, unit_scale=True, seed=3)
    ids, w = bad_routes(tokens, 16, 4, kind)
    b, sts = run_stages(wl, g, ids, w)
    assert sts[0] == N.MOE_ERR_INVALID_ROUTE
    all_intact(b, f"stages, {kind} route")
    lb, st = run_layer_guarded(wl, g, ids, w)
    assert st == N.MOE_ERR_INVALID_ROUTE
    all_intact(lb, f"layer, {kind} route")


@pytest.mark.parametrize("tokens", [8, 300])
def test_capacity_overflow_stays_in_bounds(tokens):
    wl = synth.Workload("cap", tokens, 64, 8, 2, 64)
    g = inputs(wl, unit_scale=True, seed=4)
    ids = torch.zeros(tokens, 2, dtype=torch.int32, device=dev())
    ids[:, 1] = 1
    w = torch.full((tokens, 2), 0.5, device=dev())
    b, sts = run_stages(wl, g, ids, w, capacity=tokens - 1)
    assert sts[0] == N.MOE_ERR_CAPACITY
    all_intact(b, "stages over capacity")
    lb, st = run_layer_guarded(wl, g, ids, w, capacity=tokens - 1)
    assert st == N.MOE_ERR_CAPACITY
    all_intact(lb, "layer over capacity")


EDGE = {
    "ragged": synth.Workload("ragged", 37, 136, 33, 5, 72),
    "ragged_relu2": synth.Workload("ragged_relu2", 53, 200, 7, 3, 264, act=synth.ACT_RELU2),
    "k_eq_e": synth.Workload("k_eq_e", 40, 128, 8, 8, 64),
    "max_e": synth.Workload("max_e", 300, 64, 1024, 32, 32),
    "t1": synth.Workload("t1", 1, 256, 16, 4, 128),
    "small_fused": synth.Workload("small_fused", 16, 200, 240, 9, 264, act=synth.ACT_RELU2),
    # the fused decode FFN (2..16 tokens, whole 64-column chunks): ragged 128-row
    # blocks of W13 and W2, both activations
    "decode_ffn_relu2": synth.Workload("decode_ffn_relu2", 7, 320, 20, 5, 192, act=synth.ACT_RELU2),
    "decode_ffn_swiglu": synth.Workload("decode_ffn_swiglu", 12, 192, 24, 6, 320),
    "shared_ragged": synth.Workload("shared_ragged", 45, 136, 12, 2, 72, shared=2, shared_inter=40),
    "pair_ragged": synth.Workload("pair_ragged", 600, 200, 3, 2, 264, act=synth.ACT_RELU2),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_shapes_stay_in_bounds_and_match(name):
    wl = EDGE[name]
    g = inputs(wl, unit_scale=True, seed=5)
    kw = dict(ws13=bits(g["ws13"]), ws2=bits(g["ws2"])) if wl.shared else {}
    ref = oracle.layer(bits(g["x"]), bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, wl.cap,
                       logits=g["logits"].cpu().numpy(), **kw)
    b, sts = run_stages(wl, g)
    assert sts == [N.MOE_OK] * 4
    all_intact(b, f"{name} stages")
    assert_close(bits(b["out"].t), ref["out"], f"{name} staged out")
    lb, st = run_layer_guarded(wl, g)
    assert st == N.MOE_OK
    all_intact(lb, f"{name} layer")
    assert torch.equal(lb["out"].t.view(torch.int16), b["out"].t.view(torch.int16))


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("tokens", [5, 300])       # small-row kernel with one chunk / many 64-row chunks
def test_quantized_layer_stays_in_bounds(fmt, tokens):
    wl = synth.Workload("q", tokens, 96 if fmt == "fp8" else 160, 12, 3, 80 if fmt == "fp8" else 96)
    g = synth.make_inputs(wl, seed=6, device=dev(), unit_scale=True, weights=False)
    shape = N.shape_of(wl)
    wsg = guarded_workspace(shape)
    out = Guarded((wl.tokens, wl.hidden), torch.bfloat16)
    if fmt == "fp8":
        q = synth.make_fp8_weights(wl, seed=6, device=dev(), unit_scale=True)
        N.moe_layer_fp8(shape, g["logits"], None, None, g["x"], q["w13"], q["s13"], q["w2"], q["s2"], out.t, wsg.t)
    else:
        q = synth.make_nvfp4_weights(wl, seed=6, device=dev(), unit_scale=True)
        N.moe_layer_nvfp4(shape, g["logits"], None, None, g["x"], q["w13"], q["b13"], q["s13"], q["w2"], q["b2"],
                          q["s2"], out.t, wsg.t)
    assert N.moe_status_read(wsg.t) == N.MOE_OK
    all_intact(dict(out=out, workspace=wsg), f"{fmt} layer")
    assert torch.all(torch.isfinite(out.t.float()))


def test_guard_detects_a_write_past_the_end():
    """The check itself: a copy one element too long is caught."""
    gb = Guarded((64,), torch.int32)
    src = torch.ones(65, dtype=torch.int32, device=dev())
    gb.buf[BAND:BAND + 65 * 4].view(torch.int32).copy_(src)
    assert not gb.intact()
    assert np.array_equal(gb.t.cpu().numpy(), np.ones(64, np.int32))
