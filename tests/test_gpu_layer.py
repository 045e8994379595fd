"""GPU parity of the whole layer (moe_layer) against the oracle, plus the
properties the pages state: internal routing equals preselected routing
bitwise (ONNX Runtime PR #33963), graph capture, determinism and batch
invariance (the RL-Kernel timestep_mlp record's batch-invariance probes)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

from gpu_util import alloc_stage_outputs, assert_close, bits, dev, inputs, run_layer
from test_gpu_stages import SMALL, oracle_stages

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS


@pytest.mark.parametrize("unit", [False, True])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_layer_small(name, unit):
    wl = SMALL[name]
    g = inputs(wl, unit_scale=unit, seed=21)
    ref = oracle_stages(wl, g)
    out, st = run_layer(wl, g)
    assert st == N.MOE_OK
    err, mref = assert_close(bits(out), ref["out"], f"{name} out")
    if unit:
        assert mref > 0.1          # the unit-scale twin is not trivially inside the floor


def test_internal_routing_equals_preselected_bitwise():
    for name in ("tiny", "decode_16_distinct", "deepseek_t96"):
        wl = SMALL[name] if name in SMALL else W[name]
        g = inputs(wl, unit_scale=True, seed=2)
        shape = N.shape_of(wl)
        ws = N.workspace(shape, dev())
        ids = torch.empty(wl.tokens, wl.top_k, dtype=torch.int32, device=dev())
        w = torch.empty(wl.tokens, wl.top_k, dtype=torch.float32, device=dev())
        N.moe_route(shape, g["logits"], ids, w, ws)
        a, sa = run_layer(wl, g)
        b, sb = run_layer(wl, g, preselected=(ids, w))
        assert sa == sb == N.MOE_OK
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layer_is_deterministic_and_graph_capturable():
    wl = W["count_first"].with_(tokens=512)
    g = inputs(wl, unit_scale=True, seed=3)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws, s)
    s.synchronize()
    eager = out.clone()
    for _ in range(2):
        with torch.cuda.stream(s):
            N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws, s)
        s.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    graph = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(graph, stream=s):
        N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws, s)
    for _ in range(4):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert N.moe_status_read(ws) == N.MOE_OK


def test_batch_invariance():
    """A token's output row does not depend on which other tokens share the
    call: the first 100 tokens alone give the same rows as in the full batch."""
    wl = W["deepseek"].with_(tokens=600)
    g = inputs(wl, unit_scale=True, seed=4)
    full, st = run_layer(wl, g)
    assert st == 0
    sub = wl.with_(tokens=100)
    gs = dict(g)
    gs["x"] = g["x"][:100].contiguous()
    gs["logits"] = g["logits"][:100].contiguous()
    part, st = run_layer(sub, gs)
    assert st == 0
    assert torch.equal(part.view(torch.int16), full[:100].view(torch.int16))


def test_layer_error_statuses():
    wl = SMALL["tiny"]
    g = inputs(wl, seed=5)
    lg = g["logits"].clone()
    lg[3, 4] = float("nan")
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_layer(shape, lg, None, None, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_ERR_NONFINITE
    # preselected ids with a wide route: invalid-route status, no fault
    ids = torch.zeros(wl.tokens, wl.top_k, dtype=torch.int32, device=dev())
    ids[:, 1] = 1
    ids[5, 1] = 16
    w = torch.full((wl.tokens, wl.top_k), 0.5, device=dev())
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_ERR_INVALID_ROUTE
    # capacity exceeded: every token on experts 0 and 1 with capacity 32 < 64
    shape.capacity = 32
    ids[5, 1] = 1
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_ERR_CAPACITY
    # host-side errors raise at once
    with pytest.raises(N.MoEError) as e:
        N.moe_layer(shape, None, ids, None, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert e.value.status == N.MOE_ERR_INVALID_ARG
    # and the workspace is still usable afterwards
    shape.capacity = wl.tokens
    N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_OK


def test_layer_with_residual():
    wl = SMALL["deepseek_t96"]
    g = inputs(wl, unit_scale=True, seed=31)
    res = synth.normal((wl.tokens, wl.hidden), 1.0, 31, "residual", dev())
    ref = oracle.layer(bits(g["x"]), bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, wl.cap,
                       logits=g["logits"].cpu().numpy(), ws13=bits(g["ws13"]), ws2=bits(g["ws2"]),
                       residual=bits(res))
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], g["ws13"], g["ws2"], out, ws,
                residual=res)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), ref["out"], "layer + residual")


def test_layer_error_statuses_small_batch():
    """The same device errors at 8 tokens, where routing, counting and the
    scatter run as one fused kernel: non-finite logits, invalid preselected
    routes, and a capacity overflow that moves no payload."""
    wl = synth.Workload("small_err", 8, 64, 16, 2, 64)
    g = inputs(wl, seed=6)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    lg = g["logits"].clone()
    lg[2, 5] = float("inf")
    N.moe_layer(shape, lg, None, None, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_ERR_NONFINITE
    ids = torch.zeros(wl.tokens, wl.top_k, dtype=torch.int32, device=dev())
    ids[:, 1] = 1
    w = torch.full((wl.tokens, wl.top_k), 0.5, device=dev())
    for bad in (-1, 16, 0):                         # negative, wide, duplicate of slot 0
        ids2 = ids.clone()
        ids2[3, 1] = bad
        N.moe_layer(shape, None, ids2, w, g["x"], g["w13"], g["w2"], None, None, out, ws)
        assert N.moe_status_read(ws) == N.MOE_ERR_INVALID_ROUTE
    shape.capacity = 4                              # 8 rows on experts 0 and 1
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_ERR_CAPACITY
    shape.capacity = wl.tokens
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], None, None, out, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    # a valid call afterwards matches the oracle
    ref = oracle.layer(bits(g["x"]), bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, wl.cap,
                       ids_in=ids.cpu().numpy(), w_in=w.cpu().numpy())
    assert_close(bits(out), ref["out"], "small batch after errors")


def random_workloads(n, seed):
    """Seeded small shapes across the kernels' paths: 1..300 tokens (fused,
    single-CTA and CTA-pair dispatch / GEMM paths), hidden and intermediate
    any multiple of 8, 1..64 experts, top-k up to min(E, 32), both
    activations, with and without shared experts."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 65))
        k = int(rng.integers(1, min(E, 32) + 1))
        T = int(rng.choice([1, 3, 16, 17, 64, 65, 150, 300]))
        H = int(8 * rng.integers(1, 41))
        I = int(8 * rng.integers(1, 41))
        act = int(rng.integers(0, 2))
        S = int(rng.choice([0, 0, 1, 2]))
        Is = int(8 * rng.integers(1, 21)) if S else 0
        out.append(synth.Workload(f"rand{i}", T, H, E, k, I, act=act, shared=S, shared_inter=Is))
    # and two shapes with 256+ rows per expert (the CTA-pair GEMM with swapped tails)
    out.append(synth.Workload(f"rand{n}", 300, 136, 2, 2, 120, act=1, shared=1, shared_inter=40))
    out.append(synth.Workload(f"rand{n + 1}", 300, 264, 3, 1, 200, act=0))
    return out


@pytest.mark.parametrize("wl", random_workloads(12, 2026), ids=lambda w: f"{w.name}-T{w.tokens}H{w.hidden}E{w.experts}k{w.top_k}I{w.inter}a{w.act}S{w.shared}")
def test_layer_random_shapes(wl):
    g = inputs(wl, unit_scale=True, seed=97)
    res = synth.normal((wl.tokens, wl.hidden), 1.0, 97, "residual", dev())
    kw = dict(ws13=bits(g["ws13"]), ws2=bits(g["ws2"])) if wl.shared else {}
    ref = oracle.layer(bits(g["x"]), bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, wl.cap,
                       logits=g["logits"].cpu().numpy(), residual=bits(res), **kw)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], g.get("ws13"), g.get("ws2"), out, ws,
                residual=res)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), ref["out"], f"{wl.name} layer")


# Decode-sized layers (2 to 16 tokens) run the expert FFN and the combine as
# one persistent kernel after the fused dispatch; the separate calls (route, dispatch, expert
# FFN, combine) run the small-row GEMM and the combine kernel.  Same MMA
# order, same epilogue and combine arithmetic: equal bit for bit.
FUSED = {
    "decode_2_shared": W["decode_1_shared"].with_(tokens=2, name="decode_2_shared"),
    "decode_16_distinct": W["decode_16_distinct"],
    "swiglu_t16": synth.Workload("swiglu_t16", 16, 512, 8, 2, 384),              # a partial last down stage
    "swiglu_t2_e64": synth.Workload("swiglu_t2_e64", 2, 256, 64, 8, 192),        # ragged 128-row blocks
    "relu2_t5_h320": synth.Workload("relu2_t5_h320", 5, 320, 12, 3, 64, act=synth.ACT_RELU2),
    # the ABI's largest expert count and top-k: up to 512 non-empty experts in the
    # group list, six bucket bounds per thread
    "max_e_t16": synth.Workload("max_e_t16", 16, 128, 1024, 32, 64),
    # a DeepSeek-sized hidden dimension: 112 K chunks, one-chunk-wide down stages
    "relu2_t16_h7168": synth.Workload("relu2_t16_h7168", 16, 7168, 16, 2, 256, act=synth.ACT_RELU2),
}


def staged_layer(wl, g, residual=None, preselected=None):
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    if preselected is None:
        N.moe_route(shape, g["logits"], o["ids"], o["w"], ws)
        ids, w = o["ids"], o["w"]
    else:
        ids, w = preselected
    N.moe_dispatch(shape, g["x"], ids, o["counts"], o["offsets"], o["dest"], o["sorted_pair"], o["x_perm"], ws)
    N.moe_expert_ffn(shape, o["x_perm"], o["offsets"], g["w13"], g["w2"], None, None, None, o["h"], o["y_perm"], None,
                     ws)
    N.moe_combine(shape, o["y_perm"], o["dest"], w, None, o["out"], ws, residual=residual)
    return o["out"], N.moe_status_read(ws)


@pytest.mark.parametrize("name", sorted(FUSED))
def test_decode_fused_layer_equals_separate_kernels(name):
    wl = FUSED[name]
    g = inputs(wl, unit_scale=True, seed=41)
    a, sa = run_layer(wl, g)
    b, sb = staged_layer(wl, g)
    assert sa == sb == N.MOE_OK
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref = oracle_stages(wl, g)
    assert_close(bits(a), ref["out"], f"{name} fused out")
    # in place on the residual, twice on one workspace (the counters start afresh)
    res = synth.normal((wl.tokens, wl.hidden), 1.0, 41, "residual", dev())
    want, st = staged_layer(wl, g, residual=res)
    assert st == N.MOE_OK
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    for _ in range(2):
        buf = res.clone()
        N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, buf, ws, residual=buf)
        assert N.moe_status_read(ws) == N.MOE_OK
        assert torch.equal(buf.view(torch.int16), want.view(torch.int16))


def test_decode_fused_layer_all_routes_invalid():
    """No routed row at all: the output is the residual (invalid pairs add
    nothing), as from the separate combine."""
    wl = FUSED["relu2_t5_h320"]
    g = inputs(wl, unit_scale=True, seed=42)
    ids = torch.full((wl.tokens, wl.top_k), -1, dtype=torch.int32, device=dev())
    w = torch.full((wl.tokens, wl.top_k), 0.25, device=dev())
    res = synth.normal((wl.tokens, wl.hidden), 1.0, 42, "residual", dev())
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_layer(shape, None, ids, w, g["x"], g["w13"], g["w2"], None, None, out, ws, residual=res)
    assert N.moe_status_read(ws) == N.MOE_ERR_INVALID_ROUTE
    want, st = staged_layer(wl, g, residual=res, preselected=(ids, w))
    assert st == N.MOE_ERR_INVALID_ROUTE
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert torch.equal(out.view(torch.int16), res.view(torch.int16))


def test_decode_fused_layer_graph_replays_and_alternates():
    """The fused decode FFN's counters are zeroed by each call's dispatch and
    route_ready is put back by the last CTA out: captured in a graph and
    replayed, and interleaved with a one-token layer (three separate kernels)
    on the same stream, every output stays bit for bit the eager one."""
    wl8 = FUSED["decode_2_shared"].with_(tokens=8, name="decode_8_fused")
    wl1 = FUSED["decode_2_shared"].with_(tokens=1, name="decode_1_sep")
    s = torch.cuda.Stream()
    runs = []
    for wl in (wl8, wl1):
        g = inputs(wl, unit_scale=True, seed=43)
        shape = N.shape_of(wl)
        ws = N.workspace(shape, dev())
        out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
        with torch.cuda.stream(s):
            N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws, s)
        s.synchronize()
        assert N.moe_status_read(ws) == N.MOE_OK
        runs.append((wl, g, shape, ws, out, out.clone()))
    graphs = []
    for wl, g, shape, ws, out, _ in runs:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], None, None, out, ws, s)
        graphs.append(gr)
    for _ in range(5):
        with torch.cuda.stream(s):
            for (wl, g, shape, ws, out, eager), gr in zip(runs, graphs):
                out.zero_()
                gr.replay()
        s.synchronize()
        for wl, g, shape, ws, out, eager in runs:
            assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    for wl, g, shape, ws, out, eager in runs:
        assert N.moe_status_read(ws) == N.MOE_OK
