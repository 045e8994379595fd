"""GPU parity, stage by stage, against the CPU oracle.

Routing ids, counts, offsets, dest, sorted_pair and x_perm must be bit-exact;
routing weights within 1e-5; h, y_perm, y_shared and out within
max|d| <= 1e-2 * max|ref| + 1e-3.  Each GPU stage is fed the oracle's
intermediates, so a failure points at one kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

from gpu_util import W_TOL, alloc_stage_outputs, assert_close, bits, dev, f32_dev, i32_dev, inputs, to_bf16_dev

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
DECODE = [f"decode_{r}_{k}" for r in (1, 8, 16) for k in ("shared", "distinct")]
# small and reduced workloads: the oracle finishes the whole layer in seconds,
# and they still span several tiles with ragged tails
SMALL = {
    "tiny": W["tiny"],
    "count_first_t160": W["count_first"].with_(tokens=160, name="count_first_t160"),
    "deepseek_t96": W["deepseek"].with_(tokens=96, name="deepseek_t96"),
    "ragged": synth.Workload("ragged", 37, 136, 33, 5, 72),                  # H, I not multiples of 64
    "ragged_relu2": synth.Workload("ragged_relu2", 53, 200, 7, 3, 264, act=synth.ACT_RELU2),
    "one_expert": synth.Workload("one_expert", 300, 64, 1, 1, 128),
    "k_eq_e": synth.Workload("k_eq_e", 40, 128, 8, 8, 64),
    "wide_e": synth.Workload("wide_e", 70, 64, 1000, 32, 32),
    "max_e": synth.Workload("max_e", 300, 64, 1024, 32, 32),                 # the ABI's largest E and k
    "t1": synth.Workload("t1", 1, 256, 16, 4, 128),
    "shared3": synth.Workload("shared3", 50, 128, 12, 2, 64, shared=3, shared_inter=72),
    # reductions of 4096 and more take the 256-row two-accumulator tile: full
    # tiles, tails whose second half is partly or wholly empty, a ragged K tail
    "longk": synth.Workload("longk", 300, 4096, 4, 2, 136),
    "longk_relu2": synth.Workload("longk_relu2", 200, 4160, 3, 2, 264, act=synth.ACT_RELU2),
    "longk_shared": synth.Workload("longk_shared", 40, 4096, 6, 2, 64, shared=4, shared_inter=1024),
    # 256 or more rows per group take the CTA-pair kernel: full 256-row tiles,
    # 128-row tails, ragged N and K, ReLU^2, long K, shared experts
    "pair_swiglu": synth.Workload("pair_swiglu", 640, 256, 4, 2, 200),
    "pair_relu2": synth.Workload("pair_relu2", 600, 200, 3, 2, 264, act=synth.ACT_RELU2),
    "pair_shared": synth.Workload("pair_shared", 300, 128, 2, 2, 64, shared=2, shared_inter=72),
    "pair_longk": synth.Workload("pair_longk", 300, 4096, 2, 2, 136),
    # the pair kernel with K of an odd number of 64-column chunks, and two shared
    # experts summed over K segments (their down projection) on the pair path
    "pair_oddk": synth.Workload("pair_oddk", 600, 320, 2, 1, 192, shared=2, shared_inter=192),
}
for _n in DECODE:
    SMALL[_n] = W[_n]


def oracle_stages(wl, g):
    """Full oracle layer from generator inputs (host copies)."""
    x = bits(g["x"])
    kw = {}
    if wl.shared:
        kw = dict(ws13=bits(g["ws13"]), ws2=bits(g["ws2"]))
    return oracle.layer(x, bits(g["w13"]), bits(g["w2"]), wl.act, wl.top_k, wl.cap,
                        logits=g["logits"].cpu().numpy(), **kw)


# ---------------------------------------------------------------------------
# route
# ---------------------------------------------------------------------------
ROUTE_CASES = {**{k: v for k, v in W.items()},
               **{k: SMALL[k] for k in ("ragged", "wide_e", "max_e", "t1", "k_eq_e")}}


@pytest.mark.parametrize("name", sorted(ROUTE_CASES))
def test_route(name):
    wl = ROUTE_CASES[name]
    lg = synth.make_logits(wl, seed=3, device=dev())
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    N.moe_route(shape, lg, o["ids"], o["w"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    st, ids, w = oracle.route(lg.cpu().numpy(), wl.top_k)
    assert st == 0
    assert np.array_equal(o["ids"].cpu().numpy(), ids)
    gw = o["w"].cpu().numpy()
    assert np.abs(gw - w).max() <= W_TOL
    assert np.abs(gw.astype(np.float64).sum(1) - 1).max() <= W_TOL


@pytest.mark.parametrize("E,k", [(5, 3), (16, 4), (64, 6), (130, 8)])
def test_route_ties(E, k):
    # small integer logits: most selections are decided by the index rule
    g = torch.Generator().manual_seed(E)
    lg = torch.randint(-2, 3, (257, E), generator=g).float()
    lg[lg == 0] = -0.0 if E % 2 else 0.0
    wl = synth.Workload("ties", 257, 64, E, k, 64)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    ids = torch.empty(257, k, dtype=torch.int32, device=dev())
    w = torch.empty(257, k, dtype=torch.float32, device=dev())
    N.moe_route(shape, lg.to(dev()), ids, w, ws)
    assert N.moe_status_read(ws) == 0
    st, oi, ow = oracle.route(lg.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), oi)
    assert np.abs(w.cpu().numpy() - ow).max() <= W_TOL


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
def test_route_nonfinite_raises_status(bad):
    wl = synth.Workload("nf", 40, 64, 16, 2, 64)
    lg = synth.make_logits(wl, device=dev())
    lg[17, 3] = bad
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    N.moe_route(shape, lg, o["ids"], o["w"], ws)
    assert N.moe_status_read(ws) == N.MOE_ERR_NONFINITE
    # the status is cleared by the read
    N.moe_route(shape, synth.make_logits(wl, device=dev()), o["ids"], o["w"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------
def gpu_dispatch(wl, x_dev, ids_np, cap=None):
    shape = N.shape_of(wl)
    if cap is not None:
        shape.capacity = cap
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    o["dest"].fill_(-7)
    o["sorted_pair"].fill_(-7)
    o["x_perm"].zero_()
    N.moe_dispatch(shape, x_dev, i32_dev(ids_np), o["counts"], o["offsets"], o["dest"], o["sorted_pair"],
                   o["x_perm"], ws)
    return o, N.moe_status_read(ws)


DISPATCH_CASES = ["tiny", "count_first", "deepseek", "large", "ragged", "one_expert", "k_eq_e", "wide_e", "max_e",
                  "t1"] + DECODE


@pytest.mark.parametrize("name", DISPATCH_CASES)
def test_dispatch(name):
    wl = W.get(name) or SMALL[name]
    lg = synth.make_logits(wl, seed=1, device="cpu").numpy()
    _, ids, _ = oracle.route(lg, wl.top_k)
    x_dev = synth.normal((wl.tokens, wl.hidden), 1.0, 1, "x", dev())
    x = bits(x_dev)
    st, counts, offsets, dest, sp, xp = oracle.dispatch(ids, x, wl.experts, wl.cap)
    assert st == 0
    o, gst = gpu_dispatch(wl, x_dev, ids)
    assert gst == N.MOE_OK
    assert np.array_equal(o["counts"].cpu().numpy(), counts)
    assert np.array_equal(o["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(o["dest"].cpu().numpy(), dest)
    assert np.array_equal(o["sorted_pair"].cpu().numpy(), sp)
    # x_perm is a copy: bit-exact (compared on the device for the 1.9 GB case)
    assert torch.equal(o["x_perm"].view(torch.int16), torch.from_numpy(xp.view(np.int16)).to(dev()))


def test_dispatch_capacity_overflow_moves_no_payload():
    wl = synth.Workload("cap", 300, 64, 8, 2, 64)
    ids = np.tile(np.array([[0, 1]], np.int32), (300, 1))
    ids[::3, 1] = 5
    x_dev = synth.normal((300, 64), 1.0, 2, "x", dev())
    st, counts, offsets, *_ = oracle.dispatch(ids, bits(x_dev), 8, 250)
    assert st == oracle.ST_CAPACITY
    o, gst = gpu_dispatch(wl, x_dev, ids, cap=250)
    assert gst == N.MOE_ERR_CAPACITY
    assert np.array_equal(o["counts"].cpu().numpy(), counts)
    assert np.array_equal(o["offsets"].cpu().numpy(), offsets)
    assert torch.all(o["dest"] == -7) and torch.all(o["sorted_pair"] == -7)
    assert torch.all(o["x_perm"].view(torch.int16) == 0)
    # exactly at capacity (300 on expert 0) passes
    o, gst = gpu_dispatch(wl, x_dev, ids, cap=300)
    assert gst == N.MOE_OK


@pytest.mark.parametrize("kind", ["negative", "wide", "duplicate", "dummy"])
def test_dispatch_invalid_routes(kind):
    wl = synth.Workload("bad", 1500, 64, 16, 4, 64)     # 6000 pairs: several count tiles
    g = torch.Generator().manual_seed(9)
    ids = torch.stack([torch.randperm(16, generator=g)[:4] for _ in range(1500)]).int().numpy()
    if kind == "negative":
        ids[700, 2] = -5
    elif kind == "wide":
        ids[700, 2] = 16
    elif kind == "duplicate":
        ids[700, 2] = ids[700, 0]
    else:
        ids[700, 2] = -1
    ids[1499, 3] = 99
    x_dev = synth.normal((1500, 64), 1.0, 3, "x", dev())
    st, counts, offsets, dest, sp, xp = oracle.dispatch(ids, bits(x_dev), 16, 1500)
    assert st == oracle.ST_INVALID_ROUTE
    o, gst = gpu_dispatch(wl, x_dev, ids)
    assert gst == N.MOE_ERR_INVALID_ROUTE
    # invalid pairs are neither counted nor placed; the valid ones match the oracle
    assert np.array_equal(o["counts"].cpu().numpy(), counts)
    assert np.array_equal(o["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(o["dest"].cpu().numpy(), dest)
    n = offsets[-1]
    assert np.array_equal(o["sorted_pair"].cpu().numpy()[:n], sp[:n])


def test_dispatch_is_deterministic():
    wl = W["count_first"]
    lg = synth.make_logits(wl, seed=5).numpy()
    _, ids, _ = oracle.route(lg, wl.top_k)
    x_dev = synth.normal((wl.tokens, wl.hidden), 1.0, 5, "x", dev())
    a, _ = gpu_dispatch(wl, x_dev, ids)
    for _ in range(3):
        b, _ = gpu_dispatch(wl, x_dev, ids)
        for key in ("counts", "offsets", "dest", "sorted_pair"):
            assert torch.equal(a[key], b[key])


# ---------------------------------------------------------------------------
# expert FFN (up, down, shared)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("unit", [False, True])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_expert_ffn_full(name, unit):
    wl = SMALL[name]
    g = inputs(wl, unit_scale=unit, seed=11)
    ref = oracle_stages(wl, g)
    assert ref["status"] == 0
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    offsets = i32_dev(ref["offsets"])
    # up projection on the oracle's x_perm
    N.moe_expert_up(shape, to_bf16_dev(ref["x_perm"]), offsets, g["w13"], g["x"], g.get("ws13"), o["h"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), ref["h"], f"{name} h")
    # down projection on the oracle's h (shared part reads the workspace the up call filled)
    N.moe_expert_down(shape, to_bf16_dev(ref["h"]), offsets, g["w2"], g.get("ws2"), o["y_perm"], o["y_shared"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["y_perm"]), ref["y_perm"], f"{name} y_perm")
    if wl.shared:
        assert_close(bits(o["y_shared"]), ref["y_shared"], f"{name} y_shared")


@pytest.mark.parametrize("act", [synth.ACT_SWIGLU, synth.ACT_RELU2])
def test_expert_ffn_buckets_above_the_row_bound(act):
    """Caller-made offsets may hold more rows in a group than the token count
    (here 100 and 28 rows at 16 tokens): the small-row kernel, picked from the
    token count, then takes such a group in 16-row chunks."""
    wl = synth.Workload("chunked", 16, 192, 8, 8, 96, act=act)
    g = inputs(wl, unit_scale=True, seed=12)
    R = wl.pairs
    x_perm = synth.normal((R, wl.hidden), 1.0, 12, "x_perm", dev())
    offsets = np.array([0, 100, 100, 100, 128, 128, 128, 128, 128], np.int32)
    h_ref, y_ref, _, _ = oracle.expert_ffn(bits(x_perm), offsets, bits(g["w13"]), bits(g["w2"]), wl.act)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    N.moe_expert_up(shape, x_perm, i32_dev(offsets), g["w13"], g["x"], None, o["h"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), h_ref, "chunked h")
    N.moe_expert_down(shape, to_bf16_dev(h_ref), i32_dev(offsets), g["w2"], None, o["y_perm"], None, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["y_perm"]), y_ref, "chunked y_perm")


# one full 256-row tile plus a tail of every padded size class per group (16
# to 256 rows, 8 to 128 per CTA of the pair), and exact multiples of 256
PAIR_TAILS = [0, 1, 8, 9, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 255]


@pytest.mark.parametrize("act,hidden", [(synth.ACT_SWIGLU, 320), (synth.ACT_RELU2, 576)])
def test_expert_ffn_pair_kernel_partial_tiles(act, hidden):
    """Caller-made offsets whose groups (two of them empty) hold 256 + t rows
    for every tail size t above: the CTA-pair kernel computes each group's
    full tile, then its tail with the operands swapped (weights on M, the
    tail's rows padded to 16 on N); K of 5 and 9 chunks of 64, and the down
    projection's 3."""
    sizes = [256 + t for t in PAIR_TAILS]
    sizes[3:3] = [0]
    sizes[10:10] = [0]
    E, R = len(sizes), sum(sizes)
    wl = synth.Workload("pair_tails", R, hidden, E, 1, 192, act=act)
    g = inputs(wl, unit_scale=True, seed=13)
    x_perm = synth.normal((R, hidden), 1.0, 13, "x_perm", dev())
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    h_ref, y_ref, _, _ = oracle.expert_ffn(bits(x_perm), offsets, bits(g["w13"]), bits(g["w2"]), wl.act)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    N.moe_expert_up(shape, x_perm, i32_dev(offsets), g["w13"], g["x"], None, o["h"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), h_ref, "pair tails h")
    N.moe_expert_down(shape, to_bf16_dev(h_ref), i32_dev(offsets), g["w2"], None, o["y_perm"], None, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["y_perm"]), y_ref, "pair tails y_perm")


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "count_first", "deepseek_t96", "k_eq_e", "t1"] + DECODE[:2])
def test_combine(name):
    wl = W.get(name) or SMALL[name]
    lg = synth.make_logits(wl, seed=4).numpy()
    _, ids, w = oracle.route(lg, wl.top_k)
    st, counts, offsets, dest, sp, _ = oracle.dispatch(ids, np.zeros((wl.tokens, 8), np.uint16), wl.experts, wl.cap)
    y_dev = synth.normal((wl.pairs, wl.hidden), 1.0, 4, "y_perm", dev())
    ys_dev = synth.normal((wl.tokens, wl.hidden), 1.0, 4, "y_shared", dev()) if wl.shared else None
    want = oracle.combine(bits(y_dev), dest, w, None if ys_dev is None else bits(ys_dev))
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_combine(shape, y_dev, i32_dev(dest), f32_dev(w), ys_dev, out, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), want, f"{name} out")


def test_combine_skips_invalid_pairs():
    wl = synth.Workload("c", 64, 128, 8, 3, 64)
    g = torch.Generator().manual_seed(2)
    dest = torch.randperm(192, generator=g).int().numpy()
    dest[10] = -1
    dest[20] = 5000          # out of range: treated as invalid, never read
    w = np.full((64, 3), 1.0 / 3, np.float32)
    y_dev = synth.normal((192, 128), 1.0, 6, "y", dev())
    dref = dest.copy()
    dref[20] = -1
    want = oracle.combine(bits(y_dev), dref, w)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(64, 128, dtype=torch.bfloat16, device=dev())
    N.moe_combine(shape, y_dev, i32_dev(dest), f32_dev(w), None, out, ws)
    assert_close(bits(out), want, "combine invalid")


@pytest.mark.parametrize("in_place", [False, True])
def test_combine_with_residual(in_place):
    """The MOE_COMBINE_RESIDUAL form: out = sum_j w y + y_shared + residual,
    also with out written over the residual buffer."""
    wl = W["deepseek"].with_(tokens=200)
    lg = synth.make_logits(wl, seed=12).numpy()
    _, ids, w = oracle.route(lg, wl.top_k)
    st, counts, offsets, dest, sp, _ = oracle.dispatch(ids, np.zeros((wl.tokens, 8), np.uint16), wl.experts, wl.cap)
    y_dev = synth.normal((wl.pairs, wl.hidden), 1.0, 12, "y_perm", dev())
    ys_dev = synth.normal((wl.tokens, wl.hidden), 1.0, 12, "y_shared", dev())
    res_dev = synth.normal((wl.tokens, wl.hidden), 1.0, 12, "residual", dev())
    want = oracle.combine(bits(y_dev), dest, w, bits(ys_dev), bits(res_dev))
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = res_dev if in_place else torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_combine(shape, y_dev, i32_dev(dest), f32_dev(w), ys_dev, out, ws, residual=res_dev)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), want, "combine + residual")
