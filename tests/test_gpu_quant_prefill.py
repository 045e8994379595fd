"""Quantized expert weights (FP8 E4M3, NVFP4) at prefill sizes: the tile
kernel with converted weight tiles (groups of more than 64 rows), against the
oracle's FP64 sums on the codes and scales.

Small prefill shapes are compared in full (h, y_perm, out); the count-first
and DeepSeek-shaped prefills (2048 and 1024 tokens; the DeepSeek shape without
its shared experts, which the quantized entry points omit) on sampled rows of
h and y_perm -- the first and last row of the hottest, the coldest and random
experts, plus seeded random rows -- recomputed by the oracle from the
generator inputs.  With power-of-two row scales (and, for NVFP4, weights
formed exactly) the quantized layer must equal the BF16 layer on the
dequantized weights bit for bit: the same tiles, the same FP32 sums.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

from gpu_util import alloc_stage_outputs, assert_close, bits, dev, i32_dev, inputs, to_bf16_dev

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS

CASES = {
    "cf_t160": W["count_first"].with_(tokens=160, name="cf_t160"),                 # 10 rows per expert on average
    "ds_t200": synth.Workload("ds_t200", 200, 2048, 64, 6, 1408),                  # SwiGLU, ~19 rows per expert
    "relu2_t300": synth.Workload("relu2_t300", 300, 1024, 16, 4, 1536, act=synth.ACT_RELU2),   # 75 rows
    "ragged_n_k": synth.Workload("ragged_n_k", 150, 288, 5, 2, 224),              # N and K tails
    "one_big_group": synth.Workload("one_big_group", 700, 256, 2, 1, 192, act=synth.ACT_RELU2),  # 350 rows
    # groups of 100-160 rows: a full 128-row tile and a tail of up to 64 rows (M = 64)
    # or more (M = 128) per group; ragged N and K
    "tails_mix": synth.Workload("tails_mix", 400, 256, 6, 2, 192),                 # ~133 rows per group
    "tails_relu2": synth.Workload("tails_relu2", 500, 320, 4, 1, 224, act=synth.ACT_RELU2),     # ~125 rows
}
FULL = {
    "count_first": W["count_first"],
    "deepseek_routed": W["deepseek_routed"],
}


def host(t):
    return t.detach().cpu().numpy()


def qweights(fmt, wl, seed):
    if fmt == "fp8":
        return synth.make_fp8_weights(wl, seed=seed, device=dev(), unit_scale=True)
    return synth.make_nvfp4_weights(wl, seed=seed, device=dev(), unit_scale=True)


def oracle_ffn(fmt, x_perm, offsets, q, act):
    if fmt == "fp8":
        return oracle.expert_ffn_fp8(x_perm, offsets, host(q["w13"]), host(q["s13"]), host(q["w2"]), host(q["s2"]),
                                     act)
    return oracle.expert_ffn_nvfp4(x_perm, offsets, host(q["w13"]), host(q["b13"]), host(q["s13"]), host(q["w2"]),
                                   host(q["b2"]), host(q["s2"]), act)


def oracle_layer(fmt, wl, g, q):
    lg = g["logits"].cpu().numpy()
    if fmt == "fp8":
        return oracle.layer_fp8(bits(g["x"]), host(q["w13"]), host(q["s13"]), host(q["w2"]), host(q["s2"]), wl.act,
                                wl.top_k, wl.cap, logits=lg)
    return oracle.layer_nvfp4(bits(g["x"]), host(q["w13"]), host(q["b13"]), host(q["s13"]), host(q["w2"]),
                              host(q["b2"]), host(q["s2"]), wl.act, wl.top_k, wl.cap, logits=lg)


def up(fmt, shape, x_perm, offsets, q, h, ws):
    if fmt == "fp8":
        N.moe_expert_up_fp8(shape, x_perm, offsets, q["w13"], q["s13"], h, ws)
    else:
        N.moe_expert_up_nvfp4(shape, x_perm, offsets, q["w13"], q["b13"], q["s13"], h, ws)


def down(fmt, shape, h, offsets, q, y, ws):
    if fmt == "fp8":
        N.moe_expert_down_fp8(shape, h, offsets, q["w2"], q["s2"], y, ws)
    else:
        N.moe_expert_down_nvfp4(shape, h, offsets, q["w2"], q["b2"], q["s2"], y, ws)


def layer(fmt, shape, g, q, out, ws):
    if fmt == "fp8":
        N.moe_layer_fp8(shape, g["logits"], None, None, g["x"], q["w13"], q["s13"], q["w2"], q["s2"], out, ws)
    else:
        N.moe_layer_nvfp4(shape, g["logits"], None, None, g["x"], q["w13"], q["b13"], q["s13"], q["w2"], q["b2"],
                          q["s2"], out, ws)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_stages_and_layer(fmt, name):
    wl = CASES[name]
    g = inputs(wl, unit_scale=True, seed=71)
    q = qweights(fmt, wl, 71)
    ref = oracle_layer(fmt, wl, g, q)
    assert ref["status"] == 0
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    offsets = i32_dev(ref["offsets"])
    up(fmt, shape, to_bf16_dev(ref["x_perm"]), offsets, q, o["h"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), ref["h"], f"{name} {fmt} h")
    down(fmt, shape, to_bf16_dev(ref["h"]), offsets, q, o["y_perm"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["y_perm"]), ref["y_perm"], f"{name} {fmt} y_perm")
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    layer(fmt, shape, g, q, out, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    err, mref = assert_close(bits(out), ref["out"], f"{name} {fmt} out")
    assert mref > 0.1


def test_fp8_prefill_layer_equals_bf16_layer_on_exact_weights():
    """Power-of-two row scales make the dequantized weights exact in BF16; the
    converted tiles then feed the tensor core the very BF16 tiles of the BF16
    layer, and the scale commutes with the FP32 sums."""
    wl = CASES["cf_t160"]
    g = inputs(wl, unit_scale=True, seed=72)
    q = qweights("fp8", wl, 72)
    gen = torch.Generator(device=dev())
    gen.manual_seed(72)
    q["s13"] = torch.exp2(torch.randint(-3, 4, q["s13"].shape, device=dev(), generator=gen).float()) * 2.0 ** -6
    q["s2"] = torch.exp2(torch.randint(-3, 4, q["s2"].shape, device=dev(), generator=gen).float()) * 2.0 ** -6
    w13 = (q["w13"].view(torch.float8_e4m3fn).float() * q["s13"][..., None]).to(torch.bfloat16)
    w2 = (q["w2"].view(torch.float8_e4m3fn).float() * q["s2"][..., None]).to(torch.bfloat16)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    a = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    b = torch.empty_like(a)
    layer("fp8", shape, g, q, a, ws)
    N.moe_layer(shape, g["logits"], None, None, g["x"], w13, w2, None, None, b, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _sample_rows(counts, offsets, R, rng, n):
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    rows = set()
    for e in list(order[:2]) + list(order[-3:]) + list(rng.choice(nz, 6, replace=False)):
        rows |= {int(offsets[e]), int(offsets[e + 1]) - 1}
    while len(rows) < n:
        rows.add(int(rng.integers(0, R)))
    return np.array(sorted(rows), np.int64)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("name", sorted(FULL))
def test_prefill_full_size_sampled_rows(fmt, name):
    wl = FULL[name]
    k = wl.top_k
    g = inputs(wl, seed=0)
    q = qweights(fmt, wl, 0)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    N.moe_route(shape, g["logits"], o["ids"], o["w"], ws)
    N.moe_dispatch(shape, g["x"], o["ids"], o["counts"], o["offsets"], o["dest"], o["sorted_pair"], o["x_perm"], ws)
    up(fmt, shape, o["x_perm"], o["offsets"], q, o["h"], ws)
    down(fmt, shape, o["h"], o["offsets"], q, o["y_perm"], ws)
    N.moe_combine(shape, o["y_perm"], o["dest"], o["w"], None, o["out"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    # placement from the oracle (routing and dispatch are bit-exact elsewhere)
    x = bits(g["x"])
    _, ids, _ = oracle.route(g["logits"].cpu().numpy(), k)
    _, counts, offsets, _, sp, _ = oracle.dispatch(ids, x[:, :8], wl.experts, wl.cap)
    assert np.array_equal(o["offsets"].cpu().numpy(), offsets)
    rows = _sample_rows(counts, offsets, wl.pairs, np.random.default_rng(5), 512)
    # the sampled rows as a small bucketed batch for the oracle, from x alone
    row_exp = np.searchsorted(offsets, rows, side="right") - 1
    mini_x = x[sp[rows] // k]
    mini_off = np.searchsorted(row_exp, np.arange(wl.experts + 1), side="left").astype(np.int32)
    h_ref, y_ref = oracle_ffn(fmt, mini_x, mini_off, q, wl.act)
    ridx = torch.from_numpy(rows).to(dev())
    assert_close(bits(o["h"][ridx]), h_ref, f"{name} {fmt} h ({len(rows)} rows)")
    assert_close(bits(o["y_perm"][ridx]), y_ref, f"{name} {fmt} y_perm ({len(rows)} rows)")
    # the layer call gives the staged output bitwise
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    layer(fmt, shape, g, q, out, N.workspace(shape, dev()))
    assert torch.equal(out.view(torch.int16), o["out"].view(torch.int16))
