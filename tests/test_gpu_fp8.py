"""GPU parity of the FP8 E4M3 expert-weight entry points against the oracle.

The weights are E4M3 codes with one FP32 scale per weight row (quantized on
the device from the same BF16 draws as the BF16 tests).  h, y_perm and out
must be within max|d| <= 1e-2 * max|ref| + 1e-3 of the oracle's FP64 sums
of x * decode(code), times the row scale; routing and dispatch stay
bit-exact.  With codes and power-of-two scales the FP8 layer must equal the
BF16 layer on the dequantized weights bit for bit (the scale commutes with
the FP32 accumulation)."""
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
    "tiny": W["tiny"],                                                          # SwiGLU, 64 rows
    "t1": synth.Workload("t1", 1, 256, 16, 4, 128),
    "k_eq_e": synth.Workload("k_eq_e", 40, 128, 8, 8, 64),
    "relu2_k_tail": synth.Workload("relu2_k_tail", 24, 208, 7, 3, 176, act=synth.ACT_RELU2),  # K % 64 != 0
    "mid_t96": synth.Workload("mid_t96", 96, 256, 8, 2, 192),                  # > 64 tokens: 64-row chunks
    "big_groups": synth.Workload("big_groups", 200, 128, 2, 1, 64, act=synth.ACT_RELU2),   # ~100-row groups
    "decode_1_shared": W["decode_1_shared"],
    "decode_16_distinct": W["decode_16_distinct"],
}


def host(t):
    return t.detach().cpu().numpy()


def fp8_inputs(wl, seed, unit=True):
    g = inputs(wl, unit_scale=unit, seed=seed)
    q = synth.make_fp8_weights(wl, seed=seed, device=dev(), unit_scale=unit)
    return g, q


def oracle_fp8_layer(wl, g, q, residual=None):
    return oracle.layer_fp8(bits(g["x"]), host(q["w13"]), host(q["s13"]), host(q["w2"]), host(q["s2"]), wl.act,
                            wl.top_k, wl.cap, logits=g["logits"].cpu().numpy(),
                            residual=None if residual is None else bits(residual))


@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8_expert_ffn(name):
    wl = CASES[name]
    g, q = fp8_inputs(wl, seed=51)
    ref = oracle_fp8_layer(wl, g, q)
    assert ref["status"] == 0
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    offsets = i32_dev(ref["offsets"])
    N.moe_expert_up_fp8(shape, to_bf16_dev(ref["x_perm"]), offsets, q["w13"], q["s13"], o["h"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), ref["h"], f"{name} fp8 h")
    N.moe_expert_down_fp8(shape, to_bf16_dev(ref["h"]), offsets, q["w2"], q["s2"], o["y_perm"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["y_perm"]), ref["y_perm"], f"{name} fp8 y_perm")


@pytest.mark.parametrize("act", [synth.ACT_SWIGLU, synth.ACT_RELU2])
def test_fp8_buckets_above_the_row_bound(act):
    """Caller-made offsets with 100- and 28-row groups at 16 tokens."""
    wl = synth.Workload("chunked", 16, 192, 8, 8, 96, act=act)
    _, q = fp8_inputs(wl, seed=52)
    x_perm = synth.normal((wl.pairs, wl.hidden), 1.0, 52, "x_perm", dev())
    offsets = np.array([0, 100, 100, 100, 128, 128, 128, 128, 128], np.int32)
    h_ref, y_ref = oracle.expert_ffn_fp8(bits(x_perm), offsets, host(q["w13"]), host(q["s13"]), host(q["w2"]),
                                         host(q["s2"]), wl.act)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    N.moe_expert_up_fp8(shape, x_perm, i32_dev(offsets), q["w13"], q["s13"], o["h"], ws)
    N.moe_expert_down_fp8(shape, to_bf16_dev(h_ref), i32_dev(offsets), q["w2"], q["s2"], o["y_perm"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), h_ref, "chunked fp8 h")
    assert_close(bits(o["y_perm"]), y_ref, "chunked fp8 y_perm")


@pytest.mark.parametrize("name", ["tiny", "mid_t96", "decode_1_shared", "decode_16_distinct"])
def test_fp8_layer(name):
    wl = CASES[name]
    g, q = fp8_inputs(wl, seed=53)
    res = synth.normal((wl.tokens, wl.hidden), 1.0, 53, "residual", dev()) if name == "tiny" else None
    ref = oracle_fp8_layer(wl, g, q, res)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_layer_fp8(shape, g["logits"], None, None, g["x"], q["w13"], q["s13"], q["w2"], q["s2"], out, ws,
                    residual=res)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), ref["out"], f"{name} fp8 layer")


@pytest.mark.parametrize("name", ["tiny", "mid_t96", "decode_16_distinct"])
def test_fp8_layer_equals_bf16_layer_on_exact_weights(name):
    """Codes with power-of-two row scales: dequantized weights are exact in
    BF16, so the BF16 layer on them is the same computation."""
    wl = CASES[name]
    g = inputs(wl, unit_scale=True, seed=54)
    gen = torch.Generator(device=dev())
    gen.manual_seed(54)
    q = synth.make_fp8_weights(wl, seed=54, device=dev(), unit_scale=True)
    q["s13"] = torch.exp2(torch.randint(-3, 4, q["s13"].shape, device=dev(), generator=gen).float()) * 2.0 ** -6
    q["s2"] = torch.exp2(torch.randint(-3, 4, q["s2"].shape, device=dev(), generator=gen).float()) * 2.0 ** -6
    w13 = (q["w13"].view(torch.float8_e4m3fn).float() * q["s13"][..., None]).to(torch.bfloat16)
    w2 = (q["w2"].view(torch.float8_e4m3fn).float() * q["s2"][..., None]).to(torch.bfloat16)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    a = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    b = torch.empty_like(a)
    N.moe_layer_fp8(shape, g["logits"], None, None, g["x"], q["w13"], q["s13"], q["w2"], q["s2"], a, ws)
    N.moe_layer(shape, g["logits"], None, None, g["x"], w13, w2, None, None, b, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fp8_layer_is_graph_capturable_and_deterministic():
    wl = CASES["decode_1_shared"]
    g, q = fp8_inputs(wl, seed=55)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    s = torch.cuda.Stream()
    run = lambda: N.moe_layer_fp8(shape, g["logits"], None, None, g["x"], q["w13"], q["s13"], q["w2"], q["s2"],
                                  out, ws, s)
    with torch.cuda.stream(s):
        run()
    s.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run()
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert N.moe_status_read(ws) == N.MOE_OK


def test_fp8_every_finite_code_decodes_exactly():
    """The down projection on one-hot rows returns single weights: y[r][c] =
    decode(W2[c][r]) * 1, exact in BF16.  W2 cycles through all 254 finite
    E4M3 codes (both zeros, the subnormals, +-448), so every code's decode in
    the kernel -- subnormals included -- is checked bit for bit against the
    oracle's decode."""
    H = I = R = 256
    wl = synth.Workload("codes", R, H, 1, 1, I, act=synth.ACT_RELU2)
    codes = np.arange(H * I, dtype=np.int64) % 256
    codes[(codes == 0x7F) | (codes == 0xFF)] = 0x38                    # the two NaN codes are not weights
    codes = codes.astype(np.uint8).reshape(1, H, I)
    rng = np.random.default_rng(3)
    codes[0] = codes[0][:, rng.permutation(I)]                          # every column sees many codes
    w2 = torch.from_numpy(codes).to(dev())
    s2 = torch.ones(1, H, dtype=torch.float32, device=dev())
    h = torch.eye(R, I, dtype=torch.bfloat16, device=dev())
    offsets = i32_dev(np.array([0, R], np.int32))
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    y = torch.empty(R, H, dtype=torch.bfloat16, device=dev())
    N.moe_expert_down_fp8(shape, h, offsets, w2, s2, y, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    want = oracle.fp8_e4m3_decode(codes[0].T)                           # y[r][c] = decode(W2[c][r])
    want_bits = torch.from_numpy(want).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = bits(y)
    # the sum adds the other columns' +0 products, so code 0x80 (-0) comes out
    # as +0: compare values (equal as numbers, -0 == +0), every other code bitwise
    neg_zero = codes[0].T == 0x80
    assert np.array_equal(got[~neg_zero], want_bits[~neg_zero]), int((got != want_bits)[~neg_zero].sum())
    assert np.all(got[neg_zero] == 0)


def random_fp8_workloads(n, seed):
    """Seeded small shapes for the FP8 entry points: hidden and intermediate
    multiples of 16 (K tails included), 1..100 tokens, both activations."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 41))
        k = int(rng.integers(1, min(E, 16) + 1))
        T = int(rng.choice([1, 5, 16, 40, 100]))
        H = int(16 * rng.integers(1, 25))
        I = int(16 * rng.integers(1, 25))
        out.append(synth.Workload(f"fp8rand{i}", T, H, E, k, I, act=int(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("wl", random_fp8_workloads(6, 2027),
                         ids=lambda w: f"{w.name}-T{w.tokens}H{w.hidden}E{w.experts}k{w.top_k}I{w.inter}a{w.act}")
def test_fp8_layer_random_shapes(wl):
    g, q = fp8_inputs(wl, seed=98)
    ref = oracle_fp8_layer(wl, g, q)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    N.moe_layer_fp8(shape, g["logits"], None, None, g["x"], q["w13"], q["s13"], q["w2"], q["s2"], out, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), ref["out"], f"{wl.name} fp8 layer")
