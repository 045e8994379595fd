"""GPU parity of the NVFP4 expert-weight entry points against the oracle.

The weights are E2M1 codes with an E4M3 scale per 16 elements and an FP32
scale per row (quantized on the device from the same BF16 draws as the BF16
tests).  h, y_perm and out must be within max|d| <= 1e-2 * max|ref| + 1e-3 of
the oracle's FP64 sums of x * e2m1 * block scale, times the row scale; routing
and dispatch stay bit-exact.  With power-of-two row scales every dequantized
weight is exact in BF16, so the NVFP4 layer must equal the BF16 layer on the
dequantized weights bit for bit."""
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
    "relu2_k_tail": synth.Workload("relu2_k_tail", 24, 224, 7, 3, 160, act=synth.ACT_RELU2),  # K % 256 != 0
    "k_over_256": synth.Workload("k_over_256", 12, 288, 5, 2, 352),            # two stages, the second partial
    "mid_t96": synth.Workload("mid_t96", 96, 256, 8, 2, 192),                  # > 64 tokens: 64-row chunks
    "big_groups": synth.Workload("big_groups", 200, 128, 2, 1, 64, act=synth.ACT_RELU2),   # ~100-row groups
    "decode_1_shared": W["decode_1_shared"],
    "decode_16_distinct": W["decode_16_distinct"],
}


def host(t):
    return t.detach().cpu().numpy()


def nvfp4_inputs(wl, seed, unit=True):
    g = inputs(wl, unit_scale=unit, seed=seed)
    q = synth.make_nvfp4_weights(wl, seed=seed, device=dev(), unit_scale=unit)
    return g, q


def oracle_nvfp4_layer(wl, g, q, residual=None):
    return oracle.layer_nvfp4(bits(g["x"]), host(q["w13"]), host(q["b13"]), host(q["s13"]), host(q["w2"]),
                              host(q["b2"]), host(q["s2"]), wl.act, wl.top_k, wl.cap,
                              logits=g["logits"].cpu().numpy(), residual=None if residual is None else bits(residual))


def run_layer(wl, g, q, out, ws, stream=None, residual=None):
    N.moe_layer_nvfp4(N.shape_of(wl), g["logits"], None, None, g["x"], q["w13"], q["b13"], q["s13"], q["w2"],
                      q["b2"], q["s2"], out, ws, stream, residual=residual)


@pytest.mark.parametrize("name", sorted(CASES))
def test_nvfp4_expert_ffn(name):
    wl = CASES[name]
    g, q = nvfp4_inputs(wl, seed=61)
    ref = oracle_nvfp4_layer(wl, g, q)
    assert ref["status"] == 0
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    offsets = i32_dev(ref["offsets"])
    N.moe_expert_up_nvfp4(shape, to_bf16_dev(ref["x_perm"]), offsets, q["w13"], q["b13"], q["s13"], o["h"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), ref["h"], f"{name} nvfp4 h")
    N.moe_expert_down_nvfp4(shape, to_bf16_dev(ref["h"]), offsets, q["w2"], q["b2"], q["s2"], o["y_perm"], ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["y_perm"]), ref["y_perm"], f"{name} nvfp4 y_perm")


@pytest.mark.parametrize("act", [synth.ACT_SWIGLU, synth.ACT_RELU2])
def test_nvfp4_buckets_above_the_row_bound(act):
    """Caller-made offsets with 100- and 28-row groups at 16 tokens."""
    wl = synth.Workload("chunked", 16, 192, 8, 8, 96, act=act)
    _, q = nvfp4_inputs(wl, seed=62)
    x_perm = synth.normal((wl.pairs, wl.hidden), 1.0, 62, "x_perm", dev())
    offsets = np.array([0, 100, 100, 100, 128, 128, 128, 128, 128], np.int32)
    h_ref, y_ref = oracle.expert_ffn_nvfp4(bits(x_perm), offsets, host(q["w13"]), host(q["b13"]), host(q["s13"]),
                                           host(q["w2"]), host(q["b2"]), host(q["s2"]), wl.act)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    o = alloc_stage_outputs(wl)
    N.moe_expert_up_nvfp4(shape, x_perm, i32_dev(offsets), q["w13"], q["b13"], q["s13"], o["h"], ws)
    N.moe_expert_down_nvfp4(shape, to_bf16_dev(h_ref), i32_dev(offsets), q["w2"], q["b2"], q["s2"], o["y_perm"],
                            ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(o["h"]), h_ref, "chunked nvfp4 h")
    assert_close(bits(o["y_perm"]), y_ref, "chunked nvfp4 y_perm")


@pytest.mark.parametrize("name", ["tiny", "mid_t96", "decode_1_shared", "decode_16_distinct"])
def test_nvfp4_layer(name):
    wl = CASES[name]
    g, q = nvfp4_inputs(wl, seed=63)
    res = synth.normal((wl.tokens, wl.hidden), 1.0, 63, "residual", dev()) if name == "tiny" else None
    ref = oracle_nvfp4_layer(wl, g, q, res)
    ws = N.workspace(N.shape_of(wl), dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    run_layer(wl, g, q, out, ws, residual=res)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), ref["out"], f"{name} nvfp4 layer")


def dequantize(codes, bscale, rscale, K):
    """e2m1 * block scale * row scale, formed on the device from the E2M1
    value list and torch's E4M3 decode (exact in BF16 for power-of-two row
    scales)."""
    mags = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device=codes.device)
    nib = torch.stack([codes & 15, codes >> 4], dim=-1).flatten(-2).long()
    e = torch.where(nib >= 8, -1.0, 1.0) * mags[nib & 7]
    sb = bscale[..., :K // 16].view(torch.float8_e4m3fn).float().repeat_interleave(16, dim=-1)
    return (e * sb * rscale[..., None]).to(torch.bfloat16)


@pytest.mark.parametrize("name", ["tiny", "mid_t96", "decode_16_distinct", "k_over_256"])
def test_nvfp4_layer_equals_bf16_layer_on_exact_weights(name):
    wl = CASES[name]
    g = inputs(wl, unit_scale=True, seed=64)
    gen = torch.Generator(device=dev())
    gen.manual_seed(64)
    q = synth.make_nvfp4_weights(wl, seed=64, device=dev(), unit_scale=True)
    q["s13"] = torch.exp2(torch.randint(-3, 4, q["s13"].shape, device=dev(), generator=gen).float()) * 2.0 ** -4
    q["s2"] = torch.exp2(torch.randint(-3, 4, q["s2"].shape, device=dev(), generator=gen).float()) * 2.0 ** -4
    w13 = dequantize(q["w13"], q["b13"], q["s13"], wl.hidden)
    w2 = dequantize(q["w2"], q["b2"], q["s2"], wl.inter)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    a = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    b = torch.empty_like(a)
    run_layer(wl, g, q, a, ws)
    N.moe_layer(shape, g["logits"], None, None, g["x"], w13, w2, None, None, b, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_nvfp4_layer_is_graph_capturable_and_deterministic():
    wl = CASES["decode_1_shared"]
    g, q = nvfp4_inputs(wl, seed=65)
    ws = N.workspace(N.shape_of(wl), dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_layer(wl, g, q, out, ws, s)
    s.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run_layer(wl, g, q, out, ws, s)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert N.moe_status_read(ws) == N.MOE_OK


def test_nvfp4_every_code_and_block_scale_decodes_exactly():
    """The down projection on one-hot rows returns single weights: y[r][c] =
    e2m1(W2[c][r]) * e4m3(bscale[c][r/16]), exact in BF16 (row scales 1).  The
    codes are random and the block scales run through all 254 finite E4M3
    codes (both signs, subnormals, +-448), so every E2M1 code and every block
    scale, with the nibble order and the block indexing, is checked bit for bit
    against the oracle's decode."""
    H = I = R = 256
    wl = synth.Workload("codes", R, H, 1, 1, I, act=synth.ACT_RELU2)
    rng = np.random.default_rng(5)
    nib = rng.integers(0, 16, (H, I))
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    sb = np.arange(H * (I // 16), dtype=np.int64) % 256
    sb[(sb == 0x7F) | (sb == 0xFF)] = 0x38                              # the two NaN codes are not scales
    sb = rng.permutation(sb).astype(np.uint8).reshape(H, I // 16)
    w2 = torch.from_numpy(codes[None]).to(dev())
    b2 = torch.from_numpy(sb[None]).to(dev())
    s2 = torch.ones(1, H, dtype=torch.float32, device=dev())
    h = torch.eye(R, I, dtype=torch.bfloat16, device=dev())
    offsets = i32_dev(np.array([0, R], np.int32))
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    y = torch.empty(R, H, dtype=torch.bfloat16, device=dev())
    N.moe_expert_down_nvfp4(shape, h, offsets, w2, b2, s2, y, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    want = (oracle.fp4_e2m1_decode(nib.astype(np.uint8)) *
            np.repeat(oracle.fp8_e4m3_decode(sb), 16, axis=1)).T          # y[r][c] = W2[c][r]
    want_bits = torch.from_numpy(want).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = bits(y)
    # the sum adds the other columns' +0 products, so a -0 weight comes out as
    # +0: compare zeros as numbers, every other weight bitwise
    zero = want == 0
    assert np.array_equal(got[~zero], want_bits[~zero]), int((got != want_bits)[~zero].sum())
    assert np.all((got[zero] & 0x7FFF) == 0)


def random_nvfp4_workloads(n, seed):
    """Seeded small shapes for the NVFP4 entry points: hidden and intermediate
    multiples of 32 (K tails below and above 256 included), 1..100 tokens,
    both activations."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 41))
        k = int(rng.integers(1, min(E, 16) + 1))
        T = int(rng.choice([1, 5, 16, 40, 100]))
        H = int(32 * rng.integers(1, 19))
        I = int(32 * rng.integers(1, 19))
        out.append(synth.Workload(f"nvfp4rand{i}", T, H, E, k, I, act=int(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("wl", random_nvfp4_workloads(6, 2029),
                         ids=lambda w: f"{w.name}-T{w.tokens}H{w.hidden}E{w.experts}k{w.top_k}I{w.inter}a{w.act}")
def test_nvfp4_layer_random_shapes(wl):
    g, q = nvfp4_inputs(wl, seed=99)
    ref = oracle_nvfp4_layer(wl, g, q)
    ws = N.workspace(N.shape_of(wl), dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    run_layer(wl, g, q, out, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    assert_close(bits(out), ref["out"], f"{wl.name} nvfp4 layer")
