"""GPU parity of the router front end: the gate projection (FP32 logits from
x and W_gate) and sigmoid routing with a selection-only correction bias
(ONNX Runtime PR #33963, Description bullet 2), against the oracle.
Routing ids are bit-exact; weights within 1e-5 (times the route scale);
FP32 logits within 1e-4 * max|ref| + 1e-5."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

from gpu_util import bits, dev, W_TOL

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS


def gpu_route_sigmoid(wl, logits, bias, scale):
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    ids = torch.empty(wl.tokens, wl.top_k, dtype=torch.int32, device=dev())
    w = torch.empty(wl.tokens, wl.top_k, dtype=torch.float32, device=dev())
    N.moe_route_sigmoid(shape, logits, bias, scale, ids, w, ws)
    return ids.cpu().numpy(), w.cpu().numpy(), N.moe_status_read(ws)


@pytest.mark.parametrize("bias_kind", ["none", "small", "dominant"])
@pytest.mark.parametrize("name", ["tiny", "count_first", "deepseek", "large", "decode_16_distinct"])
def test_route_sigmoid(name, bias_kind):
    wl = W[name]
    lg = synth.make_logits(wl, seed=7, device=dev())
    bias = None
    if bias_kind == "small":
        bias = synth.correction_bias(wl, seed=7, device=dev())
    elif bias_kind == "dominant":
        bias = torch.zeros(wl.experts, device=dev())
        bias[torch.arange(0, wl.experts, 5, device=dev())[: wl.top_k]] = 2.0
    scale = 2.5
    ids, w, st = gpu_route_sigmoid(wl, lg, bias, scale)
    assert st == N.MOE_OK
    ost, oids, ow = oracle.route_sigmoid(lg.cpu().numpy(), wl.top_k,
                                         None if bias is None else bias.cpu().numpy(), scale)
    assert ost == 0
    assert np.array_equal(ids, oids)
    assert np.abs(w - ow).max() <= W_TOL * scale


def test_route_sigmoid_ties_and_nonfinite():
    wl = synth.Workload("sig", 300, 64, 24, 4, 64)
    g = torch.Generator().manual_seed(5)
    lg = torch.randint(-1, 2, (300, 24), generator=g).float()       # many equal scores
    ids, w, st = gpu_route_sigmoid(wl, lg.to(dev()), None, 1.0)
    _, oids, ow = oracle.route_sigmoid(lg.numpy(), 4)
    assert st == 0 and np.array_equal(ids, oids) and np.abs(w - ow).max() <= W_TOL
    lg[10, 3] = float("nan")
    _, _, st = gpu_route_sigmoid(wl, lg.to(dev()), None, 1.0)
    assert st == N.MOE_ERR_NONFINITE


GATE_CASES = {
    "tiny": W["tiny"],                                        # 64 rows: small-row kernel
    "decode_16": W["decode_16_distinct"],                     # 16 rows, 240 experts: small-row kernel
    "count_first": W["count_first"],                          # 2048 rows: CTA pair
    "ragged": synth.Workload("ragged", 300, 136, 33, 2, 64),  # E = 33: element stores, K tail
    "large": W["large"],                                      # the large layer, sampled rows
}


@pytest.mark.parametrize("name", sorted(GATE_CASES))
def test_gate_projection(name):
    wl = GATE_CASES[name]
    x = synth.normal((wl.tokens, wl.hidden), 1.0, 8, "x", dev())
    wg = synth.gate_weights(wl, seed=8, device=dev())
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    logits = torch.empty(wl.tokens, wl.experts, dtype=torch.float32, device=dev())
    N.moe_gate(shape, x, wg, logits, ws)
    assert N.moe_status_read(ws) == N.MOE_OK
    rows = np.arange(wl.tokens)
    if wl.tokens > 4096:
        rows = np.unique(np.concatenate([[0, wl.tokens - 1], np.random.default_rng(0).choice(wl.tokens, 254)]))
    want = oracle.gate(bits(x)[rows], bits(wg)).astype(np.float64)
    got = logits.cpu().numpy()[rows].astype(np.float64)
    err = np.abs(got - want).max()
    assert err <= 1e-4 * np.abs(want).max() + 1e-5, (err, np.abs(want).max())
