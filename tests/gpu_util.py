"""Helpers of the GPU parity tests: seeded inputs on the device, host copies
for the oracle, and the tolerance of the floating-point outputs.

Direction of data: the oracle sees only generator inputs (host copies of the
seeded tensors); a GPU stage may be fed the oracle's intermediates so that it
is checked in isolation.  Nothing computed by the CUDA library is ever given
to the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_routing_router_gb300 import native as N
from mixture_experts_routing_router_gb300 import synth

# max|d| <= REL * max|ref| + ABS, per tensor, for FP32-accumulated BF16 outputs
REL = 1e-2
ABS = 1e-3
W_TOL = 1e-5          # routing weights


def dev():
    return torch.device("cuda:0")


def f64(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def to_bf16_dev(a: np.ndarray) -> torch.Tensor:
    return synth.from_bf16_bits(a, dev())


def i32_dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev())


def f32_dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev())


def assert_close(got_bits, want_bits, what, rel=REL, abs_=ABS):
    g, w = f64(got_bits), f64(want_bits)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = float(np.abs(g - w).max()) if g.size else 0.0
    ref = float(np.abs(w).max()) if w.size else 0.0
    assert err <= rel * ref + abs_, f"{what}: max|d| {err:.4e} > {rel}*{ref:.4e} + {abs_}"
    # the floor must not make the check vacuous where outputs are large enough
    return err, ref


def inputs(wl, unit_scale=False, seed=0):
    """Seeded inputs generated on the GPU, plus lazy host copies."""
    return synth.make_inputs(wl, seed=seed, device=dev(), unit_scale=unit_scale)


def alloc_stage_outputs(wl):
    T, H, E, k, I = wl.tokens, wl.hidden, wl.experts, wl.top_k, wl.inter
    R = T * k
    d = dev()
    o = dict(ids=torch.empty(T, k, dtype=torch.int32, device=d), w=torch.empty(T, k, dtype=torch.float32, device=d),
             counts=torch.empty(E, dtype=torch.int32, device=d), offsets=torch.empty(E + 1, dtype=torch.int32, device=d),
             dest=torch.empty(R, dtype=torch.int32, device=d), sorted_pair=torch.empty(R, dtype=torch.int32, device=d),
             x_perm=torch.empty(R, H, dtype=torch.bfloat16, device=d), h=torch.empty(R, I, dtype=torch.bfloat16, device=d),
             y_perm=torch.empty(R, H, dtype=torch.bfloat16, device=d),
             y_shared=torch.empty(T, H, dtype=torch.bfloat16, device=d) if wl.shared else None,
             out=torch.empty(T, H, dtype=torch.bfloat16, device=d))
    return o


def run_layer(wl, g, preselected=None, stream=None):
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev())
    out = torch.empty(wl.tokens, wl.hidden, dtype=torch.bfloat16, device=dev())
    if preselected is None:
        N.moe_layer(shape, g["logits"], None, None, g["x"], g["w13"], g["w2"], g.get("ws13"), g.get("ws2"), out, ws,
                    stream)
    else:
        N.moe_layer(shape, None, preselected[0], preselected[1], g["x"], g["w13"], g["w2"], g.get("ws13"),
                    g.get("ws2"), out, ws, stream)
    return out, N.moe_status_read(ws, stream)


def oracle_expert_rows(wl, g, x_host, rows_tok, rows_exp):
    """Oracle h and y for routed rows given (token, expert) pairs, from generator inputs only."""
    hs, ys = [], []
    cache = {}
    for t, e in zip(rows_tok, rows_exp):
        if e not in cache:
            cache[e] = (bits(g["w13"][e]), bits(g["w2"][e]))
        w13e, w2e = cache[e]
        h, y = oracle.expert_row(x_host[t], w13e, w2e, wl.act)
        hs.append(h)
        ys.append(y)
    return np.stack(hs), np.stack(ys)


def oracle_token_out(wl, g, x_host, ids_o, w_o, tokens, shared_w=None):
    """Oracle out rows of sampled tokens: k routed rows each, then the combine
    (plus the shared experts), all from generator inputs."""
    outs = []
    for t in tokens:
        _, ys = oracle_expert_rows(wl, g, x_host, [t] * wl.top_k, list(ids_o[t]))
        ysh = None
        if wl.shared:
            _, ysh = oracle.shared_row(x_host[t], shared_w[0], shared_w[1], wl.act)
        outs.append(oracle.combine_row(ys, np.arange(wl.top_k, dtype=np.int32), w_o[t], ysh))
    return np.stack(outs)
