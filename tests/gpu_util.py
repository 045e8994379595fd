"""Helpers of the GPU parity tests: seeded inputs on the device, host copies
for the oracle, and the tolerance of the floating-point outputs.

Direction of data: the oracle sees only generator inputs (host copies of the
seeded tensors); a GPU stage may be fed the oracle's intermediates so that it
is checked in isolation.  Nothing computed by the CUDA library is ever given
to the oracle.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

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


def oracle_threads() -> int:
    """Host threads for the oracle's independent rows (ctypes releases the GIL
    inside the C++ oracle, which keeps no shared state between calls)."""
    return max(1, min(os.cpu_count() or 1, 32))


def oracle_rows_parallel(wl, g, x_host, pairs):
    """Oracle (h, y) of routed rows, given unique (token, expert) pairs, from
    generator inputs only.  Rows are grouped by expert so each expert's
    weights are copied to the host once; the rows of an expert run on a pool
    of host threads.  -> dict (token, expert) -> (h_row, y_row)."""
    by_e = {}
    for t, e in pairs:
        by_e.setdefault(int(e), []).append(int(t))
    res = {}
    with cf.ThreadPoolExecutor(oracle_threads()) as ex:
        for e, toks in sorted(by_e.items()):
            w13e, w2e = bits(g["w13"][e]), bits(g["w2"][e])
            for t, hy in zip(toks, ex.map(lambda t: oracle.expert_row(x_host[t], w13e, w2e, wl.act), toks)):
                res[(t, e)] = hy
    return res


def oracle_shared_rows_parallel(wl, g, x_host, tokens):
    """Oracle y_shared rows of the given tokens (generator inputs only)."""
    ws13, ws2 = bits(g["ws13"]), bits(g["ws2"])
    with cf.ThreadPoolExecutor(oracle_threads()) as ex:
        ys = list(ex.map(lambda t: oracle.shared_row(x_host[t], ws13, ws2, wl.act)[1], tokens))
    return np.stack(ys)
