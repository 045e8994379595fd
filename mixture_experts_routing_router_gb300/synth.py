"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws numbers: it holds none of the layer's arithmetic
(no routing, counting, permuting, FFN or combine).  The same tensors feed the
GPU library and the CPU oracle.  Every draw comes from a ``torch.Generator``
seeded from (seed, tensor tag), so a tensor does not depend on which other
tensors were drawn before it.  Generation runs on the device the caller names:
the CPU for the small workloads, the GPU for the 22.5 GB of weights of the
large layer.  Draws are reproducible per device type, not across CPU and GPU.

Workloads (shapes and value laws of the pages' workloads):
  tiny          64 tokens, H 256, E 16, top-2, I 512, SwiGLU, x and W ~ N(0, 0.02)
  count_first   2048 tokens, H 2048, E 128, top-8, I 768, SwiGLU, capacity 2048
                (afdEP-comm count-first validation record, .setup)
  decode        1/8/16 rows, H 1024, E 240, top-9, I 1536, ReLU^2, selected
                logits +16 and the rest -16, routes shared or distinct
                (ONNX Runtime PR #33963, "Measured CUDA kernel latency")
  deepseek      1024 tokens, H 2048, E 64, top-6, I 1408, SwiGLU, plus two
                always-on shared experts of intermediate 1408
                (DeepSeek fleet megakernel REPORT.md, model shape);
                deepseek_routed is the same without the shared experts
  large         16384 tokens, H 7168, E 256, top-8, I 2048, SwiGLU, logits
                N(0,1) plus a Zipf(1.2) expert bias (hot experts)
Router logits are N(0,1) unless stated; x ~ N(0,1) and W ~ N(0, 0.02) where a
workload gives no activation scale.  ``unit_scale=True`` gives the twin with
x ~ N(0,1) and W ~ N(0, 1/sqrt(fan_in)), whose outputs are O(1) so a
tolerance of 1e-2 * max|ref| + 1e-3 is not met trivially.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import torch

ACT_SWIGLU = 0
ACT_RELU2 = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    hidden: int
    experts: int
    top_k: int
    inter: int
    act: int = ACT_SWIGLU
    shared: int = 0
    shared_inter: int = 0
    capacity: int = 0          # 0: the number of tokens
    x_std: float = 1.0
    w_std: float = 0.02
    logits: str = "normal"     # normal | zipf | pm16_shared | pm16_distinct
    zipf_s: float = 1.2

    @property
    def up(self) -> int:
        return 2 * self.inter if self.act == ACT_SWIGLU else self.inter

    @property
    def shared_up(self) -> int:
        return 2 * self.shared_inter if self.act == ACT_SWIGLU else self.shared_inter

    @property
    def pairs(self) -> int:
        return self.tokens * self.top_k

    @property
    def cap(self) -> int:
        return self.capacity if self.capacity > 0 else self.tokens

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 16, 2, 512, x_std=0.02),
    "count_first": Workload("count_first", 2048, 2048, 128, 8, 768, capacity=2048),
    "deepseek": Workload("deepseek", 1024, 2048, 64, 6, 1408, shared=2, shared_inter=1408),
    "large": Workload("large", 16384, 7168, 256, 8, 2048, logits="zipf"),
    # the DeepSeek shape without its shared experts (the quantized entry points
    # take routed experts only)
    "deepseek_routed": Workload("deepseek_routed", 1024, 2048, 64, 6, 1408),
    # profiling case of the large layer's kernels: same hidden / intermediate /
    # top-k, 32 experts and 4096 tokens (about 3 GB on the device)
    "large_e32": Workload("large_e32", 4096, 7168, 32, 8, 2048, logits="zipf"),
}
for _rows in (1, 8, 16):
    for _kind in ("shared", "distinct"):
        WORKLOADS[f"decode_{_rows}_{_kind}"] = Workload(
            f"decode_{_rows}_{_kind}", _rows, 1024, 240, 9, 1536, act=ACT_RELU2,
            logits=f"pm16_{_kind}")


def _gen(seed: int, tag: str, device) -> torch.Generator:
    h = hashlib.sha256(f"{seed}/{tag}".encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def normal(shape, std, seed, tag, device="cpu", dtype=torch.bfloat16):
    """N(0, std^2) draws, rounded once to ``dtype``."""
    g = _gen(seed, tag, device)
    if dtype == torch.float32:
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        return t.mul_(std)
    # draw in float32 in bounded chunks, scale, round once to bf16
    out = torch.empty(shape, device=device, dtype=dtype)
    flat = out.view(-1)
    n = flat.numel()
    chunk = 1 << 28
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        t = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        flat[s:e] = t.mul_(std)
    return out


def decode_route_sets(wl: Workload):
    """Expert sets of the decode workload: 'shared' gives every row experts
    {0..k-1}; 'distinct' gives row r experts {k*r .. k*r+k-1}."""
    rows, k = wl.tokens, wl.top_k
    if wl.logits == "pm16_shared":
        return [list(range(k)) for _ in range(rows)]
    return [list(range(k * r, k * r + k)) for r in range(rows)]


def make_logits(wl: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    T, E = wl.tokens, wl.experts
    if wl.logits.startswith("pm16"):
        lg = torch.full((T, E), -16.0, dtype=torch.float32)
        for r, s in enumerate(decode_route_sets(wl)):
            lg[r, s] = 16.0
        return lg.to(device)
    lg = normal((T, E), 1.0, seed, "logits", device, torch.float32)
    if wl.logits == "zipf":
        # A seeded random ranking of the experts; expert of rank r (0-based)
        # gets bias -s * ln(r + 1), the log of a Zipf(s) pmf up to a constant.
        g = _gen(seed, "zipf_rank", "cpu")
        rank = torch.randperm(E, generator=g)
        bias = -wl.zipf_s * torch.log(rank.to(torch.float64) + 1.0)
        lg += bias.to(torch.float32).to(device)[None, :]
    return lg


def make_inputs(wl: Workload, seed: int = 0, device="cpu", unit_scale: bool = False,
                weights: bool = True) -> dict:
    """All inputs of one layer call as torch tensors on ``device``:
    logits f32 [T,E], x bf16 [T,H], w13 bf16 [E,up,H], w2 bf16 [E,H,I],
    and ws13 [S,shared_up,H], ws2 [S,H,Is] when the workload has shared experts."""
    T, H, E, I = wl.tokens, wl.hidden, wl.experts, wl.inter
    x_std = 1.0 if unit_scale else wl.x_std
    d = {"logits": make_logits(wl, seed, device),
         "x": normal((T, H), x_std, seed, "x", device)}
    if weights:
        d["w13"] = torch.empty((E, wl.up, H), dtype=torch.bfloat16, device=device)
        d["w2"] = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
        for e in range(E):
            d["w13"][e], d["w2"][e] = expert_weights(wl, e, seed, device, unit_scale)
        if wl.shared > 0:
            d["ws13"] = torch.empty((wl.shared, wl.shared_up, H), dtype=torch.bfloat16, device=device)
            d["ws2"] = torch.empty((wl.shared, H, wl.shared_inter), dtype=torch.bfloat16, device=device)
            for s in range(wl.shared):
                d["ws13"][s], d["ws2"][s] = shared_expert_weights(wl, s, seed, device, unit_scale)
    return d


def expert_weights(wl: Workload, e: int, seed: int = 0, device="cpu", unit_scale: bool = False):
    """(W13[e] [up,H], W2[e] [H,I]) of routed expert e, drawn from streams of
    their own, so one expert can be regenerated without the others."""
    H, I = wl.hidden, wl.inter
    s13 = 1.0 / math.sqrt(H) if unit_scale else wl.w_std
    s2 = 1.0 / math.sqrt(I) if unit_scale else wl.w_std
    return (normal((wl.up, H), s13, seed, f"w13/{e}", device),
            normal((H, I), s2, seed, f"w2/{e}", device))


def shared_expert_weights(wl: Workload, s: int, seed: int = 0, device="cpu", unit_scale: bool = False):
    H, Is = wl.hidden, wl.shared_inter
    s13 = 1.0 / math.sqrt(H) if unit_scale else wl.w_std
    s2 = 1.0 / math.sqrt(Is) if unit_scale else wl.w_std
    return (normal((wl.shared_up, H), s13, seed, f"ws13/{s}", device),
            normal((H, Is), s2, seed, f"ws2/{s}", device))


def quantize_rows_fp8(w: torch.Tensor):
    """Input preparation for FP8 expert weights: each row of ``w`` [..., rows, K]
    becomes E4M3 codes (torch's round-to-nearest float8_e4m3fn conversion) of
    w / scale with scale = max|row| / 448 (1 for an all-zero row).
    -> (codes uint8 [..., rows, K], scale float32 [..., rows])."""
    wf = w.float()
    amax = wf.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (wf / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.squeeze(-1).contiguous()


def make_fp8_weights(wl: Workload, seed: int = 0, device="cpu", unit_scale: bool = False) -> dict:
    """FP8 E4M3 expert weights with one FP32 scale per weight row, quantized
    from the same per-expert BF16 draws as make_inputs:
    w13 uint8 [E, up, H], s13 float32 [E, up], w2 uint8 [E, H, I], s2 float32 [E, H]."""
    E, H, I = wl.experts, wl.hidden, wl.inter
    d = {"w13": torch.empty((E, wl.up, H), dtype=torch.uint8, device=device),
         "s13": torch.empty((E, wl.up), dtype=torch.float32, device=device),
         "w2": torch.empty((E, H, I), dtype=torch.uint8, device=device),
         "s2": torch.empty((E, H), dtype=torch.float32, device=device)}
    for e in range(E):
        a, b = expert_weights(wl, e, seed, device, unit_scale)
        d["w13"][e], d["s13"][e] = quantize_rows_fp8(a)
        d["w2"][e], d["s2"][e] = quantize_rows_fp8(b)
    return d


E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_rows_nvfp4(w: torch.Tensor):
    """Input preparation for NVFP4 expert weights: each row of ``w`` [..., rows,
    K] (K a multiple of 16) gets a row scale max|row| / (6 * 448) (1 for an
    all-zero row), E4M3 block scales (torch's round-to-nearest float8_e4m3fn
    conversion) of max|block| / (6 * row scale) per 16 elements, and E2M1
    codes of w / (block scale * row scale) rounded to the nearest magnitude.
    -> (codes uint8 [..., rows, K/2], two per byte, low nibble first;
        bscale uint8 [..., rows, 16*ceil(K/256)], zero padded;
        scale float32 [..., rows])."""
    wf = w.float()
    K = wf.shape[-1]
    amax = wf.abs().amax(dim=-1, keepdim=True)
    rs = torch.where(amax > 0, amax / (6.0 * 448.0), torch.ones_like(amax))
    blk = wf.unflatten(-1, (K // 16, 16))
    bmax = blk.abs().amax(dim=-1) / (6.0 * rs)
    bs = bmax.to(torch.float8_e4m3fn)
    bsf = bs.float()
    v = blk / torch.where(bsf > 0, bsf, torch.ones_like(bsf)).unsqueeze(-1) / rs.unsqueeze(-1)
    mags = torch.tensor(E2M1_MAGNITUDES, device=w.device)
    mid = (mags[1:] + mags[:-1]) / 2
    code = torch.bucketize(v.abs(), mid) | torch.where(v < 0, 8, 0)
    code = code.flatten(-2).to(torch.uint8)
    codes = (code[..., 0::2] | (code[..., 1::2] << 4)).contiguous()
    bscale = torch.zeros(wf.shape[:-1] + (16 * ((K + 255) // 256),), dtype=torch.uint8, device=w.device)
    bscale[..., :K // 16] = bs.view(torch.uint8)
    return codes, bscale, rs.squeeze(-1).contiguous()


def make_nvfp4_weights(wl: Workload, seed: int = 0, device="cpu", unit_scale: bool = False) -> dict:
    """NVFP4 expert weights quantized from the same per-expert BF16 draws as
    make_inputs: w13 uint8 [E, up, H/2], b13 uint8 [E, up, 16*ceil(H/256)],
    s13 float32 [E, up]; w2 uint8 [E, H, I/2], b2 uint8 [E, H, 16*ceil(I/256)],
    s2 float32 [E, H]."""
    E, H, I = wl.experts, wl.hidden, wl.inter
    d = {"w13": torch.empty((E, wl.up, H // 2), dtype=torch.uint8, device=device),
         "b13": torch.empty((E, wl.up, 16 * ((H + 255) // 256)), dtype=torch.uint8, device=device),
         "s13": torch.empty((E, wl.up), dtype=torch.float32, device=device),
         "w2": torch.empty((E, H, I // 2), dtype=torch.uint8, device=device),
         "b2": torch.empty((E, H, 16 * ((I + 255) // 256)), dtype=torch.uint8, device=device),
         "s2": torch.empty((E, H), dtype=torch.float32, device=device)}
    for e in range(E):
        a, b = expert_weights(wl, e, seed, device, unit_scale)
        d["w13"][e], d["b13"][e], d["s13"][e] = quantize_rows_nvfp4(a)
        d["w2"][e], d["b2"][e], d["s2"][e] = quantize_rows_nvfp4(b)
    return d


def gate_weights(wl: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    """Router projection W_gate [E, H] ~ N(0, 1/H): x ~ N(0,1) gives logits of
    about unit scale."""
    return normal((wl.experts, wl.hidden), 1.0 / math.sqrt(wl.hidden), seed, "w_gate", device)


def correction_bias(wl: Workload, seed: int = 0, device="cpu", std: float = 0.05) -> torch.Tensor:
    """FP32 selection-only routing bias [E] ~ N(0, std^2)."""
    return normal((wl.experts,), std, seed, "bias", device, torch.float32)


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's bit patterns as a numpy uint16 array (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def from_bf16_bits(a, device="cpu") -> torch.Tensor:
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
