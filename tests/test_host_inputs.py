"""Host-side input preparation and byte accounting, on CPU.

The quantized-weight generators are input preparation (the library takes
codes and scales as given), so they are checked here against the oracle's
decode of what they produce: the quantization error stays within half a
step of the format, the packing is the one the entry points document, and
the block-scale padding is zero.  The bench's algorithmic byte counts per
weight format are checked against the formats' sizes."""
import os
import sys

import numpy as np
import torch

import oracle
from mixture_experts_routing_router_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fp8_quantizer_round_trips_within_half_a_step(oracle_mod):
    torch.manual_seed(0)
    w = torch.randn(3, 40, 96) * 0.02
    codes, scale = synth.quantize_rows_fp8(w)
    assert codes.dtype == torch.uint8 and codes.shape == w.shape and scale.shape == (3, 40)
    deq = oracle_mod.fp8_e4m3_decode(codes.numpy()) * scale.numpy()[..., None]
    amax = np.abs(w.numpy()).max(axis=-1, keepdims=True)
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 at and above the row's largest normal code
    err = np.abs(deq - w.numpy().astype(np.float64))
    assert np.all(err <= 2.0 ** -4 * np.abs(w.numpy()) + amax / 448 * 2.0 ** -9 + 1e-12)


def test_nvfp4_quantizer_layout_and_error(oracle_mod):
    torch.manual_seed(1)
    K = 288                                          # two 16-byte scale groups, the second partial
    w = torch.randn(2, 24, K) * 0.02
    w[0, 3] = 0.0                                    # an all-zero row
    codes, bscale, rscale = synth.quantize_rows_nvfp4(w)
    assert codes.shape == (2, 24, K // 2) and bscale.shape == (2, 24, 32) and rscale.shape == (2, 24)
    assert np.all(bscale.numpy()[..., K // 16:] == 0)            # padding
    c = codes.numpy()
    nib = np.stack([c & 15, c >> 4], axis=-1).reshape(2, 24, K)  # element 2j in the low nibble of byte j
    e = oracle_mod.fp4_e2m1_decode(nib.astype(np.uint8))
    sb = oracle_mod.fp8_e4m3_decode(bscale.numpy()[..., :K // 16])
    deq = e * np.repeat(sb, 16, axis=-1) * rscale.numpy().astype(np.float64)[..., None]
    wf = w.numpy().astype(np.float64)
    # each element is within half an E2M1 step (at most 1 at the top of the range) of w / (scales)
    step = np.repeat(sb, 16, axis=-1) * rscale.numpy().astype(np.float64)[..., None]
    assert np.all(np.abs(deq - wf) <= 1.0 * step + 1e-12)
    assert np.all(deq[0, 3] == 0)
    # the block scale makes each block's largest magnitude land near the top code (6)
    blk = np.abs(wf).reshape(2, 24, K // 16, 16).max(axis=-1)
    big = blk > 1e-6
    ratio = blk[big] / (sb[big] * np.repeat(rscale.numpy()[..., None], K // 16, axis=-1)[big])
    assert np.all((ratio > 5.0) & (ratio < 7.0))


def test_bench_weight_bytes_per_format():
    sys.path.insert(0, ROOT)
    import bench
    K = 7168
    assert bench.weight_row_bytes(K, "bf16") == 2 * K
    assert bench.weight_row_bytes(K, "fp8") == K + 4
    assert bench.weight_row_bytes(K, "nvfp4") == K // 2 + K // 16 + 4
    wl = synth.WORKLOADS["decode_16_distinct"]
    counts = np.zeros(wl.experts, np.int64)
    counts[:144] = 1
    a = bench.algorithmic(wl, counts, "nvfp4")
    R = wl.tokens * wl.top_k
    H, I = wl.hidden, wl.inter
    assert a["up_bytes"] == 144 * wl.up * (H // 2 + H // 16 + 4) + R * H * 2 + R * I * 2
    assert a["down_bytes"] == 144 * H * (I // 2 + I // 16 + 4) + R * I * 2 + R * H * 2
    assert a["nonempty_experts"] == 144
