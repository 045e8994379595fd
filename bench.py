"""Benchmark of the MoE layer hot path on one GB300 (or N data-parallel replicas).

One step = one moe_layer call (captured once in a CUDA graph and replayed) over the large workload: 16384 tokens, hidden
7168, 256 experts top-8, intermediate 2048, SwiGLU, Zipf(1.2)-biased router
logits -- route, count-first dispatch, grouped expert FFN and combine.  Inputs
(22.5 GB of weights, 235 MB of x) are larger than the 129 MB L2, so no flush
is needed between steps.  Under torchrun every rank runs its own replica on its
own 16384 tokens (weak scaling, no data-path collective); the elapsed time is
the max over ranks.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
prints one JSON line.  --impl reference times the CPU oracle (the program the
GPU path is checked against) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_routing_router_gb300 import synth  # noqa: E402

WORKLOAD = "large"
METRIC = "MoE layer tokens/s; dispatch+combine HBM GB/s; expert GEMM TFLOP/s vs peak"


def describe(wl):
    return (f"{wl.name}: {wl.tokens} tokens, hidden {wl.hidden}, {wl.experts} experts top-{wl.top_k}, "
            f"intermediate {wl.inter}, {'SwiGLU' if wl.act == 0 else 'ReLU^2'}, "
            f"router logits N(0,1)" + (f" + Zipf({wl.zipf_s}) expert bias" if wl.logits == "zipf" else "")
            + ", W ~ N(0,0.02), x ~ N(0,1), seed 0")


def weight_row_bytes(K, wfmt="bf16"):
    """Bytes of one expert weight row of K elements: BF16 2 per element; FP8 1
    per element + a 4-byte row scale; NVFP4 half a byte per element + one
    E4M3 block scale per 16 elements + a 4-byte row scale."""
    if wfmt == "fp8":
        return K + 4
    if wfmt == "nvfp4":
        return K // 2 + K // 16 + 4
    return 2 * K


def algorithmic(wl, counts=None, wfmt="bf16"):
    """Bytes / FLOPs the method itself must move or compute (no padding)."""
    T, H, E, k, I = wl.tokens, wl.hidden, wl.experts, wl.top_k, wl.inter
    R = T * k
    up = wl.up
    d = {
        "dispatch_bytes": T * H * 2 + R * H * 2 + R * 8 + E * 8,
        "combine_bytes": R * H * 2 + T * H * 2 + R * 8,
        "up_flops": 2 * R * H * up + 2 * T * H * wl.shared * wl.shared_up,
        "down_flops": 2 * R * I * H + 2 * T * wl.shared * wl.shared_inter * H,
    }
    if counts is not None:
        nz = int((counts > 0).sum())
        d["nonempty_experts"] = nz
        d["up_bytes"] = nz * up * weight_row_bytes(H, wfmt) + R * H * 2 + R * I * 2
        d["down_bytes"] = nz * H * weight_row_bytes(I, wfmt) + R * I * 2 + R * H * 2
    return d


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


WEIGHT_FORMATS = {
    "bf16": "BF16",
    "fp8": "FP8 E4M3 codes + one FP32 scale per weight row (quantized from the BF16 draws); BF16 activations and MMA",
    "nvfp4": ("NVFP4: E2M1 codes + one E4M3 scale per 16 elements + one FP32 scale per weight row (quantized from "
              "the BF16 draws); BF16 activations and MMA"),
}


def fused_decode(wl, wfmt):
    """Whether moe_layer runs the fused decode FFN (expert up, down and the
    combine in one kernel after the fused dispatch): the library's own host
    rule -- BF16 weights, 2 to 16 tokens, no shared experts, hidden and
    intermediate whole 64-column chunks."""
    return (wfmt == "bf16" and 2 <= wl.tokens <= 16 and wl.shared == 0 and wl.hidden % 64 == 0 and
            wl.inter % 64 == 0 and wl.act in (synth.ACT_SWIGLU, synth.ACT_RELU2))


def up_kernel_name(wl, sms, quant=False):
    """Which kernel the library runs for the up projection (the library's own
    host rule: the small-row kernel for quantized weights, or when a group
    holds at most 64 rows and its items fit in two waves; the CTA-pair kernel
    when groups average 256 rows)."""
    R = wl.tokens * wl.top_k
    if quant or (wl.tokens <= 64 and min(wl.experts, R) * ((wl.inter + 127) // 128) <= 2 * sms):
        return "decode_gemm_kernel (expert up projection)"
    if R // wl.experts >= 256:
        return "grouped_gemm_pair_kernel (expert up projection)"
    return "grouped_gemm_kernel (expert up projection)"


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("common.cuh", "gemm.cu"):
        h.update(open(os.path.join(ROOT, "mixture_experts_routing_router_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per launch of the up-projection GEMM from the committed ncu
    summary, only while the kernel source is the one that was captured."""
    p = os.path.join(ROOT, "profiles", "gemm_up_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_source_sha") != kernel_source_sha():
        return None
    return d.get("dram_bytes_per_launch_full_size")


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest value over all ranks (timing only; no data-path collective)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def host_description():
    """The host the oracle runs on: logical CPUs and the CPU model."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "cpu model"):
            for ln in info.splitlines():
                if ln.lower().startswith(key.lower()) and ":" in ln:
                    model = ln.split(":", 1)[1].strip()
                    break
            if model:
                break
        if not model:       # Arm: implementer / part numbers
            parts = {ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU part")}
            impl = {ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU implementer")}
            if parts:
                model = f"Arm CPU implementer {'/'.join(sorted(impl))} part {'/'.join(sorted(parts))}"
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown"}


def oracle_macs_per_token(wl):
    """Multiply-adds of the oracle per token: k routed rows plus the shared experts."""
    H, I, up = wl.hidden, wl.inter, wl.up
    return wl.top_k * (H * up + I * H) + wl.shared * (H * wl.shared_up + wl.shared_inter * H)


def oracle_sample(wl, g_logits_host, x_host, tokens, weight_device, seed=0, threads=1):
    """Time the oracle on `tokens` tokens of the workload: routing of those
    tokens, their k expert rows (up projection, activation, down projection)
    and the combine, the rows on a pool of `threads` host threads (the C++
    oracle releases the interpreter lock).  Expert weights are regenerated
    from their seeded streams one expert at a time, outside the timed part.
    Returns (seconds, tokens)."""
    import concurrent.futures as cf

    import oracle
    from mixture_experts_routing_router_gb300.synth import bf16_bits, expert_weights
    t0 = time.perf_counter()
    _, ids, w = oracle.route(g_logits_host[tokens], wl.top_k)
    timed = time.perf_counter() - t0
    by_e = {}
    for i in range(len(tokens)):
        for j in range(wl.top_k):
            by_e.setdefault(int(ids[i, j]), []).append((i, j))
    ys = {}
    with cf.ThreadPoolExecutor(threads) as ex:
        for e, rows in sorted(by_e.items()):
            a, b = expert_weights(wl, e, seed, weight_device)
            w13e, w2e = bf16_bits(a), bf16_bits(b)
            t0 = time.perf_counter()
            res = list(ex.map(lambda ij: oracle.expert_row(x_host[tokens[ij[0]]], w13e, w2e, wl.act)[1], rows))
            timed += time.perf_counter() - t0
            for ij, y in zip(rows, res):
                ys[ij] = y
    t0 = time.perf_counter()
    for i in range(len(tokens)):
        oracle.combine_row(np.stack([ys[(i, j)] for j in range(wl.top_k)]), np.arange(wl.top_k, dtype=np.int32), w[i])
    timed += time.perf_counter() - t0
    return timed, len(tokens)


def oracle_full(wl, g):
    """Time the whole oracle layer, single-threaded, on the workload's batch."""
    import oracle
    kw = dict(ws13=synth.bf16_bits(g["ws13"]), ws2=synth.bf16_bits(g["ws2"])) if wl.shared else {}
    x, w13, w2 = synth.bf16_bits(g["x"]), synth.bf16_bits(g["w13"]), synth.bf16_bits(g["w2"])
    lg = g["logits"].cpu().numpy()
    t0 = time.perf_counter()
    ref = oracle.layer(x, w13, w2, wl.act, wl.top_k, wl.cap, logits=lg, **kw)
    secs = time.perf_counter() - t0
    assert ref["status"] == 0
    return secs


# The oracle's rate, roughly (FP64 multiply-adds per second per core): sizes the
# bounded sample so the CPU baseline stays at about 20 core-seconds.
ORACLE_MACS_PER_CORE_S = 1.0e9
CPU_BUDGET_CORE_S = 20.0


def cpu_baseline(wl, g, dev, seed):
    """The oracle on the machine's host cores.  Workloads whose whole oracle layer
    fits the budget run it in full, single-threaded (the oracle as it stands);
    larger ones time a seeded sample of tokens with the rows spread over every
    host core, the thread count stated."""
    host = host_description()
    T = wl.tokens
    per_tok = oracle_macs_per_token(wl)
    if T * per_tok <= CPU_BUDGET_CORE_S * ORACLE_MACS_PER_CORE_S and g.get("w13") is not None:
        secs = oracle_full(wl, g)
        return {"value": T / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle", **host,
                "sample": f"the whole {T}-token layer (routing, dispatch, expert FFN with FP64 sums, combine), "
                          f"single-threaded, {secs:.1f} s"}
    threads = max(1, os.cpu_count() or 1)
    n = int(min(T, max(8, CPU_BUDGET_CORE_S * ORACLE_MACS_PER_CORE_S // per_tok)))
    rng = np.random.default_rng(0)
    toks = sorted(rng.choice(T, n, replace=False).tolist())
    secs, n = oracle_sample(wl, g["logits"].cpu().numpy(), synth.bf16_bits(g["x"]), toks, dev, seed=seed,
                            threads=threads)
    return {"value": n / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle", **host,
            "sample": f"{n} seeded random tokens of the {T}-token batch: their routing, top-{wl.top_k} expert rows "
                      f"(FP64 sums, rows spread over {threads} host threads) and combine; {secs:.1f} s wall"}


def run_reference(args, wl, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    logits = synth.make_logits(wl, 0, dev).cpu().numpy()
    x = synth.bf16_bits(synth.normal((wl.tokens, wl.hidden), 1.0, 0, "x", dev))
    rng = np.random.default_rng(0)
    threads = max(1, os.cpu_count() or 1)
    # each step a bounded sample: as many tokens as there are host threads
    per_step = min(wl.tokens, threads)
    times, toks = [], 0
    for step in range(args.warmup + args.steps):
        tokens = sorted(rng.choice(wl.tokens, per_step, replace=False).tolist())
        s, n = oracle_sample(wl, logits, x, tokens, dev, threads=threads)
        if step >= args.warmup:
            times.append(s)
            toks += n
    total = sum(times)
    value = toks / total
    sample = (f"{per_step} seeded random token(s) per step of the {wl.tokens}-token batch: routing, the top-{wl.top_k} "
              f"expert rows (FP64 sums, spread over {threads} host threads) and the combine")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": describe(wl), "tokens_per_step": per_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             **host_description(), "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def capture(fn, stream):
    """A CUDA graph of the work `fn` enqueues on `stream`."""
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    return graph


def ws_counts(N, shape, g, ws, stream, dev):
    """Per-expert counts of this workload's routing (one route + dispatch)."""
    T, k, E, H = shape.tokens, shape.top_k, shape.experts, shape.hidden
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    dest = torch.empty(T * k, dtype=torch.int32, device=dev)
    sp = torch.empty(T * k, dtype=torch.int32, device=dev)
    xp = torch.empty(T * k, H, dtype=torch.bfloat16, device=dev)
    N.moe_route(shape, g["logits"], ids, w, ws, stream)
    N.moe_dispatch(shape, g["x"], ids, counts, offsets, dest, sp, xp, ws, stream)
    stream.synchronize()
    return counts.cpu().numpy()


def run_native(args, wl, world, rank, local):
    from mixture_experts_routing_router_gb300 import native as N
    N.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    wfmt = args.weights
    quant = wfmt != "bf16"
    if quant and wl.shared:
        raise SystemExit("quantized expert weights: the workload has shared experts, which the quantized entry "
                         "points omit")
    g = synth.make_inputs(wl, seed=rank, device=dev, weights=not quant)
    q = (synth.make_fp8_weights(wl, seed=rank, device=dev) if wfmt == "fp8" else
         synth.make_nvfp4_weights(wl, seed=rank, device=dev) if wfmt == "nvfp4" else None)
    shape = N.shape_of(wl)
    ws = N.workspace(shape, dev)
    T, H, E, k, I = wl.tokens, wl.hidden, wl.experts, wl.top_k, wl.inter
    R = T * k
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    # route, count (+ clearing its look-back state when R > 1024 pairs), scatter
    # -- one fused kernel for batches of at most 16 tokens --, up, down, combine
    # (+ the shared experts' up and down)
    # -- or, from 2 to 16 tokens, the fused dispatch and the fused decode FFN
    dispatch_kernels = 1 if T <= 16 else 3 + (1 if R > 1024 else 0)
    fused = fused_decode(wl, wfmt)
    kernels_per_layer = 2 if fused else dispatch_kernels + 3 + (2 if wl.shared else 0)

    def layer_on(lg_d, x_d, out_d):
        if wfmt == "fp8":
            N.moe_layer_fp8(shape, lg_d, None, None, x_d, q["w13"], q["s13"], q["w2"], q["s2"], out_d, ws, stream)
        elif wfmt == "nvfp4":
            N.moe_layer_nvfp4(shape, lg_d, None, None, x_d, q["w13"], q["b13"], q["s13"], q["w2"], q["b2"], q["s2"],
                              out_d, ws, stream)
        else:
            N.moe_layer(shape, lg_d, None, None, x_d, g["w13"], g["w2"], g.get("ws13"), g.get("ws2"), out_d, ws,
                        stream)

    def layer():
        layer_on(g["logits"], g["x"], out)

    # L2: the large layer's inputs (x 235 MB, 22.5 GB of weights) exceed it;
    # smaller workloads get a write of 4x L2 before every timed step instead,
    # outside the step's own event pair.
    with torch.cuda.stream(stream):
        layer()
    stream.synchronize()
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20) or 126 * 2**20
    cnt0 = ws_counts(N, shape, g, ws, stream, dev)
    touched = int((cnt0 > 0).sum()) * (wl.up * weight_row_bytes(H, wfmt) + H * weight_row_bytes(I, wfmt)) + \
        wl.shared * (wl.shared_up * H + H * wl.shared_inter) * 2
    flush = not (g["x"].numel() * 2 > l2 and touched > 4 * l2)
    flush_buf = torch.empty(4 * l2, dtype=torch.uint8, device=dev) if flush else None
    # then a read of another buffer of 4x L2: the flush write leaves L2 full of
    # its own dirty lines, whose write-back would otherwise land inside the next
    # timed step (measured: 4 us of the one-token decode layer, 14 us of the
    # 16-token one); after the read, L2 holds clean lines of neither the layer's
    # inputs nor its weights
    clean_buf = torch.empty(4 * l2 // 8, dtype=torch.int64, device=dev) if flush else None
    clean_sink = torch.empty(1, dtype=torch.int64, device=dev) if flush else None

    def flush_l2(i):
        if flush_buf is not None:
            flush_buf.fill_(i & 0xFF)
            torch.sum(clean_buf, dim=0, keepdim=True, out=clean_sink)

    # ---- headline: K whole-layer steps, each a replay of the captured layer ----
    # (moe_layer enqueues only: it is captured once in a CUDA graph, so a step
    # costs the GPU work and one graph launch, not one host call per kernel)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            layer()
    stream.synchronize()
    st = N.moe_status_read(ws, stream)
    if st != N.MOE_OK:
        raise RuntimeError(f"device status {st} after warm-up")
    layer_graph = capture(layer, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            layer_graph.replay()
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            # one event per step boundary: back to back when no flush is needed
            # (the steps' total is first start to last end), else around each step
            pairs = []
            prev = None
            for i in range(args.steps):
                if flush:
                    flush_l2(i)
                    prev = None
                a = prev if prev is not None else torch.cuda.Event(enable_timing=True)
                if prev is None:
                    a.record(stream)
                b = torch.cuda.Event(enable_timing=True)
                layer_graph.replay()
                b.record(stream)
                pairs.append((a, b))
                prev = None if flush else b
        stream.synchronize()
    torch.cuda.synchronize(dev)
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in pairs]
    elapsed = sum(step_ms) / 1e3
    elapsed = max_over_ranks(elapsed, world, dev)
    tokens_per_s = world * T * args.steps / elapsed
    # spread of the steps: median, p95, and the drift between the first and
    # the last tenth of the run (flagged above 2 %)
    tenth = max(1, len(step_ms) // 10)
    first, last = statistics.mean(step_ms[:tenth]), statistics.mean(step_ms[-tenth:])
    step_stats = {"median_ms": statistics.median(step_ms),
                  "p95_ms": float(np.percentile(step_ms, 95)),
                  "drift_first_to_last": (last - first) / first,
                  "unstable": abs(last - first) / first > 0.02}

    # ---- per-stage times (same stream, events between the stage calls) --------
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    dest = torch.empty(R, dtype=torch.int32, device=dev)
    sp = torch.empty(R, dtype=torch.int32, device=dev)
    x_perm = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    h = torch.empty(R, I, dtype=torch.bfloat16, device=dev)
    y_perm = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    y_sh = torch.empty(T, H, dtype=torch.bfloat16, device=dev) if wl.shared else None
    names = ["route", "dispatch", "expert_up", "expert_down", "combine"]
    stage_fns = [
        lambda: N.moe_route(shape, g["logits"], ids, w, ws, stream),
        lambda: N.moe_dispatch(shape, g["x"], ids, counts, offsets, dest, sp, x_perm, ws, stream),
        (lambda: N.moe_expert_up_fp8(shape, x_perm, offsets, q["w13"], q["s13"], h, ws, stream)) if wfmt == "fp8"
        else (lambda: N.moe_expert_up_nvfp4(shape, x_perm, offsets, q["w13"], q["b13"], q["s13"], h, ws, stream))
        if wfmt == "nvfp4" else
        (lambda: N.moe_expert_up(shape, x_perm, offsets, g["w13"], g["x"], g.get("ws13"), h, ws, stream)),
        (lambda: N.moe_expert_down_fp8(shape, h, offsets, q["w2"], q["s2"], y_perm, ws, stream)) if wfmt == "fp8"
        else (lambda: N.moe_expert_down_nvfp4(shape, h, offsets, q["w2"], q["b2"], q["s2"], y_perm, ws, stream))
        if wfmt == "nvfp4" else
        (lambda: N.moe_expert_down(shape, h, offsets, g["w2"], g.get("ws2"), y_perm, y_sh, ws, stream)),
        lambda: N.moe_combine(shape, y_perm, dest, w, y_sh, out, ws, stream),
    ]
    with torch.cuda.stream(stream):
        for fn in stage_fns:
            fn()
    stream.synchronize()
    stage_graphs = [capture(fn, stream) for fn in stage_fns]
    reps = max(3, min(args.steps, 20))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(reps)]
    with torch.cuda.stream(stream):
        for r in range(reps + 2):
            e = evs[r - 2] if r >= 2 else None
            flush_l2(r)
            for i, sg in enumerate(stage_graphs):
                if e: e[i].record(stream)
                sg.replay()
            if e: e[len(names)].record(stream)
    stream.synchronize()
    stage_ms = {n: statistics.median(evs[r][i].elapsed_time(evs[r][i + 1]) for r in range(reps))
                for i, n in enumerate(names)}

    # ---- router front end (not part of the layer step): gate projection and
    # sigmoid routing with a correction bias, timed the same way --------------
    w_gate = synth.gate_weights(wl, seed=rank, device=dev)
    bias = synth.correction_bias(wl, seed=rank, device=dev)
    logits_g = torch.empty(T, E, dtype=torch.float32, device=dev)
    front_fns = [lambda: N.moe_gate(shape, g["x"], w_gate, logits_g, ws, stream),
                 lambda: N.moe_route_sigmoid(shape, logits_g, bias, 2.5, ids, w, ws, stream)]
    with torch.cuda.stream(stream):
        for fn in front_fns:
            fn()
    stream.synchronize()
    front_graphs = [capture(fn, stream) for fn in front_fns]
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    with torch.cuda.stream(stream):
        for r in range(reps + 2):
            e = fevs[r - 2] if r >= 2 else None
            flush_l2(r)
            for i, fg in enumerate(front_graphs):
                if e: e[i].record(stream)
                fg.replay()
            if e: e[2].record(stream)
    stream.synchronize()
    gate_ms = statistics.median(fevs[r][0].elapsed_time(fevs[r][1]) for r in range(reps))
    rsig_ms = statistics.median(fevs[r][1].elapsed_time(fevs[r][2]) for r in range(reps))
    router_front = {"gate_ms": gate_ms, "gate_tflops": 2.0 * T * H * E / (gate_ms / 1e3) / 1e12,
                    "route_sigmoid_ms": rsig_ms}
    st = N.moe_status_read(ws, stream)
    if st != N.MOE_OK:
        raise RuntimeError(f"device status {st} after stage timing")
    cnt = counts.cpu().numpy()
    alg = algorithmic(wl, cnt, wfmt)

    # ---- end to end through the C-ABI with host buffers -----------------------
    # Every step copies its inputs (x, logits) from pinned host memory, runs
    # moe_layer and copies its output back, all inside the timed region.  For
    # the large layer the steps are pipelined as a serving loop would run them:
    # step i+1's input copy and step i-1's output copy (copy engines, streams of
    # their own) overlap step i's layer, with double-buffered device buffers.
    # Smaller workloads flush L2 before every step, so their steps run one
    # after another.
    x_host = g["x"].cpu().pin_memory()
    lg_host = g["logits"].cpu().pin_memory()
    e2e_clk = ClockSampler(local)
    e2e_clk.__enter__()
    # as many steps as the headline, so both run in the same (power-capped) state
    e2e_steps = max(3, args.steps)

    def run_layer_on(lg_d, x_d, out_d):
        layer_on(lg_d, x_d, out_d)

    if not flush:
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        x_d = [torch.empty_like(g["x"]) for _ in range(2)]
        lg_d = [torch.empty_like(g["logits"]) for _ in range(2)]
        out_d = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        out_host = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        barrier(world)
        t0.record(s_in)
        for i in range(e2e_steps):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_done[b])           # step i-2 has finished reading these inputs
            with torch.cuda.stream(s_in):
                x_d[b].copy_(x_host, non_blocking=True)
                lg_d[b].copy_(lg_host, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])          # step i-2's output has left this buffer
            run_layer_on(lg_d[b], x_d[b], out_d[b])
            ev_done[b].record(stream)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                out_host[b].copy_(out_d[b], non_blocking=True)
                ev_out[b].record(s_out)
        t1.record(s_out)
        t1.synchronize()
        e2e_s = max_over_ranks(t0.elapsed_time(t1) / 1e3 / e2e_steps, world, dev)
        e2e_mode = "pipelined: input copy, layer and output copy of successive steps overlap"
    else:
        out_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        x_d1 = torch.empty_like(g["x"])
        lg_d1 = torch.empty_like(g["logits"])
        e2e_pairs = []
        with torch.cuda.stream(stream):
            for r in range(e2e_steps + 1):
                flush_l2(r)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                x_d1.copy_(x_host, non_blocking=True)
                lg_d1.copy_(lg_host, non_blocking=True)
                run_layer_on(lg_d1, x_d1, out)
                out_host.copy_(out, non_blocking=True)
                b.record(stream)
                if r > 0:
                    e2e_pairs.append((a, b))
            stream.synchronize()
        e2e_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_pairs) / 1e3 / e2e_steps, world, dev)
        e2e_mode = "sequential: input copy, layer, output copy per step, L2 flushed before each"
    e2e_clk.__exit__(None, None, None)
    st = N.moe_status_read(ws, stream)
    if st != N.MOE_OK:
        raise RuntimeError(f"device status {st} after the end-to-end steps")
    e2e = {"value": world * T / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": x_host.numel() * 2 + lg_host.numel() * 4,
           "d2h_bytes_per_step": T * H * 2, "mode": e2e_mode, "clocks": e2e_clk.summary()}

    peaks = load_peaks()
    up_s = stage_ms["expert_up"] / 1e3
    peak = peaks["bf16_tflops_sustained"]
    # below the ridge (sustained BF16 peak / HBM bandwidth) the up projection is
    # bound by streaming the touched weights, above it by the tensor cores
    ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if alg["up_flops"] / alg["up_bytes"] >= ridge:
        roof = {"bound": "tensor", "achieved": alg["up_flops"] / up_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                "peak_source": f"{peaks['source']} bf16_tflops_sustained"}
    else:
        roof = {"bound": "hbm", "achieved": alg["up_bytes"] / up_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{peaks['source']} hbm_gbs"}
    roof_kernel = up_kernel_name(wl, torch.cuda.get_device_properties(dev).multi_processor_count, quant)
    if fused:
        # the layer step's second and last kernel streams both projections'
        # weights; it has no stage call of its own, so it is timed as the whole
        # step (which adds the fused dispatch: a lower bound on its rate)
        step_s = statistics.median(step_ms) / 1e3
        roof = {"bound": "hbm", "achieved": (alg["up_bytes"] + alg["down_bytes"]) / step_s / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "peak_source": f"{peaks['source']} hbm_gbs",
                "timed": "whole layer step (fused dispatch + fused decode FFN)"}
        roof_kernel = "decode_ffn_kernel (expert up + down + combine)"
    roof["frac"] = roof["achieved"] / roof["peak"]
    achieved = alg["up_flops"] / up_s / 1e12
    # per clock: the up projection against the tensor pipe's own rate at the
    # median SM clock of the timed region (152 SMs x 8192 BF16 flop per cycle:
    # M128 N256 K16 per 128 cycles, measured), so box-to-box clock spread does
    # not hide the kernel's trend
    clocks = clk.summary()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    per_clock = None
    if clocks.get("sm_mhz"):
        rate = sms * 8192 * clocks["sm_mhz"] * 1e6 / 1e12
        per_clock = {"sm_mhz": clocks["sm_mhz"], "tensor_rate_at_clock_tflops": rate,
                     "expert_up_frac_of_rate": achieved / rate,
                     "gemm_frac_of_rate": (alg["up_flops"] + alg["down_flops"]) /
                     ((stage_ms["expert_up"] + stage_ms["expert_down"]) / 1e3) / 1e12 / rate}
    dc_s = (stage_ms["dispatch"] + stage_ms["combine"]) / 1e3
    dc_gbs = (alg["dispatch_bytes"] + alg["combine_bytes"]) / dc_s / 1e9
    gemm_tflops = (alg["up_flops"] + alg["down_flops"]) / ((stage_ms["expert_up"] + stage_ms["expert_down"]) / 1e3) / 1e12

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not quant:   # the oracle sample is the BF16 layer
        import oracle
        oracle.build()
        cpu = cpu_baseline(wl, g, dev, seed=rank)

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": describe(wl), "tokens_per_gpu": T, "global_tokens": world * T,
                       "parallelism": f"dp{world} (independent replicas)",
                       "l2": (f"L2 flushed before every timed step (write of {4 * l2 >> 20} MiB, then a read of "
                              f"another {4 * l2 >> 20} MiB so that the flush's dirty lines are written back outside the step's "
                              f"events)" if flush else
                              f"inputs larger than L2 (x {g['x'].numel() * 2 >> 20} MiB, touched weights "
                              f"{touched >> 20} MiB): no flush"),
                       "expert_weights": WEIGHT_FORMATS[wfmt]},
            "roofline": {"kernel": roof_kernel,
                         **roof,
                         "traffic": ncu_traffic() if wl.name == WORKLOAD and not quant else None},
            "expert_up_tflops": achieved,
            "dispatch_combine_gbs": dc_gbs, "dispatch_combine_hbm_frac": dc_gbs / peaks["hbm_gbs"],
            "gemm_tflops": gemm_tflops, "gemm_frac": gemm_tflops / peak,
            "per_clock": per_clock, "steps_ms": step_stats,
            "stages_ms": stage_ms,
            "stages_path": ("stage calls run the separate kernels (small-row GEMMs, combine); the layer step runs "
                            "the fused decode FFN" if fused else "the layer step's kernels"),
            "algorithmic": alg, "router_front": router_front,
            "e2e": e2e, "gpu_launches": kernels_per_layer * args.steps,
            "clocks": clocks, "cpu_baseline": cpu,
            "kernel_source_sha": kernel_source_sha(),
        }
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp8", "nvfp4"],
                    help="expert weight format (fp8: E4M3 codes with a scale per row, moe_layer_fp8; nvfp4: E2M1 "
                         "codes with E4M3 block scales and a scale per row, moe_layer_nvfp4)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    wl = synth.WORKLOADS[args.workload]
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, wl, world, rank)
    return run_native(args, wl, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
