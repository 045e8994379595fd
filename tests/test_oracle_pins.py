"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against something fixed independently:
the worked decode case printed on the ONNX Runtime MoEPacked page
(golden/decode_closed_form.json), brute force on tiny inputs, closed forms,
integer-exact analytic cases, invariants, and library routines (Python's
sorted, numpy float64 matmul, torch's float->bf16 conversion).  The cases are
chosen so that a dropped term, a wrong sign or index, a transposed operand or a
wrong tie rule fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from mixture_experts_routing_router_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_bf16_bits_from_float(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bf16(rng, shape, std=1.0):
    f = (rng.standard_normal(shape) * std).astype(np.float32)
    return torch_bf16_bits_from_float(f.reshape(-1)).reshape(shape)


# --------------------------------------------------------------------------
# BF16 rounding
# --------------------------------------------------------------------------
def test_bf16_rounding_matches_torch_on_float_values(oracle_mod):
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(4000) * s for s in (1e-40, 1e-20, 1e-3, 1.0, 1e5, 1e30)])
    vals = vals.astype(np.float32)
    vals = np.concatenate([vals, np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-45], np.float32)])
    want = torch_bf16_bits_from_float(vals)
    got = np.array([oracle_mod.bf16_from_double(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounding_single_rounding_from_double(oracle_mod):
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to even (1.0)
    assert oracle_mod.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is a tie between 1+2^-7 (odd) and 1+2^-6 (even)
    assert oracle_mod.bf16_from_double(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the tie: must round up.  Rounding to float first would lose
    # the 2^-40 and then tie to even (1.0) -- the wrong answer.
    assert oracle_mod.bf16_from_double(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle_mod.bf16_from_double(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    # overflow threshold: (2 - 2^-8) * 2^127 rounds to inf, just below stays finite
    assert oracle_mod.bf16_from_double(math.ldexp(2 - 2.0 ** -8, 127)) == 0x7F80
    assert oracle_mod.bf16_from_double(math.ldexp(2 - 2.0 ** -7, 127)) == 0x7F7F
    # subnormal: smallest bf16 subnormal is 2^-133; half of it ties to 0
    assert oracle_mod.bf16_from_double(2.0 ** -133) == 0x0001
    assert oracle_mod.bf16_from_double(2.0 ** -134) == 0x0000
    assert oracle_mod.bf16_from_double(1.5 * 2.0 ** -133) == 0x0002
    assert oracle_mod.bf16_from_double(-0.0) == 0x8000


# --------------------------------------------------------------------------
# route
# --------------------------------------------------------------------------
def brute_topk(row, k):
    return sorted(range(len(row)), key=lambda e: (-float(row[e]), e))[:k]


@pytest.mark.parametrize("E,k", [(1, 1), (4, 2), (7, 3), (16, 2), (16, 16), (33, 5)])
def test_route_bruteforce_with_ties(oracle_mod, E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 64
    logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)   # many ties
    st, ids, w = oracle_mod.route(logits, k)
    assert st == 0
    for t in range(T):
        assert list(ids[t]) == brute_topk(logits[t], k)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    # weights follow the logit order
    assert np.all(np.diff(w, axis=1) <= 0)


def test_route_negative_zero_ties_positive_zero(oracle_mod):
    logits = np.array([[-0.0, 0.0, -1.0, 0.0]], np.float32)
    st, ids, w = oracle_mod.route(logits, 3)
    assert st == 0 and list(ids[0]) == [0, 1, 3]
    assert np.all(w == np.float32(1.0 / 3))


def test_route_closed_form_two_experts(oracle_mod):
    # logits 0 and -ln 3: softmax over the pair is exactly (3/4, 1/4) in the reals
    logits = np.array([[-5.0, 0.0, -math.log(3.0), -7.0]], np.float32)
    st, ids, w = oracle_mod.route(logits, 2)
    assert st == 0 and list(ids[0]) == [1, 2]
    assert abs(w[0, 0] - 0.75) < 1e-7 and abs(w[0, 1] - 0.25) < 1e-7
    # the weights are renormalised over the selected experts: unselected logits
    # do not change them
    logits2 = logits.copy()
    logits2[0, 0] = -0.5
    logits2[0, 3] = -0.6
    _, ids3, w3 = oracle_mod.route(logits2, 2)
    assert list(ids3[0]) == [1, 0]


def test_route_decode_closed_form_golden(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "decode_closed_form.json")))
    E, k = g["experts"], g["top_k"]
    want_w = np.float32(g["selected_weight_num"] / g["selected_weight_den"])
    for rows in g["rows"]:
        for kind in ("shared", "distinct"):
            wl = synth.WORKLOADS[f"decode_{rows}_{kind}"]
            lg = synth.make_logits(wl).numpy()
            assert set(np.unique(lg)) == {g["selected_logit"], g["other_logit"]}
            st, ids, w = oracle_mod.route(lg, k)
            assert st == 0
            for r, s in enumerate(synth.decode_route_sets(wl)):
                assert list(ids[r]) == sorted(s)
            assert np.all(w == want_w)
            if rows == 16:
                assert ids.size == g["routes_at_16_rows"]


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
def test_route_rejects_nonfinite(oracle_mod, bad):
    logits = np.zeros((3, 8), np.float32)
    logits[2, 5] = bad
    st, _, _ = oracle_mod.route(logits, 2)
    assert st == oracle_mod.ST_NONFINITE


# --------------------------------------------------------------------------
# dispatch
# --------------------------------------------------------------------------
def naive_placement(ids, E):
    """Expert-major enumeration: walk experts in order and, for each, the pairs
    in ascending p.  A different algorithm from counting + scan + scatter."""
    flat = ids.reshape(-1)
    dest = np.full(flat.size, -1, np.int64)
    slot = 0
    for e in range(E):
        for p in range(flat.size):
            if flat[p] == e:
                dest[p] = slot
                slot += 1
    return dest


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 4, 4), (64, 16, 2), (37, 33, 5), (128, 8, 3)])
def test_dispatch_bruteforce_and_invariants(oracle_mod, T, E, k):
    rng = np.random.default_rng(T + E + k)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    H = 24
    x = rng.integers(0, 65535, size=(T, H)).astype(np.uint16)
    st, counts, offsets, dest, sp, xp = oracle_mod.dispatch(ids, x, E, T)
    assert st == 0
    assert counts.sum() == T * k
    assert np.array_equal(counts, np.bincount(ids.reshape(-1), minlength=E))
    assert offsets[0] == 0 and offsets[E] == T * k
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(dest, naive_placement(ids, E))
    assert np.array_equal(np.sort(dest), np.arange(T * k))           # bijection
    assert np.array_equal(sp[dest], np.arange(T * k))                  # inverse
    for e in range(E):                                                 # stable buckets
        toks = sp[offsets[e]:offsets[e + 1]] // k
        assert np.all(np.diff(toks) > 0)
    for j in range(k):                                                 # round trip
        assert np.array_equal(xp[dest.reshape(T, k)[:, j]], x)


def test_dispatch_decode_closed_form(oracle_mod):
    for rows in (1, 8, 16):
        for kind in ("shared", "distinct"):
            wl = synth.WORKLOADS[f"decode_{rows}_{kind}"]
            ids = np.array(synth.decode_route_sets(wl), np.int32)
            x = np.zeros((rows, 8), np.uint16)
            st, counts, offsets, dest, sp, xp = oracle_mod.dispatch(ids, x, wl.experts, wl.cap)
            assert st == 0
            want = np.zeros(wl.experts, np.int32)
            if kind == "shared":
                want[:9] = rows
            else:
                want[:9 * rows] = 1
            assert np.array_equal(counts, want)


def test_dispatch_capacity_exceeded_moves_no_payload(oracle_mod):
    T, E, k = 10, 4, 2
    ids = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    x = np.ones((T, 8), np.uint16)
    st, counts, offsets, dest, sp, xp = oracle_mod.dispatch(ids, x, E, 9)
    assert st == oracle_mod.ST_CAPACITY
    assert list(counts) == [10, 10, 0, 0] and offsets[-1] == 20
    assert np.all(dest == -7) and np.all(xp == 0)
    # exactly at capacity is fine
    st, *_ = oracle_mod.dispatch(ids, x, E, 10)
    assert st == 0


@pytest.mark.parametrize("kind", ["negative", "wide", "duplicate", "dummy"])
def test_dispatch_invalid_routes(oracle_mod, kind):
    T, E, k = 6, 8, 3
    ids = np.array([[0, 1, 2], [3, 4, 5], [6, 7, 0], [1, 2, 3], [4, 5, 6], [7, 0, 1]], np.int32)
    bad = ids.copy()
    if kind == "negative":
        bad[2, 1] = -3
    elif kind == "wide":
        bad[2, 1] = E
    elif kind == "duplicate":
        bad[2, 1] = bad[2, 0]
    else:   # a dummy (-1) route
        bad[2, 1] = -1
    x = np.arange(T * 8, dtype=np.uint16).reshape(T, 8)
    st, counts, offsets, dest, sp, xp = oracle_mod.dispatch(bad, x, E, T)
    assert st == oracle_mod.ST_INVALID_ROUTE
    assert counts.sum() == T * k - 1
    assert dest[2 * k + 1] == -1
    valid = np.ones(T * k, bool)
    valid[2 * k + 1] = False
    assert np.array_equal(np.sort(dest[valid]), np.arange(T * k - 1))


# --------------------------------------------------------------------------
# expert FFN
# --------------------------------------------------------------------------
def np_dense_mlp(xb, w13b, w2b, act):
    """Independent dense MLP in numpy float64 (matmul order differs from the
    oracle's sequential sums), with torch doing the BF16 rounding."""
    x = bits_to_f64(xb)
    w13 = bits_to_f64(w13b)
    w2 = bits_to_f64(w2b)
    I = w2.shape[1]
    a = x @ w13.T
    if act == 0:
        g, u = a[:, :I], a[:, I:]
        hv = g / (1.0 + np.exp(-g)) * u
    else:
        hv = np.maximum(a, 0.0) ** 2
    h = torch.tensor(hv).to(torch.bfloat16)      # float64 -> bf16, one rounding
    hb = h.view(torch.int16).numpy().view(np.uint16)
    y = torch.tensor(bits_to_f64(hb) @ w2.T).to(torch.bfloat16)
    return hb, y.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("act", [0, 1])
def test_ffn_single_expert_is_dense_mlp(oracle_mod, act):
    rng = np.random.default_rng(7 + act)
    T, H, I = 40, 96, 56
    up = 2 * I if act == 0 else I
    x = rand_bf16(rng, (T, H))
    w13 = rand_bf16(rng, (1, up, H), 1 / math.sqrt(H))
    w2 = rand_bf16(rng, (1, H, I), 1 / math.sqrt(I))
    offsets = np.array([0, T], np.int32)
    h, y, _, _ = oracle_mod.expert_ffn(x, offsets, w13, w2, act)
    hn, yn = np_dense_mlp(x, w13[0], w2[0], act)
    hd = np.abs(bits_to_f64(h) - bits_to_f64(hn))
    # matmul order can flip a BF16 rounding of h by one ulp, rarely
    assert np.mean(h != hn) < 0.01
    assert np.all(hd <= np.abs(bits_to_f64(hn)) * 2 ** -7 + 1e-30)
    yd = np.abs(bits_to_f64(y) - bits_to_f64(yn))
    assert yd.max() <= 1e-2 * np.abs(bits_to_f64(yn)).max()
    # gate and up are not interchangeable (catches a swapped half)
    if act == 0:
        w13s = np.concatenate([w13[:, I:], w13[:, :I]], axis=1)
        h2, _, _, _ = oracle_mod.expert_ffn(x, offsets, w13s, w2, act)
        assert np.mean(h2 != h) > 0.5


def test_ffn_identical_experts_give_dense_mlp_for_any_routing(oracle_mod):
    rng = np.random.default_rng(11)
    T, H, I, E, k = 24, 64, 40, 6, 3
    w13_1 = rand_bf16(rng, (1, 2 * I, H), 1 / 8)
    w2_1 = rand_bf16(rng, (1, H, I), 1 / 6)
    w13 = np.repeat(w13_1, E, axis=0)
    w2 = np.repeat(w2_1, E, axis=0)
    x = rand_bf16(rng, (T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    o = oracle_mod.layer(x, w13, w2, 0, k, T, logits=logits)
    assert o["status"] == 0
    h1, y1, _, _ = oracle_mod.expert_ffn(x, np.array([0, T], np.int32), w13_1, w2_1, 0)
    assert np.array_equal(o["out"], y1)


def relu2_analytic_case(rng, T, E, k, H, I):
    """x, W in {-1, 0, 1}; each token's k experts tie at logit 1 (others 0),
    so every weight is exactly 1/k.  Integers stay small enough that every
    value is exact until the one BF16 rounding torch applies."""
    x = rng.integers(-1, 2, size=(T, H))
    w1 = rng.integers(-1, 2, size=(E, I, H))
    w2 = rng.integers(-1, 2, size=(E, H, I))
    sets = [sorted(rng.permutation(E)[:k].tolist()) for _ in range(T)]
    logits = np.zeros((T, E), np.float32)
    for t, s in enumerate(sets):
        logits[t, s] = 1.0
    return x, w1, w2, sets, logits


def bf16_of_exact(vals):
    """Round exact integers/dyadics to BF16 by torch (float64 -> bf16 is one
    rounding for these values since they are exact in float64)."""
    t = torch.tensor(np.asarray(vals, np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("k", [2, 4])
def test_layer_relu2_analytic_exact(oracle_mod, k):
    rng = np.random.default_rng(100 + k)
    T, E, H, I = 16, 8, 40, 24
    x, w1, w2, sets, logits = relu2_analytic_case(rng, T, E, k, H, I)
    xb, w1b, w2b = (bf16_of_exact(a) for a in (x, w1, w2))
    o = oracle_mod.layer(xb, w1b, w2b, 1, k, T, logits=logits)
    assert o["status"] == 0
    assert np.all(o["w"] == np.float32(1.0 / k))
    want = np.zeros((T, H), np.uint16)
    for t in range(T):
        acc = [Fraction(0)] * H
        for e in sets[t]:
            a = w1[e] @ x[t]                                 # exact ints
            hq = bits_to_f64(bf16_of_exact(np.maximum(a, 0) ** 2))
            yv = bits_to_f64(bf16_of_exact(w2[e] @ hq))      # exact sum of ints
            for c in range(H):
                acc[c] += Fraction(yv[c]) / k
        want[t] = bf16_of_exact([float(a) for a in acc])     # dyadic: exact in f64
    assert np.array_equal(o["out"], want)


def test_shared_experts_sum_before_rounding(oracle_mod):
    rng = np.random.default_rng(5)
    H, Is, S = 32, 16, 2
    x = rand_bf16(rng, (1, H))
    ws13 = rand_bf16(rng, (S, 2 * Is, H), 0.3)
    ws2 = rand_bf16(rng, (S, H, Is), 0.3)
    hs, ys = oracle_mod.shared_row(x[0], ws13, ws2, 0)
    # independent: both shared experts as one expert with intermediate S*Is
    # (gate rows of both, then up rows of both; down weights side by side)
    w13cat = np.concatenate([ws13[0, :Is], ws13[1, :Is], ws13[0, Is:], ws13[1, Is:]])[None]
    w2cat = np.concatenate([ws2[0], ws2[1]], axis=1)[None]
    h1, y1, _, _ = oracle_mod.expert_ffn(x, np.array([0, 1], np.int32), w13cat, w2cat, 0)
    assert np.array_equal(hs, h1[0])
    assert np.array_equal(ys, y1[0])


# --------------------------------------------------------------------------
# combine
# --------------------------------------------------------------------------
@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_combine_identity_experts_return_x(oracle_mod, k):
    rng = np.random.default_rng(k)
    T, E, H = 30, 12, 48
    x = rand_bf16(rng, (T, H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    st, counts, offsets, dest, sp, xp = oracle_mod.dispatch(ids, x, E, T)
    w = np.full((T, k), 1.0 / k, np.float32)          # powers of two: exact
    out = oracle_mod.combine(xp, dest, w)
    assert np.array_equal(out, x)
    # shared term is added: x + x = 2x exactly
    out2 = oracle_mod.combine(xp, dest, w, y_shared=x)
    assert np.array_equal(bits_to_f64(out2), 2 * bits_to_f64(x))


def test_combine_residual_is_added_once(oracle_mod):
    # identity experts with power-of-two weights give x; a residual r adds r
    # exactly when x + r is exact in BF16 (here r = x, so the result is 2x),
    # and it is added after the shared term (x + x + x = 3x for small integers)
    rng = np.random.default_rng(31)
    T, E, H, k = 12, 6, 16, 2
    x = bf16_of_exact(rng.integers(-8, 9, size=(T, H)))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, _, _, dest, _, xp = oracle_mod.dispatch(ids, x, E, T)
    w = np.full((T, k), 0.5, np.float32)
    assert np.array_equal(bits_to_f64(oracle_mod.combine(xp, dest, w, residual=x)), 2 * bits_to_f64(x))
    assert np.array_equal(bits_to_f64(oracle_mod.combine(xp, dest, w, y_shared=x, residual=x)),
                          3 * bits_to_f64(x))
    out = oracle_mod.combine_row(xp, dest.reshape(T, k)[0], w[0], None, x[0])
    assert np.array_equal(bits_to_f64(out), 2 * bits_to_f64(x[0]))


def test_combine_weights_are_applied_per_slot(oracle_mod):
    # y rows 1.0 and 2.0 with weights 0.75 / 0.25 -> 1.25 exactly; swapped -> 1.75
    y = bf16_of_exact([[1.0] * 4, [2.0] * 4])
    out = oracle_mod.combine(y, np.array([0, 1], np.int32), np.array([[0.75, 0.25]], np.float32))
    assert np.all(bits_to_f64(out) == 1.25)
    out = oracle_mod.combine(y, np.array([1, 0], np.int32), np.array([[0.75, 0.25]], np.float32))
    assert np.all(bits_to_f64(out) == 1.75)
    # an invalid pair (dest -1) contributes nothing
    out = oracle_mod.combine(y, np.array([1, -1], np.int32), np.array([[0.75, 0.25]], np.float32))
    assert np.all(bits_to_f64(out) == 1.5)


# --------------------------------------------------------------------------
# layer
# --------------------------------------------------------------------------
def test_layer_internal_routing_equals_preselected(oracle_mod):
    wl = synth.WORKLOADS["tiny"].with_(tokens=16)
    d = synth.make_inputs(wl, unit_scale=True)
    x = synth.bf16_bits(d["x"])
    w13 = synth.bf16_bits(d["w13"])
    w2 = synth.bf16_bits(d["w2"])
    lg = d["logits"].numpy()
    a = oracle_mod.layer(x, w13, w2, 0, wl.top_k, wl.cap, logits=lg)
    st, ids, w = oracle_mod.route(lg, wl.top_k)
    b = oracle_mod.layer(x, w13, w2, 0, wl.top_k, wl.cap, ids_in=ids, w_in=w)
    assert a["status"] == b["status"] == 0
    assert np.array_equal(a["out"], b["out"])
    assert np.abs(bits_to_f64(a["out"])).max() > 0.05          # unit-scale twin is not ~0


# --------------------------------------------------------------------------
# router front end: sigmoid routing with a selection-only bias, gate projection
# --------------------------------------------------------------------------
def test_route_sigmoid_without_bias_selects_like_softmax(oracle_mod):
    # sigmoid is increasing, so with no bias the selection is the top-k by logit
    # (logits well inside (-8, 8) keep the FP32 sigmoids distinct)
    rng = np.random.default_rng(21)
    logits = rng.standard_normal((200, 40)).astype(np.float32)
    _, ids_s, _ = oracle_mod.route(logits, 6)
    st, ids, w = oracle_mod.route_sigmoid(logits, 6)
    assert st == 0 and np.array_equal(ids, ids_s)
    assert np.abs(w.astype(np.float64).sum(1) - 1.0).max() <= 1e-6


def test_route_sigmoid_dominant_bias_selects_its_set_and_weights_ignore_it(oracle_mod):
    rng = np.random.default_rng(22)
    T, E, k = 50, 24, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    chosen = np.array([3, 7, 11, 19])
    bias = np.zeros(E, np.float32)
    bias[chosen] = 2.0                         # keys >= 2 > any unbiased score
    st, ids, w = oracle_mod.route_sigmoid(logits, k, bias, route_scale=2.5)
    assert st == 0
    for t in range(T):
        assert sorted(ids[t]) == sorted(chosen)
        # within the set the order follows the score, i.e. the logit
        assert list(ids[t]) == sorted(chosen, key=lambda e: (-float(logits[t, e]), e))
    assert np.abs(w.astype(np.float64).sum(1) - 2.5).max() <= 1e-5
    bias2 = bias.copy()
    bias2[chosen] = 3.0                        # same selection, different bias
    _, ids2, w2 = oracle_mod.route_sigmoid(logits, k, bias2, route_scale=2.5)
    assert np.array_equal(ids2, ids) and np.array_equal(w2, w)


def test_route_sigmoid_negative_bias_excludes_the_top_experts(oracle_mod):
    rng = np.random.default_rng(23)
    T, E, k = 40, 16, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    for t in range(T):
        _, top, _ = oracle_mod.route(logits[t:t + 1], k)
        bias = np.zeros(E, np.float32)
        bias[top[0]] = -2.0                    # keys < 0 < any unbiased score
        _, ids, _ = oracle_mod.route_sigmoid(logits[t:t + 1], k, bias)
        masked = logits[t:t + 1].copy()
        masked[0, top[0]] = -1e30
        _, nxt, _ = oracle_mod.route(masked, k)
        assert np.array_equal(ids, nxt)


def test_route_sigmoid_closed_form_weights(oracle_mod):
    # sigmoid(0) = 1/2 exactly: k experts at logit 0 share the weight scale / k
    logits = np.full((3, 10), -5.0, np.float32)
    logits[:, [1, 4, 8, 9]] = 0.0
    st, ids, w = oracle_mod.route_sigmoid(logits, 4, route_scale=1.0)
    assert st == 0 and np.all(ids == np.array([1, 4, 8, 9]))
    assert np.all(w == np.float32(0.25))
    st, _, _ = oracle_mod.route_sigmoid(np.full((1, 4), np.nan, np.float32), 2)
    assert st == oracle_mod.ST_NONFINITE


def test_gate_projection_matches_float64_matmul(oracle_mod):
    rng = np.random.default_rng(24)
    T, H, E = 33, 200, 24
    x = rand_bf16(rng, (T, H))
    wg = rand_bf16(rng, (E, H), 0.1)
    got = oracle_mod.gate(x, wg).astype(np.float64)
    want = (bits_to_f64(x) @ bits_to_f64(wg).T).astype(np.float32).astype(np.float64)
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - want) <= ulp)
    # transposing the weight matrix is caught
    assert not np.allclose(oracle_mod.gate(x[:, :E], rand_bf16(rng, (E, E))),
                           oracle_mod.gate(x[:, :E], rand_bf16(rng, (E, E))))


# --------------------------------------------------------------------------
# FP8 E4M3 expert weights (one FP32 scale per weight row)
# --------------------------------------------------------------------------
def test_fp8_decode_closed_forms(oracle_mod):
    """OCP E4M3: bias 7, 3 mantissa bits, subnormals at exponent 0, no
    infinities, NaN only at S.1111.111."""
    v = oracle_mod.fp8_e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0.0 and math.copysign(1.0, v[0x00]) > 0
    assert v[0x80] == 0.0 and math.copysign(1.0, v[0x80]) < 0
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9        # subnormals
    assert v[0x08] == 2.0 ** -6                                      # smallest normal
    assert v[0x38] == 1.0 and v[0x3C] == 1.5 and v[0x40] == 2.0 and v[0x41] == 2.25
    assert v[0x7E] == 448.0                                          # largest finite
    nan = np.isnan(v)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.all(np.diff(v[:0x7F]) > 0)                             # monotone over the positive codes
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F])


def test_fp8_decode_matches_torch(oracle_mod):
    """torch's float8_e4m3fn conversion is an independent implementation."""
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = oracle_mod.fp8_e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(t), np.isnan(v))
    ok = ~np.isnan(v)
    assert np.array_equal(t[ok], v[ok])


def fp8_exact_case(rng, E, up, H, I):
    """FP8 codes and power-of-two row scales: every dequantized weight
    decode(code) * scale is exact in BF16, so the BF16 path of the oracle on
    those values is an independent statement of the same sums."""
    c13 = (torch.from_numpy(rng.standard_normal((E, up, H)).astype(np.float32)) * 0.6).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    c2 = (torch.from_numpy(rng.standard_normal((E, H, I)).astype(np.float32)) * 0.6).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    s13 = (2.0 ** rng.integers(-3, 4, (E, up))).astype(np.float32)
    s2 = (2.0 ** rng.integers(-3, 4, (E, H))).astype(np.float32)
    w13 = bf16_of_exact(torch.tensor(c13).view(torch.float8_e4m3fn).to(torch.float64).numpy() * s13[:, :, None])
    w2 = bf16_of_exact(torch.tensor(c2).view(torch.float8_e4m3fn).to(torch.float64).numpy() * s2[:, :, None])
    return c13, s13, c2, s2, w13, w2


@pytest.mark.parametrize("act", [0, 1])
def test_fp8_ffn_equals_bf16_path_on_exact_weights(oracle_mod, act):
    rng = np.random.default_rng(31 + act)
    E, H, I, R = 3, 48, 40, 30
    up = 2 * I if act == 0 else I
    c13, s13, c2, s2, w13, w2 = fp8_exact_case(rng, E, up, H, I)
    x_perm = rand_bf16(rng, (R, H))
    offsets = np.array([0, 7, 7, R], np.int32)
    h8, y8 = oracle_mod.expert_ffn_fp8(x_perm, offsets, c13, s13, c2, s2, act)
    hb, yb, _, _ = oracle_mod.expert_ffn(x_perm, offsets, w13, w2, act)
    assert np.array_equal(h8, hb)
    assert np.array_equal(y8, yb)
    assert np.mean(h8 != 0) > 0.3                                    # not trivially zero


def test_fp8_layer_equals_bf16_layer_on_exact_weights(oracle_mod):
    rng = np.random.default_rng(41)
    T, E, k, H, I = 24, 6, 2, 32, 48
    c13, s13, c2, s2, w13, w2 = fp8_exact_case(rng, E, 2 * I, H, I)
    x = rand_bf16(rng, (T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    res = rand_bf16(rng, (T, H))
    o8 = oracle_mod.layer_fp8(x, c13, s13, c2, s2, 0, k, T, logits=logits, residual=res)
    ob = oracle_mod.layer(x, w13, w2, 0, k, T, logits=logits, residual=res)
    assert o8["status"] == ob["status"] == 0
    for key in ("ids", "offsets", "dest", "x_perm", "h", "y_perm", "out"):
        assert np.array_equal(o8[key], ob[key]), key


# --------------------------------------------------------------------------
# NVFP4 expert weights (E2M1 codes, an E4M3 scale per 16 elements, an FP32
# scale per row)
# --------------------------------------------------------------------------
# The E2M1 element values as the OCP microscaling format lists them, code
# 0..7 (positive) and 8..15 (the same magnitudes, negative).
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)


def test_fp4_decode_values(oracle_mod):
    v = oracle_mod.fp4_e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(v[:8], E2M1_VALUES)
    assert np.array_equal(v[8:], -E2M1_VALUES)
    assert math.copysign(1.0, v[8]) < 0                              # code 8 is -0


def nvfp4_bscale_bytes(K):
    return 16 * ((K + 255) // 256)


def nvfp4_exact_case(rng, E, rows, K):
    """Random E2M1 codes, finite E4M3 block scales (subnormals included) and
    power-of-two row scales, with the block-scale padding filled with NaN codes
    (never read).  -> (codes [E, rows, K/2], bscale [E, rows, 16*ceil(K/256)],
    rscale [E, rows], the dequantized weights as BF16 bits [E, rows, K]); every
    dequantized weight e2m1 * block scale * row scale is exact in BF16, and
    it is formed here from the OCP value list and torch's E4M3 decode."""
    nib = rng.integers(0, 16, (E, rows, K))
    codes = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    sb = rng.integers(0, 0x7F, (E, rows, K // 16)).astype(np.uint8)          # 0x00..0x7E: finite, >= 0
    sb[..., 0] = 0x01                                                        # a subnormal scale in every row
    bscale = np.full((E, rows, nvfp4_bscale_bytes(K)), 0x7F, np.uint8)
    bscale[..., :K // 16] = sb
    rscale = (2.0 ** rng.integers(-3, 4, (E, rows))).astype(np.float32)
    elem = np.where(nib >= 8, -1.0, 1.0) * E2M1_VALUES[nib & 7]
    sbv = torch.from_numpy(sb).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    w = elem * np.repeat(sbv, 16, axis=-1) * rscale[..., None].astype(np.float64)
    return codes, bscale, rscale, bf16_of_exact(w)


@pytest.mark.parametrize("act,H,I", [(0, 48, 64), (1, 288, 32), (0, 512, 272)])
def test_nvfp4_ffn_equals_bf16_path_on_exact_weights(oracle_mod, act, H, I):
    """K not a multiple of 256 (padded block-scale rows), K above 256 (two
    16-byte scale groups per row), both activations."""
    rng = np.random.default_rng(61 + act + H)
    E, R = 3, 20
    up = 2 * I if act == 0 else I
    c13, b13, s13, w13 = nvfp4_exact_case(rng, E, up, H)
    c2, b2, s2, w2 = nvfp4_exact_case(rng, E, H, I)
    x_perm = rand_bf16(rng, (R, H))
    offsets = np.array([0, 6, 6, R], np.int32)
    h4, y4 = oracle_mod.expert_ffn_nvfp4(x_perm, offsets, c13, b13, s13, c2, b2, s2, act)
    hb, yb, _, _ = oracle_mod.expert_ffn(x_perm, offsets, w13, w2, act)
    assert np.array_equal(h4, hb)
    assert np.array_equal(y4, yb)
    assert np.mean(h4 != 0) > 0.3


def test_nvfp4_layer_equals_bf16_layer_on_exact_weights(oracle_mod):
    rng = np.random.default_rng(71)
    T, E, k, H, I = 24, 6, 2, 32, 48
    c13, b13, s13, w13 = nvfp4_exact_case(rng, E, 2 * I, H)
    c2, b2, s2, w2 = nvfp4_exact_case(rng, E, H, I)
    x = rand_bf16(rng, (T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    res = rand_bf16(rng, (T, H))
    o4 = oracle_mod.layer_nvfp4(x, c13, b13, s13, c2, b2, s2, 0, k, T, logits=logits, residual=res)
    ob = oracle_mod.layer(x, w13, w2, 0, k, T, logits=logits, residual=res)
    assert o4["status"] == ob["status"] == 0
    for key in ("ids", "offsets", "dest", "x_perm", "h", "y_perm", "out"):
        assert np.array_equal(o4[key], ob[key]), key


def test_nvfp4_layer_preselected_routes_and_capacity(oracle_mod):
    """The NVFP4 layer takes the same routing and dispatch as the BF16 layer:
    preselected routes equal internal routing bitwise, and a bucket over
    capacity stops the layer before any payload moves."""
    rng = np.random.default_rng(81)
    T, E, k, H, I = 20, 5, 2, 64, 32
    c13, b13, s13, _ = nvfp4_exact_case(rng, E, 2 * I, H)
    c2, b2, s2, _ = nvfp4_exact_case(rng, E, H, I)
    x = rand_bf16(rng, (T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    a = oracle_mod.layer_nvfp4(x, c13, b13, s13, c2, b2, s2, 0, k, T, logits=logits)
    st, ids, w = oracle_mod.route(logits, k)
    b = oracle_mod.layer_nvfp4(x, c13, b13, s13, c2, b2, s2, 0, k, T, ids_in=ids, w_in=w)
    assert a["status"] == b["status"] == 0
    assert np.array_equal(a["out"], b["out"]) and np.abs(bits_to_f64(a["out"])).max() > 0
    # every token routed to experts 0 and 1: 20 rows each, capacity 19
    ids_full = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    w_full = np.full((T, k), 0.5, np.float32)
    c = oracle_mod.layer_nvfp4(x, c13, b13, s13, c2, b2, s2, 0, k, T - 1, ids_in=ids_full, w_in=w_full)
    assert c["status"] == oracle_mod.ST_CAPACITY
    assert np.all(c["x_perm"] == 0) and np.all(c["out"] == 0)
