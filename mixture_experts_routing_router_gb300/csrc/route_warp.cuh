// route_warp.cuh -- one token's softmax top-k routing on one warp (shared by
// route_kernel and the fused small-batch dispatch, so both give the same bits).
//
// ONNX Runtime PR #33963 ("Measured CUDA kernel latency"): the operator routes
// internally by softmax over FP32 router logits.  Selection is keyed on the
// logits (softmax is monotone, and keying on rounded probabilities could create
// false ties) under the order "larger logit first, then lower expert index",
// so -0 == +0 and every other equality goes to the lower index; slot j of the
// result is the j-th expert in that order.  The weights are the softmax over
// the k selected logits, in FP32 with the max subtracted.
//
// The warp finds the k winners without k dependent rounds of argmax: each
// logit becomes an unsigned key with the same order (-0 and +0 the same key),
// the k-th largest key is found by bisection on its bits (a warp-wide count of
// keys at or above each candidate, stopping as soon as exactly k keys remain),
// the keys above it and the lowest-index keys equal to it are taken, and the
// k winners -- gathered into lanes 0..k-1 in expert order -- are ranked among
// themselves and permuted into slot order.
#pragma once

#include "common.cuh"

#include <climits>

namespace moe {

// "a ranks before b" under larger value first, then lower index; bi == INT_MAX
// marks "nothing yet" (the sigmoid routing's k rounds of argmax use it).
__device__ __forceinline__ bool route_better(float av, int ai, float bv, int bi) {
    return bi == INT_MAX || av > bv || (av == bv && ai < bi);
}

// Unsigned key with the order of the float: larger logit -> larger key, and
// -0 and +0 the same key.  -inf maps to 0x007fffff, above the key 0 that marks
// an unused lane slot.
__device__ __forceinline__ uint32_t route_key(float x) {
    if (x == 0.0f) x = 0.0f;
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Lane of the n-th (0-based) set bit of b (n < popc(b)).
__device__ __forceinline__ int nth_set_bit(unsigned b, int n) {
    int s = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
        if (__popc(b & ((1u << (s + step)) - 1u)) <= n) s += step;
    return s;
}

// EPL = logits per lane (E <= 32 * EPL); lane l holds experts l, l+32, ...
// Lane j < k receives the j-th selected expert and its weight.  Returns true
// (on every lane) if any logit of the row is NaN or infinite; such a logit is
// read as -inf.
template <int EPL>
__device__ __forceinline__ bool route_token_softmax(const float* row, int E, int k, int lane, int& sel_out,
                                                    float& w_out) {
    constexpr unsigned kAll = 0xffffffffu;
    float v[EPL];
    uint32_t key[EPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        float x = -INFINITY;
        if (e < E) {
            x = __ldg(row + e);
            if (!isfinite(x)) { bad = true; x = -INFINITY; }
        }
        v[i] = x;
        key[i] = e < E ? route_key(x) : 0u;
    }
    const bool any_bad = __any_sync(kAll, bad);

    // tau: the k-th largest key (or a lower bound with exactly k keys >= tau)
    uint32_t tau = 0;
    unsigned cnt = (unsigned)E;
    for (int bit = 31; bit >= 0 && cnt != (unsigned)k; --bit) {
        const uint32_t cand = tau | (1u << bit);
        unsigned c = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) c += key[i] >= cand;
        c = __reduce_add_sync(kAll, c);
        if (c >= (unsigned)k) { tau = cand; cnt = c; }
    }
    // winners: every key above tau, then keys equal to tau in expert order
    unsigned gt = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) gt += key[i] > tau;
    const int m = k - (int)__reduce_add_sync(kAll, gt);
    unsigned lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
    int eq_before = 0, base = 0;
    uint32_t wk = 0;        // lane j < k: key, value and expert of the j-th winner in expert order
    float wv = 0.f;
    int we = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const unsigned beq = __ballot_sync(kAll, key[i] == tau);
        const bool take = key[i] > tau || (key[i] == tau && eq_before + __popc(beq & lt) < m);
        eq_before += __popc(beq);
        const unsigned b = __ballot_sync(kAll, take);
        const int want = lane - base;
        const bool mine = want >= 0 && want < __popc(b);
        const int src = mine ? nth_set_bit(b, want) : 0;
        const uint32_t sk = __shfl_sync(kAll, key[i], src);
        const float sv = __shfl_sync(kAll, v[i], src);
        if (mine) { wk = sk; wv = sv; we = src + 32 * i; }
        base += __popc(b);
    }
    // rank among the winners (lane order is expert order), then lane r takes
    // the winner of rank r
    int rank = 0;
    for (int s = 0; s < k; ++s) {
        const uint32_t ks = __shfl_sync(kAll, wk, s);
        rank += (ks > wk) || (ks == wk && s < lane);
    }
    unsigned cand_lanes = (k == 32) ? kAll : ((1u << k) - 1u);
#pragma unroll
    for (int b = 0; b < 5; ++b) {
        const unsigned ones = __ballot_sync(kAll, (rank >> b) & 1);
        cand_lanes &= ((lane >> b) & 1) ? ones : ~ones;
    }
    const int from = cand_lanes ? __ffs(cand_lanes) - 1 : 0;
    const float sel_v = __shfl_sync(kAll, wv, from);
    const int sel_i = __shfl_sync(kAll, we, from);
    const float mx = __shfl_sync(kAll, sel_v, 0);
    const float ex = (lane < k) ? expf(sel_v - mx) : 0.f;
    float z = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(kAll, z, off);
    sel_out = sel_i;
    w_out = ex / z;
    return any_bad;
}

}  // namespace moe
