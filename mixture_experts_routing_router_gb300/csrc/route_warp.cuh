// route_warp.cuh -- one token's softmax top-k routing on one warp (shared by
// route_kernel and the fused small-batch dispatch, so both give the same bits).
//
// ONNX Runtime PR #33963 ("Measured CUDA kernel latency"): the operator routes
// internally by softmax over FP32 router logits.  DeepSeek fleet REPORT.md
// (optimisation step 1): top-k as k rounds of a wave-wide max; here a 32-lane
// warp.  Selection is keyed on the logits (softmax is monotone, and keying on
// rounded probabilities could create false ties): each round is a warp-wide
// argmax under "larger logit first, then lower expert index", so -0 == +0 and
// every other equality goes to the lower index.  The weights are the softmax
// over the k selected logits, in FP32 with the max subtracted.
#pragma once

#include "common.cuh"

#include <climits>

namespace moe {

__device__ __forceinline__ bool route_better(float av, int ai, float bv, int bi) {
    // a ranks before b; bi == INT_MAX marks "nothing yet"
    return bi == INT_MAX || av > bv || (av == bv && ai < bi);
}

// EPL = logits per lane (E <= 32 * EPL); lane l holds experts l, l+32, ...
// Lane j < k receives the j-th selected expert and its weight.  Returns true
// (on every lane) if any logit of the row is NaN or infinite.
template <int EPL>
__device__ __forceinline__ bool route_token_softmax(const float* row, int E, int k, int lane, int& sel_out,
                                                    float& w_out) {
    float v[EPL];
    uint32_t taken = 0;   // bit i: slot i already selected or past E
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        float x = -INFINITY;
        if (e < E) {
            x = __ldg(row + e);
            if (!isfinite(x)) { bad = true; x = -INFINITY; }
        } else {
            taken |= 1u << i;
        }
        v[i] = x;
    }
    const bool any_bad = __any_sync(0xffffffffu, bad);
    float sel_v = 0.f, m = 0.f;
    int sel_i = 0;
    for (int j = 0; j < k; ++j) {
        float bv = 0.f;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (!((taken >> i) & 1u) && route_better(v[i], lane + 32 * i, bv, bi)) { bv = v[i]; bi = lane + 32 * i; }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (oi != INT_MAX && route_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        // k <= E, so a winner always exists: every lane holds the same (bv, bi)
        if (lane == (bi & 31)) taken |= 1u << (bi >> 5);
        if (j == 0) m = bv;
        if (lane == j) { sel_v = bv; sel_i = bi; }
    }
    const float ex = (lane < k) ? expf(sel_v - m) : 0.f;
    float z = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    sel_out = sel_i;
    w_out = ex / z;
    return any_bad;
}

}  // namespace moe
