// route.cu -- K1, softmax top-k routing: one warp per token.
//
// ONNX Runtime PR #33963 ("Measured CUDA kernel latency"): the operator routes
// internally by softmax over FP32 router logits; the selected weights of the
// +16/-16 case are 1/9.  DeepSeek fleet REPORT.md (optimisation step 1): top-k
// as k rounds of a wave-wide max; here a 32-lane warp.
//
// Selection is keyed on the logits themselves (softmax is monotone, and keying
// on rounded probabilities could create false ties): k rounds, each a warp-wide
// argmax under the order "larger logit first, then lower expert index", so
// -0 == +0 and every other equality goes to the lower index.  The weights are
// the softmax over the k selected logits (the full softmax renormalised over
// the selection), computed in FP32 with the max subtracted.
#include "common.cuh"
#include "route_warp.cuh"

#include <climits>

namespace moe {
namespace {

// k rounds of register argmax per token: see route_warp.cuh.
template <int EPL>
__global__ void __launch_bounds__(256)
route_kernel(int T, int E, int k, const float* __restrict__ logits, int32_t* __restrict__ ids,
             float* __restrict__ w, WsHeader* hdr) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gwarp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    for (int t = gwarp; t < T; t += nwarps) {
        int sel_i;
        float sel_w;
        if (route_token_softmax<EPL>(logits + (size_t)t * E, E, k, lane, sel_i, sel_w) && lane == 0)
            raise_status(hdr, MOE_ERR_NONFINITE);
        if (lane < k) {
            ids[(size_t)t * k + lane] = sel_i;
            w[(size_t)t * k + lane] = sel_w;
        }
    }
}

// Sigmoid routing with a selection-only correction bias (ONNX Runtime PR
// #33963, Description: fused sigmoid routing whose mixture weights come from
// the unbiased scores).  Score s = sigmoid(l), taken in double and rounded
// once to FP32 (so the selection keys are reproducible bit for bit); key =
// s + bias in FP32; the k largest keys win, ties to the lower index; the
// weights are route_scale * s / (sum of the selected s), in FP32.
template <int EPL>
__global__ void __launch_bounds__(256)
route_sigmoid_kernel(int T, int E, int k, const float* __restrict__ logits, const float* __restrict__ bias,
                     float route_scale, int32_t* __restrict__ ids, float* __restrict__ w, WsHeader* hdr) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gwarp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    for (int t = gwarp; t < T; t += nwarps) {
        const float* row = logits + (size_t)t * E;
        float key[EPL], sc[EPL];
        uint32_t taken = 0;
        bool bad = false;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            float kv = -INFINITY, sv = 0.f;
            if (e < E) {
                const float x = __ldg(row + e);
                if (!isfinite(x)) {
                    bad = true;
                } else {
                    sv = (float)(1.0 / (1.0 + exp(-(double)x)));
                    kv = sv + (bias ? __ldg(bias + e) : 0.0f);
                }
            } else {
                taken |= 1u << i;
            }
            key[i] = kv;
            sc[i] = sv;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(hdr, MOE_ERR_NONFINITE);

        float sel_s = 0.f;
        int sel_i = 0;
        for (int j = 0; j < k; ++j) {
            float bv = 0.f, bs = 0.f;
            int bi = INT_MAX;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (!((taken >> i) & 1u) && route_better(key[i], lane + 32 * i, bv, bi)) {
                    bv = key[i]; bs = sc[i]; bi = lane + 32 * i;
                }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (oi != INT_MAX && route_better(ov, oi, bv, bi)) { bv = ov; bs = os; bi = oi; }
            }
            if (lane == (bi & 31)) taken |= 1u << (bi >> 5);
            if (lane == j) { sel_s = bs; sel_i = bi; }
        }
        float z = (lane < k) ? sel_s : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (lane < k) {
            ids[(size_t)t * k + lane] = sel_i;
            w[(size_t)t * k + lane] = route_scale * sel_s / z;
        }
    }
}

template <int EPL>
cudaError_t launch_sigmoid_epl(const moe_shape& s, const float* logits, const float* bias, float scale, int32_t* ids,
                               float* w, WsHeader* hdr, cudaStream_t st) {
    const int warps_per_block = 8;
    long long blocks = ((long long)s.tokens + warps_per_block - 1) / warps_per_block;
    const long long cap = (long long)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return launch_kernel(route_sigmoid_kernel<EPL>, dim3((unsigned)blocks), dim3(32 * warps_per_block), 0, st, 1,
                         kUsePdl, s.tokens, s.experts, s.top_k, logits, bias, scale, ids, w, hdr);
}

template <int EPL>
cudaError_t launch_epl(const moe_shape& s, const float* logits, int32_t* ids, float* w, WsHeader* hdr,
                       cudaStream_t st) {
    const int warps_per_block = 8;
    long long blocks = ((long long)s.tokens + warps_per_block - 1) / warps_per_block;
    const long long cap = (long long)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return launch_kernel(route_kernel<EPL>, dim3((unsigned)blocks), dim3(32 * warps_per_block), 0, st, 1,
                         kUsePdl, s.tokens, s.experts, s.top_k, logits, ids, w, hdr);
}

}  // namespace

cudaError_t launch_route(const moe_shape& s, const float* logits, int32_t* ids, float* w, WsHeader* hdr,
                         cudaStream_t st) {
    const int E = s.experts;
    if (E <= 32) return launch_epl<1>(s, logits, ids, w, hdr, st);
    if (E <= 64) return launch_epl<2>(s, logits, ids, w, hdr, st);
    if (E <= 128) return launch_epl<4>(s, logits, ids, w, hdr, st);
    if (E <= 256) return launch_epl<8>(s, logits, ids, w, hdr, st);
    if (E <= 512) return launch_epl<16>(s, logits, ids, w, hdr, st);
    return launch_epl<32>(s, logits, ids, w, hdr, st);
}

cudaError_t launch_route_sigmoid(const moe_shape& s, const float* logits, const float* bias, float scale,
                                 int32_t* ids, float* w, WsHeader* hdr, cudaStream_t st) {
    const int E = s.experts;
    if (E <= 32) return launch_sigmoid_epl<1>(s, logits, bias, scale, ids, w, hdr, st);
    if (E <= 64) return launch_sigmoid_epl<2>(s, logits, bias, scale, ids, w, hdr, st);
    if (E <= 128) return launch_sigmoid_epl<4>(s, logits, bias, scale, ids, w, hdr, st);
    if (E <= 256) return launch_sigmoid_epl<8>(s, logits, bias, scale, ids, w, hdr, st);
    if (E <= 512) return launch_sigmoid_epl<16>(s, logits, bias, scale, ids, w, hdr, st);
    return launch_sigmoid_epl<32>(s, logits, bias, scale, ids, w, hdr, st);
}

}  // namespace moe
