// combine.cu -- K6, the weighted unpermute-combine back to token order.
//
// DeepSeek fleet REPORT.md (MOE_COMBINE_RESIDUAL row: the combine with the
// block's residual add fused) and ONNX Runtime PR #33963 ("FP32 final
// routing/reduction"):
//   out[t] = bf16( sum_{j<k} w[t,j] * y_perm[dest[t*k+j]] + y_shared[t] + residual[t] )
// accumulated in FP32, j = 0..k-1 in order, then the shared-expert term, then
// the residual (both optional).
// One block per token row; 16-byte vectors (8 BF16) per thread; the k source
// rows of a chunk are loaded together before they are summed in order.
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void acc_bf16x8(float (&a)[8], const uint4& v, float w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), a[2 * i]);
        a[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xffff0000u), a[2 * i + 1]);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(256)
combine_kernel(int T, int HV, int k, const uint4* __restrict__ y_perm, const int32_t* __restrict__ dest,
               const float* __restrict__ w, const uint4* __restrict__ y_shared, const uint4* residual,
               uint4* out,     // out may alias residual: each 16-byte group is read, then written, by one thread
               WsHeader* gate) {
    __shared__ int dsh[32];
    __shared__ float wsh[32];
    const long long R = (long long)T * k;
    const int tid = threadIdx.x, nt = blockDim.x;
    auto load_route = [&](int t) {
        if (tid < k) {
            const long long p = (long long)t * k + tid;
            const int d = __ldcg(dest + p);
            dsh[tid] = (d >= 0 && d < R) ? d : -1;
            wsh[tid] = __ldcg(w + p);
        }
    };
    // Inside moe_layer (gate set) the capacity verdict, dest and w come from
    // the layer's dispatch, which completed before this kernel could start: the
    // GEMMs between them trigger their dependents only after their own
    // programmatic waits.  So they are read (through L2) before this kernel's
    // wait, off the path behind the down projection.  A standalone call reads
    // them after the wait: its predecessor may be the one that writes them.
    bool over = false;
    if (gate) {
        over = __ldcg(&gate->cap_exceeded) != 0;
        if (blockIdx.x < T) load_route(blockIdx.x);
    }
    pdl_wait();
    pdl_trigger();
    if (gate) {
        // the layer's last kernel: the next layer call's fused dispatch will
        // publish its bucket bounds afresh
        if (blockIdx.x == 0 && threadIdx.x == 0) gate->route_ready = 0u;
        if (over) return;                       // over capacity in this layer call: out stays untouched
    }
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (!gate || t != (int)blockIdx.x) load_route(t);
        __syncthreads();
        for (int c = tid; c < HV; c += nt) {
            float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            // the residual and shared rows go out with the first batch of routed rows
            uint4 vs = make_uint4(0u, 0u, 0u, 0u), vr = make_uint4(0u, 0u, 0u, 0u);
            if (y_shared) vs = __ldcs(y_shared + (size_t)t * HV + c);
            if (residual) vr = residual[(size_t)t * HV + c];
            for (int j0 = 0; j0 < k; j0 += 8) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    if (j < k && dsh[j] >= 0) v[u] = __ldcs(y_perm + (size_t)dsh[j] * HV + c);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    if (j < k && dsh[j] >= 0) acc_bf16x8(a, v[u], wsh[j]);
                }
            }
            if (y_shared) acc_bf16x8(a, vs, 1.0f);
            if (residual) acc_bf16x8(a, vr, 1.0f);
            uint4 o;
            o.x = pack_bf16x2(a[0], a[1]);
            o.y = pack_bf16x2(a[2], a[3]);
            o.z = pack_bf16x2(a[4], a[5]);
            o.w = pack_bf16x2(a[6], a[7]);
            out[(size_t)t * HV + c] = o;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, const uint16_t* y_perm, const int32_t* dest, const float* w,
                           const uint16_t* y_shared, const uint16_t* residual, uint16_t* out, WsHeader* gate,
                           cudaStream_t st) {
    const int HV = s.hidden / 8;
    int threads = 32;
    while (threads < 256 && threads < HV) threads *= 2;
    long long blocks = s.tokens;
    const long long cap = (long long)device_sm_count() * (2048 / threads);
    if (blocks > cap) blocks = cap;
    // Launched early (programmatic dependency) only for small layers: there it
    // hides the launch behind the down projection's tail; behind a long GEMM
    // its waiting blocks measured ~1 % slower on the 16384-token layer.
    const bool pdl = kUsePdl && s.tokens <= kDecodeRows;
    return launch_kernel(combine_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, 1, pdl, s.tokens, HV,
                         s.top_k, reinterpret_cast<const uint4*>(y_perm), dest, w, reinterpret_cast<const uint4*>(y_shared),
                         reinterpret_cast<const uint4*>(residual), reinterpret_cast<uint4*>(out), gate);
}

}  // namespace moe
