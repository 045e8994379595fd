// small_dispatch.cu -- route + count + scatter in one kernel for decode-sized
// batches (at most kSmallDispatchTokens tokens).
//
// The count-first dispatch of dispatch.cu (afdEP-comm count-first record:
// counts and their prefix sums before any payload row moves; capacity checked
// first; invalid routes isolated) and the softmax top-k routing of route.cu
// (ONNX Runtime PR #33963, "Measured CUDA kernel latency"), for a batch small
// enough that one CTA can route every token and rank every pair: every CTA of
// the grid does so redundantly in shared memory, then copies the rows of its
// own tokens.  CTA 0 publishes the routing (ids, weights), the counts, the
// offsets and the capacity verdict.  This replaces three latency-bound
// launches by one at decode.
//
// The results are bit for bit those of route_kernel + count_kernel +
// scatter_kernel: the routing is the same warp routine (route_warp.cuh), and
// the slot of pair p is offsets[e] + #{p' < p : ids[p'] = e} (stable in p),
// validated the same way (0 <= id < E, no earlier duplicate in the token).
#include "common.cuh"
#include "route_warp.cuh"

#include <type_traits>

namespace moe {
namespace {

constexpr int kSDThreads = 512;                         // 16 warps: one token per warp
constexpr int kSDItems = (kSmallDispatchTokens * 32 + kSDThreads - 1) / kSDThreads;   // pairs per thread

__device__ __forceinline__ unsigned sd_lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <int EPL>
__global__ void __launch_bounds__(kSDThreads)
small_dispatch_kernel(int T, int E, int k, int capacity, const float* __restrict__ logits,
                      const int32_t* __restrict__ ids_in, int32_t* __restrict__ ids_out, float* __restrict__ w_out,
                      const uint4* __restrict__ x, int HV, int32_t* __restrict__ counts,
                      int32_t* __restrict__ offsets, int32_t* __restrict__ dest, int32_t* __restrict__ sorted_pair,
                      uint4* __restrict__ x_perm, WsHeader* hdr, unsigned* __restrict__ sync, int nsync) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int sm[];
    const int R = T * k;
    int* ids_s = sm;                  // [R]
    int* hist = ids_s + R;            // [E]   counts
    int* offs = hist + E;             // [E+1] exclusive scan
    int* dest_s = offs + E + 1;       // [R]
    __shared__ int warp_tot[kSDThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool lead = blockIdx.x == 0;

    // ---- routing (or the caller's preselected ids) ----------------------------
    if (logits) {
        for (int t = warp; t < T; t += kSDThreads / 32) {
            int sel_i;
            float sel_w;
            if (route_token_softmax<EPL>(logits + (size_t)t * E, E, k, lane, sel_i, sel_w) && lane == 0 && lead)
                raise_status(hdr, MOE_ERR_NONFINITE);
            if (lane < k) {
                ids_s[t * k + lane] = sel_i;
                if (lead) {
                    ids_out[(size_t)t * k + lane] = sel_i;
                    w_out[(size_t)t * k + lane] = sel_w;
                }
            }
        }
    } else {
        for (int p = tid; p < R; p += kSDThreads) ids_s[p] = ids_in[p];
    }
    for (int e = tid; e < E; e += kSDThreads) hist[e] = 0;
    __syncthreads();

    // ---- validity and stable ranks: warps in order, pairs in p order ------------
    int item_e[kSDItems], item_r[kSDItems];
#pragma unroll
    for (int it = 0; it < kSDItems; ++it) {
        const int p = it * kSDThreads + tid;
        int e = -1;
        if (p < R) {
            const int id = ids_s[p];
            const int t = p / k, j = p - t * k;
            bool ok = (id >= 0 && id < E);
            for (int jj = 0; jj < j && ok; ++jj)
                if (ids_s[t * k + jj] == id) ok = false;
            if (ok) e = id;
            else if (lead) raise_status(hdr, MOE_ERR_INVALID_ROUTE);
        }
        const unsigned grp = __match_any_sync(0xffffffffu, e);
        const int lrank = __popc(grp & sd_lanemask_lt());
        const bool leader = (lane == 31 - __clz(grp));
        int r = 0;
        // warps in order; only the warps that hold pairs of this item
        const int left = R - it * kSDThreads;
        const int nw = left <= 0 ? 0 : (left >= kSDThreads ? kSDThreads / 32 : (left + 31) / 32);
        for (int w = 0; w < nw; ++w) {
            if (warp == w) {
                const int base = (e >= 0) ? hist[e] : 0;
                __syncwarp();
                if (e >= 0 && leader) hist[e] = base + __popc(grp);
                r = base + lrank;
            }
            __syncthreads();
        }
        item_e[it] = e;
        item_r[it] = r;
    }

    // ---- offsets: exclusive scan of the counts; capacity ------------------------
    const int per = (E + kSDThreads - 1) / kSDThreads;
    const int e0 = tid * per;
    int loc = 0;
    for (int i = 0; i < per; ++i)
        if (e0 + i < E) loc += hist[e0 + i];
    int inc = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += n;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int run = inc - loc;
    for (int w = 0; w < warp; ++w) run += warp_tot[w];
    int over = 0;
    for (int i = 0; i < per; ++i) {
        const int e = e0 + i;
        if (e < E) {
            const int c = hist[e];
            offs[e] = run;
            if (lead) {
                counts[e] = c;
                offsets[e] = run;
            }
            if (c > capacity) over = 1;
            run += c;
        }
    }
    if (tid == kSDThreads - 1) {
        offs[E] = run;
        if (lead) offsets[E] = run;
    }
    if (lead && sync)   // the fused decode FFN's counters start from zero
        for (int i = tid; i < nsync; i += kSDThreads) sync[i] = 0u;
    const int any_over = __syncthreads_or(over);
    if (lead && tid == 0) {
        hdr->cap_exceeded = any_over;
        if (any_over) raise_status(hdr, MOE_ERR_CAPACITY);
        // ids, weights, counts, offsets, the counters and the verdict are
        // written (the block barrier above orders the other threads' stores
        // before this fence); the layer's last kernel puts route_ready back to 0
        __threadfence();
        st_release_u32(&hdr->route_ready, 1u);
    }
    if (any_over) return;                              // over capacity: no payload moves
#pragma unroll
    for (int it = 0; it < kSDItems; ++it) {
        const int p = it * kSDThreads + tid;
        if (p < R) dest_s[p] = item_e[it] >= 0 ? offs[item_e[it]] + item_r[it] : -1;
    }
    __syncthreads();

    // ---- this CTA's tokens: placement and the 16-byte row copies -----------------
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (tid < k) {
            const int p = t * k + tid;
            const int d = dest_s[p];
            dest[p] = d;
            if (d >= 0) sorted_pair[d] = p;
        }
        const uint4* src = x + (size_t)t * HV;
        for (int idx = tid; idx < k * HV; idx += kSDThreads) {
            const int j = idx / HV, c = idx - j * HV;
            const int d = dest_s[t * k + j];
            if (d >= 0) x_perm[(size_t)d * HV + c] = __ldg(src + c);
        }
    }
}

template <int EPL>
cudaError_t launch_sd(const moe_shape& s, const float* logits, const int32_t* ids_in, int32_t* ids_out, float* w_out,
                      const uint16_t* x, int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* sorted_pair,
                      uint16_t* x_perm, WsHeader* hdr, unsigned* sync, int nsync, cudaStream_t st) {
    const int R = s.tokens * s.top_k;
    const size_t smem = (size_t)(2 * R + 2 * s.experts + 1) * sizeof(int);
    const int grid = s.tokens < device_sm_count() ? s.tokens : device_sm_count();
    return launch_kernel(small_dispatch_kernel<EPL>, dim3((unsigned)grid), dim3(kSDThreads), smem, st, 1, kUsePdl,
                         s.tokens, s.experts, s.top_k, s.capacity, logits, ids_in, ids_out, w_out,
                         reinterpret_cast<const uint4*>(x), s.hidden / 8, counts, offsets, dest, sorted_pair,
                         reinterpret_cast<uint4*>(x_perm), hdr, sync, nsync);
}

}  // namespace

cudaError_t launch_small_dispatch(const moe_shape& s, const float* logits, const int32_t* ids_in, int32_t* ids_out,
                                  float* w_out, const uint16_t* x, int32_t* counts, int32_t* offsets, int32_t* dest,
                                  int32_t* sorted_pair, uint16_t* x_perm, WsHeader* hdr, unsigned* sync, int nsync,
                                  cudaStream_t st) {
    if (s.tokens > kSmallDispatchTokens) return cudaErrorInvalidValue;
    auto go = [&](auto epl) {
        return launch_sd<decltype(epl)::value>(s, logits, ids_in, ids_out, w_out, x, counts, offsets, dest,
                                               sorted_pair, x_perm, hdr, sync, nsync, st);
    };
    const int E = s.experts;
    if (E <= 32) return go(std::integral_constant<int, 1>{});
    if (E <= 64) return go(std::integral_constant<int, 2>{});
    if (E <= 128) return go(std::integral_constant<int, 4>{});
    if (E <= 256) return go(std::integral_constant<int, 8>{});
    if (E <= 512) return go(std::integral_constant<int, 16>{});
    return go(std::integral_constant<int, 32>{});
}

}  // namespace moe
