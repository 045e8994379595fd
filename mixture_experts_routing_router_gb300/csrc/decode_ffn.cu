// decode_ffn.cu -- K9, the decode layer's expert FFN and weighted combine in one
// launch (moe_layer, 2 to kSmallDispatchTokens tokens, BF16 weights, no shared
// experts, hidden and intermediate whole 64-column chunks).
//
// At decode a layer streams its experts' weights from HBM (ONNX Runtime PR
// #33963, "Measured CUDA kernel latency": 1 to 16 tokens over 9 experts of 240).
// Three kernels (up projection, down projection, combine) pay two kernel
// boundaries -- the dependent's programmatic wait returns about a microsecond
// after the last CTA of its predecessor ends -- and the down projection's
// weights cannot stream until the up projection has ended.  Here one
// persistent grid (at most one CTA per SM) takes the work items of both
// projections in one list, up items first:
//
//   up item (expert e, 128-row block nt of W13): h rows of e's bucket, columns
//     nt*128.. (SwiGLU silu(g)*u or ReLU^2, the small-row kernel's arithmetic);
//   down item (expert e, 128-row block nt of W2): y_perm rows of e's bucket,
//     columns nt*128..
//
// and each item is the small-row kernel's swapped MMA (D^T = W * X^T: 128
// weight rows on M, the bucket's rows padded to 16 on N, FP32 in TMEM), with
// stages of up to four 64-column chunks of K (one TMA box of weights, one of
// activations).  The dependencies between items are counters in the
// workspace, zeroed by the fused dispatch before it publishes the bucket
// bounds:
//
//   - an up item's activations are x_perm rows, copied by the fused dispatch
//     after it published the bounds: the producer takes the programmatic wait
//     before its first up activation load (weights go out before it);
//   - a down item's activations are the h rows of its expert: the up items'
//     epilogues count finished blocks per expert (release), and the producer of
//     a down item waits (acquire, bounded) for all of them before it loads h
//     through TMA (after a proxy fence); its weights go out before that;
//   - epilogue warp q of a down item writes columns 32q..32q+31 of its
//     128-column tile; the warps count finished experts per tile quarter
//     (acquire-release), and the one that completes a quarter combines those
//     32 columns for every token: out[t] = bf16(sum_j w[t,j] *
//     y_perm[dest[t*k+j]] + residual[t]), FP32, j in order -- the combine
//     kernel's arithmetic.
//
// A CTA takes its items in list order, up items before down items, so every up
// item is taken by a CTA that finishes it before it can wait on anything, and
// no wait closes a cycle; every wait is bounded (MOE_ERR_TIMEOUT, TMEM freed,
// no trap).  Outputs are bit for bit those of the three separate kernels.
#include "common.cuh"

#include <mutex>

namespace moe {
namespace {

constexpr int FBM = 128;                    // weight rows per item (MMA M)
constexpr int FBK = 64;                     // K chunk: 64 BF16 = one 128-byte swizzle row
constexpr int FNB = 16;                     // bucket rows per item (MMA N)
constexpr int F_WBOX = FBM * FBK * 2;       // 16 KiB: 128 weight rows of one chunk
constexpr int F_XBOX = FNB * FBK * 2;       // 2 KiB: 16 activation rows of one chunk
constexpr int F_THREADS = 192;              // producer, MMA, 4 epilogue warps
constexpr int F_MAX_STAGES = 4;
constexpr int F_MAX_SMEM = 222 * 1024;

struct FParams {
    const int32_t* offsets;     // [E + 1] bucket bounds
    const int32_t* dest;        // [T * k] slot of pair p, or negative
    const float* topk_w;        // [T * k] routing weights
    const uint4* residual;      // [T, H] BF16 or null (may alias out)
    uint16_t* h;                // [R, I] up projection output
    uint16_t* y_perm;           // [R, H] down projection output
    uint4* out;                 // [T, H] layer output
    unsigned* cnt_up;           // [E] finished epilogue warps of up items per expert (4 per item)
    unsigned* cnt_dn;           // [4 * ntn_dn] finished epilogue warps of down items per output column
                                //   tile and quarter (warp q writes columns 32q.. of a tile); one more word
                                //   counts the CTAs that have finished
    WsHeader* hdr;
    int E, T, k, R, H, I;
    int up_group_rows;          // W13 rows per expert (2I SwiGLU, I ReLU^2)
    int kc_up, kc_dn;           // K chunks per stage
    int stages, stage_bytes;
};

struct FCtl {
    unsigned long long full[F_MAX_STAGES];
    unsigned long long empty[F_MAX_STAGES];
    unsigned long long tfull[2];
    unsigned long long tempty[2];
    unsigned long long drain;
    uint32_t tmem_base;
    int abort;
    int ng;                     // non-empty experts
    int wsum[F_THREADS / 32];
};

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_acq_rel_add(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void acc8(float (&a)[8], const uint4& v, float w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), a[2 * i]);
        a[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xffff0000u), a[2 * i + 1]);
    }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// Combine 16-byte column groups [c0, c1) of every token, thread i of nthr.
// Routing and placement were written by the fused dispatch, y_perm by other
// CTAs before the acquire that led here: all read through L2.  A token's
// slots and weights are loaded together, then its rows eight at a time, and
// summed in j order.
__device__ void combine_columns(const FParams& p, int c0, int c1, int i, int nthr) {
    const int HV = p.H / 8, cols = c1 - c0;
    const uint4* yp = reinterpret_cast<const uint4*>(p.y_perm);
    for (int idx = i; idx < p.T * cols; idx += nthr) {
        const int t = idx / cols, c = c0 + idx % cols;
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint4 vr = make_uint4(0u, 0u, 0u, 0u);
        if (p.residual) vr = __ldcg(p.residual + (size_t)t * HV + c);
        for (int j0 = 0; j0 < p.k; j0 += 8) {
            int d[8];
            float w[8];
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                d[u] = -1;
                if (j < p.k) {
                    d[u] = __ldcg(p.dest + (size_t)t * p.k + j);
                    w[u] = __ldcg(p.topk_w + (size_t)t * p.k + j);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (d[u] >= 0 && d[u] < p.R) v[u] = __ldcg(yp + (size_t)d[u] * HV + c);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (d[u] >= 0 && d[u] < p.R) acc8(a, v[u], w[u]);
        }
        if (p.residual) acc8(a, vr, 1.0f);
        uint4 o;
        o.x = pack2(a[0], a[1]);
        o.y = pack2(a[2], a[3]);
        o.z = pack2(a[4], a[5]);
        o.w = pack2(a[6], a[7]);
        p.out[(size_t)t * HV + c] = o;
    }
}

template <int MODE>     // the up projection's activation: kGemmSwiGLU or kGemmReLU2
__global__ void __launch_bounds__(F_THREADS, 1)
decode_ffn_kernel(const __grid_constant__ CUtensorMap tmX,     // x_perm: 16-row boxes of kc_up chunks
                  const __grid_constant__ CUtensorMap tmW13,   // W13: 128-row boxes (SwiGLU: gate | up rows)
                  const __grid_constant__ CUtensorMap tmH,     // h: 16-row boxes of kc_dn chunks
                  const __grid_constant__ CUtensorMap tmW2,    // W2: 128-row boxes of kc_dn chunks
                  const FParams p) {
    constexpr int NW = MODE == kGemmSwiGLU ? 2 : 1;      // up: weight blocks per chunk
    constexpr uint32_t ACC_COLS = NW * FNB;                // columns of one accumulator
    constexpr uint32_t TMEM_COLS = 2 * ACC_COLS < 32 ? 32 : 2 * ACC_COLS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    FCtl* ctl = reinterpret_cast<FCtl*>(smem + (size_t)p.stages * p.stage_bytes);
    int* gid = reinterpret_cast<int*>(ctl + 1);            // [E] non-empty experts, in order
    int* gst = gid + p.E;                                   // first bucket row
    int* gcnt = gst + p.E;                                  // bucket rows
    const uint32_t smem_base = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), 4);        // the 4 epilogue warps
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW13);
        tma_prefetch_desc(&tmH);
        tma_prefetch_desc(&tmW2);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    // The bucket bounds: published by the fused dispatch (route_ready); after a
    // bounded look, the programmatic wait (every thread) is the fallback.
    __shared__ int early_ok;
    if (tid == 0) {
        const unsigned long long t0 = globaltimer_ns();
        unsigned ready;
        while ((ready = ld_acquire_u32(&p.hdr->route_ready)) == 0u && globaltimer_ns() - t0 < kEarlyWaitNs) { }
        early_ok = ready != 0u;
    }
    __syncthreads();
    const bool waited = !early_ok;
    if (waited) pdl_wait();
    const bool skip = __ldcg(&p.hdr->cap_exceeded) != 0;   // over capacity: no payload moved

    // ---- the non-empty experts (block-wide compaction of the bounds) ---------
    // each thread's experts g0 .. g0+per-1 (per <= 6: at most 1024 experts over
    // 192 threads): their per+1 bounds read once, together, through L2
    {
        constexpr int kMaxPer = 8;
        const int per = (p.E + F_THREADS - 1) / F_THREADS;
        const int g0 = tid * per;
        int bnd[kMaxPer + 1];
#pragma unroll
        for (int i = 0; i <= kMaxPer; ++i) {
            const int g = g0 + i;
            const int v = (!skip && i <= per && g <= p.E) ? __ldcg(p.offsets + g) : 0;
            bnd[i] = v < 0 ? 0 : (v > p.R ? p.R : v);
        }
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i)
            if (i < per && g0 + i < p.E) cnt += bnd[i + 1] > bnd[i];
        int inc = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        if (lane == 31) ctl->wsum[warp] = inc;
        __syncthreads();
        int kk = inc - cnt;
        for (int w = 0; w < warp; ++w) kk += ctl->wsum[w];
        if (tid == F_THREADS - 1) ctl->ng = kk + cnt;
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i) {
            const int g = g0 + i;
            if (i < per && g < p.E && bnd[i + 1] > bnd[i]) {
                gid[kk] = g;
                gst[kk] = bnd[i];
                gcnt[kk] = bnd[i + 1] - bnd[i];
                ++kk;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort = &ctl->abort;
    const int ng = ctl->ng;
    const int ntn_up = (p.I + FBM - 1) / FBM, ntn_dn = (p.H + FBM - 1) / FBM;
    const int U = ng * ntn_up, items = U + ng * ntn_dn;
    const int nch_up = p.H / FBK, nch_dn = p.I / FBK;       // K chunks of each projection
    const int nst_up = (nch_up + p.kc_up - 1) / p.kc_up, nst_dn = (nch_dn + p.kc_dn - 1) / p.kc_dn;
    // item it: up (expert slot, 128-row block of W13) for it < U, else down
    auto item = [&](int it, bool& dn, int& slot, int& nt) {
        dn = it >= U;
        const int j = dn ? it - U : it, per = dn ? ntn_dn : ntn_up;
        slot = j / per;
        nt = j - slot * per;
    };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true, dispatch_done = waited;
            long long armed = 0;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                bool dn;
                int slot, nt;
                item(it, dn, slot, nt);
                const int g = gid[slot], row0 = gst[slot];
                const int kc = dn ? p.kc_dn : p.kc_up, nst = dn ? nst_dn : nst_up;
                const uint32_t wbytes = (uint32_t)(kc * (dn ? 1 : NW) * F_WBOX);     // weights, then activations
                const uint32_t tx = wbytes + (uint32_t)(kc * F_XBOX);
                auto load_w = [&](uint32_t sa, uint32_t full, int i) {
                    if (dn)
                        tma_load_3d(sa, &tmW2, full, 0, g * p.H + nt * FBM, i * kc);
                    else if (MODE == kGemmSwiGLU)   // per chunk: 128 gate rows, then the up rows
                        tma_load_5d(sa, &tmW13, full, 0, nt * FBM, 0, g, i * kc);
                    else
                        tma_load_3d(sa, &tmW13, full, 0, g * p.up_group_rows + nt * FBM, i * kc);
                };
                // weights of the item's first stages go out before its activations are
                // ready: all the ring for an up item (the fused dispatch ends soon), one
                // stage for a down item (its wait is long, and the up items' weights
                // still stream from the same HBM)
                const int npre = dn ? 1 : (nst < p.stages ? nst : p.stages);
                {
                    int s = stage;
                    uint32_t sph = ph;
                    for (int i = 0; i < npre; ++i) {
                        if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), sph ^ 1u, abort)) { ok = false; break; }
                        const uint32_t full = smem_u32(&ctl->full[s]);
                        mbar_arrive_expect_tx(full, tx);
                        load_w(smem_base + (uint32_t)(s * p.stage_bytes), full, i);
                        ++armed;
                        if (++s == p.stages) { s = 0; sph ^= 1u; }
                    }
                }
                if (!ok) break;
                if (!dn) {
                    // x_perm rows: copied by the fused dispatch after it published the bounds
                    if (!dispatch_done) {
                        pdl_wait();
                        dispatch_done = true;
                    }
                } else {
                    // h rows of expert g: every epilogue warp of every up item of g has
                    // counted (release)
                    const unsigned* c = p.cnt_up + g;
                    const unsigned need = 4u * (unsigned)ntn_up;
                    if (ld_acquire_gpu(c) < need) {
                        const unsigned long long t0 = globaltimer_ns();
                        for (uint32_t n = 1;; ++n) {
                            if (ld_acquire_gpu(c) >= need) break;
                            if ((n & 31u) == 0u) {
                                if (*abort) { ok = false; break; }
                                if (globaltimer_ns() - t0 > kWaitLimitNs) { *abort = 1; ok = false; break; }
                            }
                        }
                    }
                    // the generic-proxy writes of h are read by the TMA (async proxy)
                    fence_proxy_async_global();
                }
                if (!ok) break;
                for (int i = 0; i < nst; ++i) {
                    const uint32_t full = smem_u32(&ctl->full[stage]);
                    const uint32_t sa = smem_base + (uint32_t)(stage * p.stage_bytes);
                    if (i >= npre) {
                        if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort)) { ok = false; break; }
                        mbar_arrive_expect_tx(full, tx);
                        load_w(sa, full, i);
                        ++armed;
                    }
                    if (dn) tma_load_3d(sa + wbytes, &tmH, full, 0, row0, i * kc);
                    else tma_load_3d(sa + wbytes, &tmX, full, 0, row0, i * kc);
                    if (++stage == p.stages) { stage = 0; ph ^= 1u; }
                }
            }
            // the grid never ends before the fused dispatch does
            if (!dispatch_done) pdl_wait();
            if (!ok) {
                // let the copies already issued land before the CTA exits (stages whose
                // activations never went out cannot complete: the fixed delay follows)
                if (!wait_armed_stages(smem_u32(&ctl->full[0]), p.stages, armed)) settle_delay();
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteDecodeFfn;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(FBM, FNB);
            int stage = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                bool dn;
                int slot, nt;
                item(it, dn, slot, nt);
                const int kc = dn ? p.kc_dn : p.kc_up, nst = dn ? nst_dn : nst_up, nch = dn ? nch_dn : nch_up;
                const int nwb = dn ? 1 : NW;                     // weight blocks per chunk
                const uint32_t wbytes = (uint32_t)(kc * nwb * F_WBOX);
                if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)acc * ACC_COLS;
                for (int i = 0; i < nst; ++i) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), ph, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_base + (uint32_t)(stage * p.stage_bytes);
                    const int nc = nch - i * kc < kc ? nch - i * kc : kc;   // chunks of K in this stage
                    for (int c = 0; c < nc; ++c) {
                        const uint32_t wa = sa + (uint32_t)(c * nwb * F_WBOX);
                        const uint64_t wd = sdesc_k_sw128(wa);
                        const uint64_t xd = sdesc_k_sw128(sa + wbytes + (uint32_t)(c * F_XBOX));
#pragma unroll
                        for (int kk = 0; kk < FBK / 16; ++kk) {
                            const uint32_t accum = (i > 0 || c > 0 || kk > 0) ? 1u : 0u;
                            tc_mma_bf16(d, wd + (uint64_t)(kk * 2), xd + (uint64_t)(kk * 2), idesc, accum);
                            if (MODE == kGemmSwiGLU && !dn)
                                tc_mma_bf16(d + (uint32_t)FNB, sdesc_k_sw128(wa + F_WBOX) + (uint64_t)(kk * 2),
                                            xd + (uint64_t)(kk * 2), idesc, accum);
                        }
                    }
                    tc_commit(smem_u32(&ctl->empty[stage]));
                    if (++stage == p.stages) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit(smem_u32(&ctl->tfull[acc]));
                if (++acc == 2) { acc = 0; aph ^= 1u; }
            }
            // drain: every MMA this thread issued has completed
            tc_commit(smem_u32(&ctl->drain));
            volatile int never = 0;
            const bool drained = mbar_wait_bounded(smem_u32(&ctl->drain), 0, &never);
            if (!ok || !drained) {
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteDecodeFfn;
                *abort = 1;
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;                                 // TMEM lane quarter
        const int tid_e = tid - 64;                             // 0..127
        int acc = 0;
        uint32_t aph = 0;
        bool ok = true, pdl_done = waited;
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            bool dn;
            int slot, nt;
            item(it, dn, slot, nt);
            const int g = gid[slot], row0 = gst[slot], rows = gcnt[slot];
            const int N = dn ? p.H : p.I;
            uint16_t* obase = dn ? p.y_perm : p.h;
            const int n = nt * FBM + 32 * q + lane;             // weight row = output column
            if (!mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort)) {
                if (lane == 0) {
                    raise_status(p.hdr, MOE_ERR_TIMEOUT);
                    p.hdr->timeout_site = kSiteDecodeFfn;
                }
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem + (uint32_t)acc * ACC_COLS + ((uint32_t)(32 * q) << 16);
            uint32_t gv[16], uv[16];
            tmem_ld_16cols(taddr, gv);
            if (MODE == kGemmSwiGLU && !dn) tmem_ld_16cols(taddr + (uint32_t)FNB, uv);
            tmem_ld_wait();
            if (n < N) {
#pragma unroll
                for (int r = 0; r < FNB; ++r) {
                    if (r < rows) {
                        const float x = __uint_as_float(gv[r]);
                        float a;
                        if (dn) a = x;
                        else if (MODE == kGemmSwiGLU) a = x / (1.0f + __expf(-x)) * __uint_as_float(uv[r]);
                        else a = x > 0.f ? x * x : 0.f;
                        reinterpret_cast<__nv_bfloat16*>(obase)[(size_t)(row0 + r) * N + n] = __float2bfloat16_rn(a);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
            if (++acc == 2) { acc = 0; aph ^= 1u; }
            // publish this warp's quarter of the block: its stores, then one count
            // (four per item; no barrier across warps, so a warp that gave up on a
            // wait leaves the others to their own bounded waits)
            __threadfence();
            __syncwarp();
            unsigned done = 0;
            if (lane == 0) {
                if (!dn) red_release_add(p.cnt_up + g, 1u);
                else done = atom_acq_rel_add(p.cnt_dn + 4 * nt + q, 1u) + 1u;
            }
            done = __shfl_sync(0xffffffffu, done, 0);
            if (dn && done == (unsigned)ng) {
                // every expert's rows of this warp's 32 columns of the tile are in
                // y_perm: combine those columns for every token
                if (!pdl_done) {
                    pdl_wait();
                    pdl_done = true;
                }
                const int c0 = nt * (FBM / 8) + 4 * q;
                const int c1 = c0 + 4 < p.H / 8 ? c0 + 4 : p.H / 8;
                if (c0 < c1) combine_columns(p, c0, c1, lane, 32);
            }
        }
        // no routed row at all (every route invalid): out is the residual, or zero
        if (ok && ng == 0 && !skip && blockIdx.x == 0) {
            if (!pdl_done) pdl_wait();
            combine_columns(p, 0, p.H / 8, tid_e, 128);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    // the last CTA out: the next layer call's fused dispatch publishes its
    // bounds afresh
    if (tid == 0 && atom_acq_rel_add(p.cnt_dn + 4 * ntn_dn, 1u) == gridDim.x - 1u) p.hdr->route_ready = 0u;
}

template <int MODE>
cudaError_t launch_f(const CUtensorMap& mx, const CUtensorMap& m13, const CUtensorMap& mh, const CUtensorMap& m2,
                     const FParams& fp, unsigned grid, size_t smem, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(decode_ffn_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        F_MAX_SMEM);
    });
    if (attr_err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(decode FFN, %d bytes): %s", F_MAX_SMEM, cudaGetErrorString(attr_err));
        return attr_err;
    }
    const cudaError_t e = launch_kernel(decode_ffn_kernel<MODE>, dim3(grid), dim3(F_THREADS), smem, st, 1, kUsePdl,
                                        mx, m13, mh, m2, fp);
    if (e != cudaSuccess) set_error("decode FFN launch: %s", cudaGetErrorString(e));
    return e;
}

}  // namespace

// One token: the three separate kernels measured level or up to a microsecond
// faster (timer quantum about 1 us); from two tokens on, this kernel is faster
// (4 tokens 35 vs 40 us, 8 tokens 35 vs 46 us on the 240-expert decode layer).
bool decode_ffn_fits(const moe_shape& s) {
    return s.tokens >= 2 && s.tokens <= kSmallDispatchTokens && s.shared == 0 && s.hidden % FBK == 0 &&
           s.inter % FBK == 0 &&
           (s.act == MOE_ACT_SWIGLU || s.act == MOE_ACT_RELU2);
}

size_t decode_ffn_sync_words(const moe_shape& s) {
    return (size_t)s.experts + 4 * (size_t)((s.hidden + FBM - 1) / FBM) + 1;
}

moe_status launch_decode_ffn(const moe_shape& s, const uint16_t* x_perm, const int32_t* offsets,
                             const uint16_t* w13, const uint16_t* w2, uint16_t* h, uint16_t* y_perm,
                             const int32_t* dest, const float* topk_w, const uint16_t* residual, uint16_t* out,
                             unsigned* sync, WsHeader* hdr, cudaStream_t st) {
    if (!decode_ffn_fits(s)) {
        set_error("decode FFN: shape outside its scope");
        return MOE_ERR_INTERNAL;
    }
    const bool glu = s.act == MOE_ACT_SWIGLU;
    const int nw = glu ? 2 : 1;
    const long long E = s.experts, H = s.hidden, I = s.inter, R = (long long)s.tokens * s.top_k;
    FParams fp;
    fp.offsets = offsets;
    fp.dest = dest;
    fp.topk_w = topk_w;
    fp.residual = reinterpret_cast<const uint4*>(residual);
    fp.h = h;
    fp.y_perm = y_perm;
    fp.out = reinterpret_cast<uint4*>(out);
    fp.cnt_up = sync;
    fp.cnt_dn = sync + E;
    fp.hdr = hdr;
    fp.E = (int)E;
    fp.T = s.tokens;
    fp.k = s.top_k;
    fp.R = (int)R;
    fp.H = (int)H;
    fp.I = (int)I;
    fp.up_group_rows = (int)(nw * I);
    // stages: as many K chunks per box as leave three stages of either projection
    const size_t fixed = 1024 + sizeof(FCtl) + (size_t)3 * E * sizeof(int);
    auto pick = [&](int wblocks) {
        int kc = 4;
        while (kc > 1 && fixed + 3 * (size_t)kc * (wblocks * F_WBOX + F_XBOX) > (size_t)F_MAX_SMEM) --kc;
        return kc;
    };
    fp.kc_up = pick(nw);
    fp.kc_dn = pick(1);
    const int sb_up = fp.kc_up * (nw * F_WBOX + F_XBOX), sb_dn = fp.kc_dn * (F_WBOX + F_XBOX);
    fp.stage_bytes = sb_up > sb_dn ? sb_up : sb_dn;
    long long stages = ((long long)F_MAX_SMEM - (long long)fixed) / fp.stage_bytes;
    if (stages > F_MAX_STAGES) stages = F_MAX_STAGES;
    if (stages < 2) {
        set_error("decode FFN: %d-byte stages do not fit shared memory", fp.stage_bytes);
        return MOE_ERR_UNSUPPORTED;
    }
    fp.stages = (int)stages;
    const size_t smem = fixed + (size_t)stages * fp.stage_bytes;
    // at most one CTA per SM; no more than the items of the largest possible batch
    const long long groups = R < E ? R : E;
    long long grid = groups * (((I + FBM - 1) / FBM) + ((H + FBM - 1) / FBM));
    const int sms = device_sm_count() - s.tokens;     // the fused dispatch holds one SM per token
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    CUtensorMap mx, m13, mh, m2;
    if (!make_tensor_map_bf16_chunks(&mx, x_perm, R, H, (unsigned)FNB, (unsigned)fp.kc_up) ||
        (glu ? !make_tensor_map_glu_chunks(&m13, w13, E * 2 * I, H, I, 2 * I, (unsigned)FBM, (unsigned)fp.kc_up)
             : !make_tensor_map_bf16_chunks(&m13, w13, E * I, H, (unsigned)FBM, (unsigned)fp.kc_up)) ||
        !make_tensor_map_bf16_chunks(&mh, h, R, I, (unsigned)FNB, (unsigned)fp.kc_dn) ||
        !make_tensor_map_bf16_chunks(&m2, w2, E * H, I, (unsigned)FBM, (unsigned)fp.kc_dn))
        return MOE_ERR_CUDA;
    const cudaError_t e = glu ? launch_f<kGemmSwiGLU>(mx, m13, mh, m2, fp, (unsigned)grid, smem, st)
                              : launch_f<kGemmReLU2>(mx, m13, mh, m2, fp, (unsigned)grid, smem, st);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
