// gemm_decode.cu -- K8, the small-row ("decode") form of the grouped GEMM.
//
// At decode a routed expert sees a handful of tokens (ONNX Runtime PR #33963,
// "Measured CUDA kernel latency": 1, 8 and 16 rows over 9 experts of 240), so
// every weight element serves a few rows and the layer streams weights.  This
// kernel swaps the operands of the grouped GEMM: D^T = W * X^T, with 128 weight
// rows on the MMA's M side and NB of the group's rows (16..64, a multiple of
// 16) on its N side, FP32 in TMEM.  A work item is one 128-row block of one
// non-empty group's weights, so a single token already spreads its experts'
// weights over ~100 SMs.  A group with more than NB rows is taken in NB-row
// chunks, re-streaming its weights per chunk (correct for any bucket; the host
// picks NB from a bound on the rows per group).
//
// Persistent CTAs (at most one per SM) take items round-robin.  Roles: warp 0
// lane 0 issues the TMA loads of a ring of stages; warp 1 lane 0 issues
// tcgen05.mma into one of two accumulators;
// warps 2..5 run the epilogue (warp w owns TMEM lanes 32(w%4)..+31, i.e. the
// output columns n0 + 32(w%4) + lane) while the next item streams.  The list
// of non-empty groups is built once per CTA from the offsets.
//
// BF16 stages: the TMA unit of an SM takes about the same time per stage for
// 16 as for 64 KiB (a streaming microbenchmark: ~45 GB/s per SM from DRAM with
// one 16 KiB box per stage, ~150 GB/s with 64 KiB stages), so a stage carries
// up to four 64-column chunks of K: the 128 weight rows of each chunk (SwiGLU:
// gate rows then the matching up rows) in one box of a (column in chunk, row,
// chunk) view, the NB activation rows of each chunk in one more.  K that is not
// a whole number of chunks takes one chunk per stage through 2-D maps.
//
// The epilogue arithmetic is the tile kernels': SwiGLU silu(g)*u, ReLU^2,
// plain, or the FP32 accumulator.  Every wait is bounded (MOE_ERR_TIMEOUT,
// TMEM freed, no trap).
//
// FP8 weights (WF = kWeightFp8E4M3): the weights arrive as OCP E4M3 codes with
// one FP32 scale per weight row -- the ONNX Runtime operator's weight-only
// quantized experts (BF16 activations), with E4M3 as the codec.  Every E4M3
// value is exact in BF16, so eight more warps (6..13) convert each TMA-loaded
// code box (128 rows x 128 bytes, 128-byte swizzle: one 128-byte request per
// weight row, as for BF16) straight into TMEM -- each thread one weight row,
// its TMEM lane -- where the MMA reads its A operand (tcgen05.mma with A in
// TMEM), in a ring of slots.  The MMA stays BF16 with FP32 accumulation; the
// row scale multiplies the accumulator in the epilogue.
// A stage holds its activation boxes first, then the code boxes.  With one
// weight block per stage (ReLU^2, plain) a stage is 256 K elements (two code
// boxes) converted as one chunk into a 128-column slot; SwiGLU (gate and up
// blocks) takes 128 K elements per stage.  The converter-to-MMA handshake per
// chunk, not the bytes, sets this kernel's pace, so larger chunks are faster.
//
// NVFP4 weights (the same page's NVFP4 cases; standard NVFP4 layout): E2M1
// codes, two per byte with the lower K index in the low nibble, an E4M3 scale
// per 16 consecutive elements of a row and an FP32 scale per row.  A stage is
// 256 K elements: one 128-byte code row per weight row and TMA request (as for
// FP8), the rows' 16 block scales (a 128 x 16-byte box) and four activation
// boxes.  The converter warps form e2m1 * block scale * 2^-8 -- exact in BF16,
// the scale applied before the cast -- into the TMEM slots (the whole stage as
// one chunk with one weight block, two 128-wide chunks for SwiGLU), and the
// epilogue multiplies by the row scale * 2^8.
#include "common.cuh"

#include <mutex>

namespace moe {
namespace {

constexpr int DBM = 128;                   // weight rows per item (MMA M)
constexpr int DBK = 64;                    // 64 BF16 = one 128-byte swizzle row
constexpr int W_BYTES = DBM * DBK * 2;     // 16 KiB weight box
constexpr int DTHREADS = 192;              // producer, MMA, 4 epilogue warps
constexpr int CONV_WARPS = 8;              // FP8 / NVFP4: converter warps (6 .. 6 + CONV_WARPS - 1)
constexpr int DTHREADS_FP8 = 192 + 32 * CONV_WARPS;
constexpr int DBK8 = 128;                  // FP8 code box: 128 codes (128 B) of each weight row
constexpr int W8_BYTES = DBM * DBK8;       // 16 KiB FP8 / NVFP4 code box
constexpr int DBK4 = 256;                  // NVFP4 stage: 256 codes (128 B) of each weight row
constexpr int S4_BYTES = DBM * 16;         // NVFP4: the 16 block scales of 128 weight rows
constexpr int MAX_CSLOTS = 4;
constexpr int MAX_DSTAGES = 16;
constexpr int MAX_DSMEM = 222 * 1024;

struct DParams {
    const int32_t* offsets;
    int groups, rows_all;
    int a_rows;                 // rows of the activation matrix (bucket bounds are clamped to it)
    int K, nseg, a_seg_col, b_seg_row;
    int N, b_group_rows, up_off;
    void* out;
    long long ldo;
    int out_group_col;
    WsHeader* hdr;
    int gated;                  // 1: no work items when hdr->cap_exceeded (the layer's capacity verdict)
    int nb;                     // activation rows per chunk (MMA N): 16, 32, 48 or 64
    int stages, stage_bytes;
    uint32_t tmem_cols;         // two accumulators of (SwiGLU ? 2 : 1) * nb columns, power of two
    uint32_t x_off;             // activation box within a stage
    uint32_t w_off;             // first weight box within a stage
    // FP8 / NVFP4 weights
    const float* wscale;        // [weight rows] FP32 scale per weight row
    uint32_t a_col;             // TMEM column of the first converted-weight slot
    int conv_slots;             // converted-weight slots in TMEM (one chunk each)
    uint32_t s_off;             // NVFP4: first block-scale box within a stage
    // When the bucket bounds are known (moe_layer): 0 = after the programmatic
    // wait (any caller); 1 = at launch (the down projection: the dispatch that
    // wrote them finished before the up projection passed its own wait); 2 =
    // once the fused dispatch has published them (hdr->route_ready).  With 1
    // or 2 the weight loads of the first ring stages go out before the wait;
    // the activation loads, which read the predecessor's output, after it.
    int early;
    // BF16 weights: 64-column K chunks per stage, loaded as one box per operand
    // through (column in chunk, row, chunk) tensor maps; 0 = one chunk per stage
    // through plain 2-D maps (K not a whole number of chunks).
    int kc;
};

template <int MODE> struct OutOfD { using T = __nv_bfloat16; };
template <> struct OutOfD<kGemmF32> { using T = float; };

struct DCtl {
    unsigned long long full[MAX_DSTAGES];
    unsigned long long empty[MAX_DSTAGES];
    unsigned long long tfull[2];
    unsigned long long tempty[2];
    unsigned long long cfull[MAX_CSLOTS];      // FP8 / NVFP4: slot converted (the converter warps)
    unsigned long long cempty[MAX_CSLOTS];     // FP8 / NVFP4: slot consumed by the MMA
    unsigned long long drain;
    uint32_t tmem_base;
    int abort;
    int ng;                     // non-empty groups
    int wsum[DTHREADS_FP8 / 32];
};


// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x K, BF16) in TMEM, one row per lane
// and two consecutive K elements per 32-bit column (lower K in the low half).
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// 32 consecutive 32-bit columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
           "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int MODE, int WF>
__global__ void __launch_bounds__(WF != kWeightBf16 ? DTHREADS_FP8 : DTHREADS, 1)
decode_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmS, const DParams p) {
    constexpr bool FP8W = WF != kWeightBf16;               // converted weights (FP8 or NVFP4)
    constexpr bool FP4W = WF == kWeightNvfp4;
    constexpr int NW = (MODE == kGemmSwiGLU) ? 2 : 1;      // weight boxes per stage
    // K per stage: 64 (BF16), 256 (NVFP4; FP8 with one weight box), 128 (FP8
    // SwiGLU).  K per converted chunk: the whole stage when one weight box fills
    // a slot, else 128.  Code boxes (128 bytes per row) per weight block.
    constexpr int KSTEP = FP4W ? DBK4 : (FP8W ? (NW == 1 ? 256 : DBK8) : DBK);
    constexpr int CK = (FP8W && NW == 1) ? 256 : 128;
    constexpr int NCH = FP8W ? KSTEP / CK : 1;
    constexpr int SLOT_COLS = NW * CK / 2;
    constexpr int NB8 = FP8W && !FP4W ? KSTEP / DBK8 : 1;
    constexpr int NTH = FP8W ? DTHREADS_FP8 : DTHREADS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    // [TMA stage ring][control block][group lists]
    DCtl* ctl = reinterpret_cast<DCtl*>(smem + (size_t)p.stages * p.stage_bytes);
    int* gid = reinterpret_cast<int*>(ctl + 1);            // [groups] non-empty groups, in order
    int* gst = gid + p.groups;                              // first row
    int* gcnt = gst + p.groups;                             // rows
    const uint32_t smem_base = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- set-up: barriers, TMEM ----------------------------------------------
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), 4);        // the 4 epilogue warps
        }
        if (FP8W)
            for (int c = 0; c < p.conv_slots; ++c) {
                mbar_init(smem_u32(&ctl->cfull[c]), CONV_WARPS);
                mbar_init(smem_u32(&ctl->cempty[c]), 1);
            }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        if (FP4W) tma_prefetch_desc(&tmS);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), p.tmem_cols);
        tmem_relinquish();
    }
    __shared__ int early_ok;
    if (p.early == 2) {
        // the fused dispatch publishes the bucket bounds before it copies rows;
        // a bounded wait, after which the programmatic wait below is the fallback
        if (tid == 0) {
            const unsigned long long t0 = globaltimer_ns();
            unsigned ready;
            while ((ready = ld_acquire_u32(&p.hdr->route_ready)) == 0u && globaltimer_ns() - t0 < kEarlyWaitNs) { }
            early_ok = ready != 0u;
        }
        __syncthreads();
    }
    const bool waited = p.early == 0 || (p.early == 2 && !early_ok);
    if (waited) {
        pdl_wait();
        pdl_trigger();
    }
    // after a capacity overflow in the same layer call no payload moved: no items
    const bool skip = p.gated && __ldcg(&p.hdr->cap_exceeded);

    // ---- the non-empty groups (block-wide compaction of the offsets) --------
    if (skip) {
        if (tid == 0) ctl->ng = 0;
    } else if (p.offsets) {
        // each thread's groups g0 .. g0+per-1 (per <= 6: at most 1024 groups over
        // at least 192 threads): their per+1 bounds are read once, together, and
        // kept in registers for both passes
        constexpr int kMaxPer = 8;
        const int per = (p.groups + NTH - 1) / NTH;
        const int g0 = tid * per;
        int bnd[kMaxPer + 1];
#pragma unroll
        for (int i = 0; i <= kMaxPer; ++i) {
            const int g = g0 + i;
            int v = (i <= per && g <= p.groups) ? __ldcg(p.offsets + g) : 0;   // from L2: before the wait too
            bnd[i] = v < 0 ? 0 : (v > p.a_rows ? p.a_rows : v);
        }
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i)
            if (i < per && g0 + i < p.groups) cnt += bnd[i + 1] > bnd[i];
        int inc = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        if (lane == 31) ctl->wsum[warp] = inc;
        __syncthreads();
        int k = inc - cnt;
        for (int w = 0; w < warp; ++w) k += ctl->wsum[w];
        if (tid == NTH - 1) ctl->ng = k + cnt;
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i) {
            const int g = g0 + i;
            if (i < per && g < p.groups && bnd[i + 1] > bnd[i]) {
                gid[k] = g;
                gst[k] = bnd[i];
                gcnt[k] = bnd[i + 1] - bnd[i];
                ++k;
            }
        }
    } else {
        for (int g = tid; g < p.groups; g += NTH) {
            gid[g] = g;
            gst[g] = 0;
            gcnt[g] = p.rows_all < p.a_rows ? p.rows_all : p.a_rows;
        }
        if (tid == 0) ctl->ng = p.groups;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort = &ctl->abort;
    const int ntn = (p.N + DBM - 1) / DBM;
    const int items = ctl->ng * ntn;
    // the MMA takes a stage in 64-wide activation boxes; BF16 stages hold kcs
    // chunks of K (a TMA stage costs an SM about the same time for 16 as for
    // 64 KiB, so wide stages stream weights faster)
    const int kcs = (!FP8W && p.kc > 0) ? p.kc : 1;
    const int kstep = FP8W ? KSTEP : DBK * kcs;
    const int nkb = (p.K + kstep - 1) / kstep;
    const int nk = nkb * p.nseg;
    const uint32_t xbox = (uint32_t)(p.nb * DBK * 2);        // one activation box (nb rows x 64)
    const int nb = p.nb;
    const uint32_t acc_cols = (uint32_t)(NW * nb);
    const uint32_t x_off = p.x_off, w_off = p.w_off;
    const uint32_t w_box = FP8W ? (uint32_t)W8_BYTES : (uint32_t)W_BYTES;

    // The TMA loads of one ring stage: its weight boxes (with the NVFP4 block
    // scales), and its activation boxes.
    auto load_weights = [&](uint32_t sa, uint32_t full, int w_row, int seg, int kb) {
        if constexpr (!FP8W) {
            if (p.kc > 0) {      // kcs chunks of the weight rows in one box
                if (MODE == kGemmSwiGLU)   // gate rows, then up rows, per chunk
                    tma_load_5d(sa + w_off, &tmW, full, 0, w_row % p.b_group_rows, 0, w_row / p.b_group_rows,
                                kb * kcs);
                else
                    tma_load_3d(sa + w_off, &tmW, full, 0, w_row + seg * p.b_seg_row, kb * kcs);
                return;
            }
        }
        const int wcol = FP4W ? kb * (DBK4 / 2) : kb * kstep;     // code bytes
#pragma unroll
        for (int h = 0; h < NB8; ++h)   // FP8, 256-wide stage: two 128-byte code boxes
            tma_load_2d(sa + w_off + (uint32_t)h * w_box, &tmW, full, wcol + h * DBK8, w_row + seg * p.b_seg_row);
        if (MODE == kGemmSwiGLU)
            tma_load_2d(sa + w_off + w_box, &tmW, full, wcol, w_row + p.up_off + seg * p.b_seg_row);
        if (FP4W) {     // the rows' block scales of these 256 elements
            tma_load_2d(sa + p.s_off, &tmS, full, kb * (DBK4 / 16), w_row);
            if (MODE == kGemmSwiGLU)
                tma_load_2d(sa + p.s_off + S4_BYTES, &tmS, full, kb * (DBK4 / 16), w_row + p.up_off);
        }
    };
    auto load_acts = [&](uint32_t sa, uint32_t full, int xr, int seg, int kb) {
        if (!FP8W && p.kc > 0) {
            tma_load_3d(sa + x_off, &tmX, full, 0, xr, seg * (p.a_seg_col / DBK) + kb * kcs);
            return;
        }
        for (int xb = 0; xb < kstep / DBK; ++xb)   // 64-wide activation boxes
            tma_load_2d(sa + x_off + (uint32_t)xb * xbox, &tmX, full, seg * p.a_seg_col + kb * kstep + xb * DBK, xr);
    };

    // Bucket bounds known before the programmatic wait: the producer arms the
    // first ring stages and sends their weight loads (weights are never written
    // by a kernel) while the predecessor finishes; every thread then waits, and
    // the activation loads of those stages follow in the main loop.  Only about
    // 64 KiB of weights (four one-chunk stages, one four-chunk stage): the TMA
    // unit takes the requests in order, and a CTA that starts late would
    // otherwise queue its first activation loads behind a ring of weight loads
    // (measured at decode: four narrow stages beat a full ring by about 1 us per
    // layer, one wide stage beats three by about 0.7 us).
    constexpr int kPreStages = 4;
    const int npre_lim = (kPreStages + kcs - 1) / kcs;        // about 64 KiB of weights
    const int npre_max = p.stages < npre_lim ? p.stages : npre_lim;
    int npre = 0;
    if (!waited) {
        if (warp == 0 && lane == 0) {
            for (int it = blockIdx.x; it < items && npre < npre_max; it += gridDim.x) {
                const int slot = it / ntn, nt = it - slot * ntn;
                const int w_row = gid[slot] * p.b_group_rows + nt * DBM;
                for (int xr = gst[slot]; xr < gst[slot] + gcnt[slot] && npre < npre_max; xr += nb)
                    for (int i = 0; i < nk && npre < npre_max; ++i) {
                        const uint32_t full = smem_u32(&ctl->full[npre]);
                        mbar_arrive_expect_tx(full, (uint32_t)p.stage_bytes);
                        load_weights(smem_base + (uint32_t)(npre * p.stage_bytes), full, w_row, i / nkb, i % nkb);
                        ++npre;
                    }
            }
        }
        pdl_wait();
        pdl_trigger();
    }

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            long long armed = 0;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                const int slot = it / ntn, nt = it - slot * ntn;
                const int g = gid[slot], row0 = gst[slot], rows = gcnt[slot];
                const int w_row = g * p.b_group_rows + nt * DBM;
                for (int xr = row0; xr < row0 + rows && ok; xr += nb) {
                    for (int i = 0; i < nk; ++i) {
                        const int seg = i / nkb, kb = i - seg * nkb;
                        const uint32_t full = smem_u32(&ctl->full[stage]);
                        const uint32_t sa = smem_base + (uint32_t)(stage * p.stage_bytes);
                        if (armed >= npre) {      // else armed with its weights before the wait
                            if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort)) { ok = false; break; }
                            mbar_arrive_expect_tx(full, (uint32_t)p.stage_bytes);
                            load_weights(sa, full, w_row, seg, kb);
                        }
                        load_acts(sa, full, xr, seg, kb);
                        ++armed;
                        if (++stage == p.stages) { stage = 0; ph ^= 1u; }
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits (stages
                // armed before the wait whose activations never went out cannot
                // complete: their wait runs out and the fixed delay follows)
                if (!wait_armed_stages(smem_u32(&ctl->full[0]), p.stages, armed > npre ? armed : npre))
                    settle_delay();
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmDecode;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(DBM, nb);
            int stage = 0, acc = 0, cs = 0;
            uint32_t ph = 0, aph = 0, cph = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                const int rows = gcnt[it / ntn];
                for (int c0 = 0; c0 < rows && ok; c0 += nb) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)acc * acc_cols;
                    for (int i = 0; i < nk; ++i) {
                        if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), ph, abort)) { ok = false; break; }
                        const uint32_t sa = smem_base + (uint32_t)(stage * p.stage_bytes);
                        if constexpr (FP8W) {
                            // each chunk ch (CK wide) of the stage's weights, converted to
                            // BF16, is in a TMEM slot cs: weight block wb, K element k of
                            // the chunk at column a_col + cs*SLOT_COLS + wb*CK/2 + k/2; its
                            // activations are boxes ch*CK/64 .. +CK/64-1
                            for (int ch = 0; ch < NCH && ok; ++ch) {
                                if (!mbar_wait_bounded(smem_u32(&ctl->cfull[cs]), cph, abort)) { ok = false; break; }
                                tc_fence_after();
                                const uint32_t aslot = tmem + p.a_col + (uint32_t)(cs * SLOT_COLS);
#pragma unroll
                                for (int xb = 0; xb < CK / 64; ++xb) {
                                    const uint64_t xd =
                                        sdesc_k_sw128(sa + x_off + (uint32_t)(ch * (CK / 64) + xb) * xbox);
#pragma unroll
                                    for (int kk = 0; kk < DBK / 16; ++kk) {
                                        const uint32_t accum = (i > 0 || ch > 0 || xb > 0 || kk > 0) ? 1u : 0u;
                                        const uint32_t acol = (uint32_t)(xb * 32 + kk * 8);
                                        tc_mma_bf16_ts(d, aslot + acol, xd + (uint64_t)(kk * 2), idesc, accum);
                                        if (MODE == kGemmSwiGLU)
                                            tc_mma_bf16_ts(d + (uint32_t)nb, aslot + CK / 2 + acol,
                                                           xd + (uint64_t)(kk * 2), idesc, accum);
                                    }
                                }
                                tc_commit(smem_u32(&ctl->cempty[cs]));
                                if (++cs == p.conv_slots) { cs = 0; cph ^= 1u; }
                            }
                            if (!ok) break;
                        } else {
                            tc_fence_after();
                            // chunk c of the stage: weights at w_off + c * NW * 16 KiB (SwiGLU:
                            // gate, then up), activations at x_off + c * xbox; chunks past
                            // this segment's K (the last stage) are not multiplied
                            const int kb0 = (i - (i / nkb) * nkb) * kcs;
                            const int nch = p.K / DBK - kb0 < kcs ? p.K / DBK - kb0 : kcs;
                            for (int c = 0; c < kcs; ++c) {
                                if (c > 0 && c >= nch) break;
                                const uint64_t wd = sdesc_k_sw128(sa + w_off + (uint32_t)(c * NW * W_BYTES));
                                const uint64_t xd = sdesc_k_sw128(sa + x_off + (uint32_t)c * xbox);
#pragma unroll
                                for (int kk = 0; kk < DBK / 16; ++kk) {
                                    const uint32_t accum = (i > 0 || c > 0 || kk > 0) ? 1u : 0u;
                                    tc_mma_bf16(d, wd + (uint64_t)(kk * 2), xd + (uint64_t)(kk * 2), idesc, accum);
                                    if (MODE == kGemmSwiGLU)
                                        tc_mma_bf16(d + (uint32_t)nb,
                                                    sdesc_k_sw128(sa + w_off + (uint32_t)(c * NW * W_BYTES) + W_BYTES) +
                                                        (uint64_t)(kk * 2),
                                                    xd + (uint64_t)(kk * 2), idesc, accum);
                                }
                            }
                        }
                        tc_commit(smem_u32(&ctl->empty[stage]));
                        if (++stage == p.stages) { stage = 0; ph ^= 1u; }
                    }
                    if (!ok) break;
                    tc_commit(smem_u32(&ctl->tfull[acc]));
                    if (++acc == 2) { acc = 0; aph ^= 1u; }
                }
            }
            // drain: wait until every MMA this thread issued has completed
            tc_commit(smem_u32(&ctl->drain));
            volatile int never = 0;
            const bool drained = mbar_wait_bounded(smem_u32(&ctl->drain), 0, &never);
            if (!ok || !drained) {
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmDecode;
                *abort = 1;
            }
        }
    } else if (FP8W && warp >= 6) {
        // ---------------- FP8 / NVFP4 -> BF16 converter (warps 6 .. 6 + CONV_WARPS - 1)
        // A code box is 128 rows x 128 bytes, 128-byte swizzled (16-byte chunk c
        // of row r at chunk c ^ (r & 7)).  Converter warp w owns TMEM lane quarter
        // w % 4, i.e. weight rows r = 32*(w % 4) + lane, and K half hf = (w - 6) / 4
        // of every chunk: each thread decodes its row's CK/2 elements of that half
        // in 64-element sub-blocks (FP8: four conflict-free 16-byte loads each;
        // NVFP4: two, with the row's four block scales of the sub-block) and stores
        // each sub-block's 32 packed BF16 pairs to its TMEM lane, columns
        // a_col + cs*SLOT_COLS + wb*CK/2 + hf*CK/4 + 32*sub-block.
        const int q = warp & 3;
        const int hf = (warp - 6) >> 2;
        const int r = 32 * q + lane;
        const int sw = r & 7;
        int stage = 0, cs = 0;
        uint32_t ph = 0, cph = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            const int rows = gcnt[it / ntn];
            for (int c0 = 0; c0 < rows && ok; c0 += nb) {
                for (int i = 0; i < nk && ok; ++i) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), ph, abort)) { ok = false; break; }
                    const uint8_t* st = smem + (size_t)stage * p.stage_bytes;
                    const uint8_t* src = st + w_off + (size_t)r * DBK8;
                    uint4 scl[NW];                              // NVFP4: the row's 16 block scales, per box
                    if (FP4W)
#pragma unroll
                        for (int wb = 0; wb < NW; ++wb)
                            scl[wb] = *reinterpret_cast<const uint4*>(st + p.s_off + wb * S4_BYTES + r * 16);
                    for (int ch = 0; ch < NCH; ++ch) {
                        if (!mbar_wait_bounded(smem_u32(&ctl->cempty[cs]), cph ^ 1u, abort)) { ok = false; break; }
                        tc_fence_after();                       // after the MMAs that read slot cs
                        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + p.a_col +
                                               (uint32_t)(cs * SLOT_COLS) + (uint32_t)(hf * (CK / 4));
#pragma unroll
                        for (int wb = 0; wb < NW; ++wb) {
#pragma unroll
                            for (int sb = 0; sb < CK / 128; ++sb) {   // 64-element sub-blocks of this half
                                uint32_t v32[32];
                                if constexpr (FP4W) {
                                    const int e0 = ch * CK + hf * (CK / 2) + sb * 64;    // within the stage
                                    const int wi = e0 >> 6;                               // its 4 block scales
                                    const uint32_t s4 = wi == 0 ? scl[wb].x : wi == 1 ? scl[wb].y
                                                      : wi == 2 ? scl[wb].z : scl[wb].w;
                                    constexpr uint32_t kTwo118 = 0x7A807A80u;     // (2^118, 2^118) in BF16
                                    uint32_t s01, s23, mb[4];
                                    e4m3x4_to_bf16x4(s4, s01, s23);
                                    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(s01) : "r"(s01), "r"(kTwo118));
                                    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(s23) : "r"(s23), "r"(kTwo118));
                                    asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(mb[0]) : "r"(s01));
                                    asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(mb[1]) : "r"(s01));
                                    asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(mb[2]) : "r"(s23));
                                    asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(mb[3]) : "r"(s23));
#pragma unroll
                                    for (int j = 0; j < 2; ++j) {
                                        const uint4 v = *reinterpret_cast<const uint4*>(
                                            src + wb * W8_BYTES + ((((e0 >> 5) + j) ^ sw) << 4));
                                        e2m1x8_to_bf16x8(v.x, mb[2 * j], &v32[16 * j + 0]);
                                        e2m1x8_to_bf16x8(v.y, mb[2 * j], &v32[16 * j + 4]);
                                        e2m1x8_to_bf16x8(v.z, mb[2 * j + 1], &v32[16 * j + 8]);
                                        e2m1x8_to_bf16x8(v.w, mb[2 * j + 1], &v32[16 * j + 12]);
                                    }
                                } else {
                                    const int e0 = ch * CK + hf * (CK / 2) + sb * 64;    // byte in the stage row
                                    const uint8_t* bsrc = src + (wb * NB8 + (e0 >> 7)) * W8_BYTES;
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        const uint4 v = *reinterpret_cast<const uint4*>(
                                            bsrc + (((((e0 & 127) >> 4) + j) ^ sw) << 4));
                                        e4m3x4_to_bf16x4(v.x, v32[8 * j + 0], v32[8 * j + 1]);
                                        e4m3x4_to_bf16x4(v.y, v32[8 * j + 2], v32[8 * j + 3]);
                                        e4m3x4_to_bf16x4(v.z, v32[8 * j + 4], v32[8 * j + 5]);
                                        e4m3x4_to_bf16x4(v.w, v32[8 * j + 6], v32[8 * j + 7]);
                                    }
                                }
                                tmem_st_32cols(taddr + (uint32_t)(wb * (CK / 2) + sb * 32), v32);
                            }
                        }
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&ctl->cfull[cs]));
                        if (++cs == p.conv_slots) { cs = 0; cph ^= 1u; }
                    }
                    if (++stage == p.stages) { stage = 0; ph ^= 1u; }
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;                                 // TMEM lane quarter
        int acc = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            const int slot = it / ntn, nt = it - slot * ntn;
            const int g = gid[slot], row0 = gst[slot], rows = gcnt[slot];
            const int n = nt * DBM + 32 * q + lane;             // weight row = output column
            typename OutOfD<MODE>::T* ocol = reinterpret_cast<typename OutOfD<MODE>::T*>(p.out) +
                                             (size_t)g * p.out_group_col + (n < p.N ? n : 0);
            // FP8 / NVFP4: the weight rows' FP32 scales (gate and up rows for
            // SwiGLU); NVFP4 weights were converted at 2^-8 of their value
            float sg = 1.f, su = 1.f;
            if (FP8W && n < p.N) {
                constexpr float kUndo = FP4W ? 256.f : 1.f;
                sg = p.wscale[(size_t)g * p.b_group_rows + n] * kUndo;
                if (MODE == kGemmSwiGLU) su = p.wscale[(size_t)g * p.b_group_rows + p.up_off + n] * kUndo;
            }
            for (int c0 = 0; c0 < rows; c0 += nb) {
                if (!mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort)) {
                    if (lane == 0) {
                        raise_status(p.hdr, MOE_ERR_TIMEOUT);
                        p.hdr->timeout_site = kSiteGemmDecode;
                    }
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + (uint32_t)acc * acc_cols + ((uint32_t)(32 * q) << 16);
                for (int c = 0; c < nb; c += 16) {
                    uint32_t gv[16], uv[16];
                    tmem_ld_16cols(taddr + (uint32_t)c, gv);
                    if (MODE == kGemmSwiGLU) tmem_ld_16cols(taddr + (uint32_t)(nb + c), uv);
                    tmem_ld_wait();
                    if (n < p.N) {
#pragma unroll
                        for (int r = 0; r < 16; ++r) {
                            const int row = c0 + c + r;
                            if (row < rows) {
                                const float x = FP8W ? __uint_as_float(gv[r]) * sg : __uint_as_float(gv[r]);
                                auto* o = ocol + (size_t)(row0 + row) * p.ldo;
                                if constexpr (MODE == kGemmF32) {
                                    *o = x;
                                } else {
                                    float a;
                                    if (MODE == kGemmSwiGLU)
                                        a = x / (1.0f + __expf(-x)) *
                                            (FP8W ? __uint_as_float(uv[r]) * su : __uint_as_float(uv[r]));
                                    else if (MODE == kGemmReLU2) a = x > 0.f ? x * x : 0.f;
                                    else a = x;
                                    *o = __float2bfloat16_rn(a);
                                }
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
                if (++acc == 2) { acc = 0; aph ^= 1u; }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

template <int MODE, int WF>
cudaError_t launch_d(const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& ms, const DParams& dp,
                     unsigned grid, size_t smem, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(decode_gemm_kernel<MODE, WF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        MAX_DSMEM);
    });
    if (attr_err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(decode GEMM, %d bytes): %s", MAX_DSMEM, cudaGetErrorString(attr_err));
        return attr_err;
    }
    const cudaError_t e =
        launch_kernel(decode_gemm_kernel<MODE, WF>, dim3(grid), dim3(WF != kWeightBf16 ? DTHREADS_FP8 : DTHREADS),
                      smem, st, 1, kUsePdl, mx, mw, ms, dp);
    if (e != cudaSuccess) set_error("decode GEMM launch: %s", cudaGetErrorString(e));
    return e;
}

}  // namespace

moe_status launch_decode_gemm(const GemmProblem& g, int nb, WsHeader* hdr, cudaStream_t st) {
    if (g.groups > 192 * 8) {       // the kernel's group list: at most 8 groups per thread
        set_error("decode GEMM: %d groups", g.groups);
        return MOE_ERR_UNSUPPORTED;
    }
    if (nb < 16 || nb > kDecodeRows || nb % 16 != 0) {
        set_error("decode GEMM: %d rows per chunk is not a multiple of 16 in [16, %d]", nb, kDecodeRows);
        return MOE_ERR_INTERNAL;
    }
    const int nw = g.mode == kGemmSwiGLU ? 2 : 1;
    const bool fp4 = g.wfmt == kWeightNvfp4;
    const bool fp8 = g.wfmt == kWeightFp8E4M3 || fp4;      // converted weights
    if (fp8 && (g.mode == kGemmF32 || !g.wscale)) {
        set_error("decode GEMM: quantized weights need a scale per weight row and a BF16 output");
        return MOE_ERR_UNSUPPORTED;
    }
    if (fp4 && (!g.bscale || g.K % 32 != 0 || g.bscale_stride % 16 != 0 || g.bscale_stride * 16 < g.K)) {
        set_error("decode GEMM: NVFP4 weights need K %% 32 == 0 and block-scale rows of 16-byte multiples");
        return MOE_ERR_UNSUPPORTED;
    }
    DParams dp;
    dp.offsets = g.offsets;
    dp.groups = g.groups;
    dp.rows_all = g.rows_all;
    dp.a_rows = (int)g.a_rows;
    dp.K = g.K;
    dp.nseg = g.nseg;
    dp.a_seg_col = g.a_seg_col;
    dp.b_seg_row = g.b_seg_row;
    dp.N = g.N;
    dp.b_group_rows = g.b_group_rows;
    dp.up_off = g.up_off;
    dp.out = g.out;
    dp.ldo = g.ldo;
    dp.out_group_col = g.out_group_col;
    dp.hdr = hdr;
    dp.gated = g.gated;
    dp.nb = nb;
    dp.wscale = g.wscale;
    dp.s_off = 0;
    dp.early = g.offsets ? g.early : 0;
    dp.kc = 0;
    if (fp4) {
        // stage (K 256): [four activation boxes: nb rows x 128 B each][code box(es):
        // 128 rows x 128 B = 16 KiB each][block-scale box(es): 128 rows x 16 B]
        dp.x_off = 0;
        dp.w_off = (uint32_t)(4 * nb * DBK * 2);
        dp.s_off = dp.w_off + (uint32_t)(nw * W8_BYTES);
        dp.stage_bytes = (int)dp.s_off + nw * S4_BYTES;
        // one weight box: whole-stage chunks of 128 columns after at most 128
        // accumulator columns (3 slots); SwiGLU: 128-wide chunks, 2 slots
        dp.a_col = nw == 1 ? 128 : 256;
        dp.conv_slots = nw == 1 ? 3 : 2;
    } else if (fp8) {
        // stage: one weight box: K 256 = [four activation boxes][two code boxes:
        // K 0..127 and 128..255 of the 128 rows]; SwiGLU: K 128 = [two activation
        // boxes][gate and up code boxes].  Boxes of codes are 128 rows x 128 B.
        const int xboxes = nw == 1 ? 4 : 2;
        dp.x_off = 0;
        dp.w_off = (uint32_t)(xboxes * nb * DBK * 2);
        dp.stage_bytes = xboxes * nb * DBK * 2 + 2 * W8_BYTES;
        // TMEM: one weight box: accumulators in columns 0..127, three 128-column
        // slots; SwiGLU: accumulators in 0..255, two slots of 2 x 64 columns
        dp.a_col = nw == 1 ? 128 : 256;
        dp.conv_slots = nw == 1 ? 3 : 2;
    } else {
        // stage: [kc chunks of the weight rows: nw x 16 KiB each][kc activation
        // boxes: nb rows x 128 B each], kc as large as leaves three stages (at
        // most four chunks); one chunk through 2-D maps when K is ragged
        const size_t fixed0 = 1024 + sizeof(DCtl) + (size_t)3 * g.groups * sizeof(int);
        const bool chunked = g.K % DBK == 0 && g.a_cols % DBK == 0 && g.b_cols % DBK == 0 && g.a_seg_col % DBK == 0 &&
                             (g.mode != kGemmSwiGLU || (g.nseg == 1 && g.b_group_rows == 2 * g.up_off));
        int kc = 1;
        if (chunked)
            for (kc = 4; kc > 1; --kc)
                if (fixed0 + 3 * (size_t)kc * (nw * W_BYTES + nb * DBK * 2) <= (size_t)MAX_DSMEM) break;
        dp.kc = chunked ? kc : 0;
        dp.w_off = 0;
        dp.x_off = (uint32_t)(kc * nw * W_BYTES);
        dp.stage_bytes = kc * (nw * W_BYTES + nb * DBK * 2);
        dp.conv_slots = 0;
        dp.a_col = 0;
    }
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * nw * nb)) cols <<= 1;
    dp.tmem_cols = fp8 ? 512u : cols;

    // items: (non-empty group) x (128-row weight block); at most one CTA per SM
    const long long ntn = (g.N + DBM - 1) / DBM;
    const long long slots = g.offsets ? (g.a_rows < g.groups ? g.a_rows : g.groups) : g.groups;
    long long grid = slots * ntn;
    const int sms = device_sm_count();
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    const size_t fixed = 1024 + sizeof(DCtl) + (size_t)3 * g.groups * sizeof(int);
    const int kstep = fp4 ? DBK4 : (fp8 ? (nw == 1 ? 256 : DBK8) : DBK * (dp.kc > 0 ? dp.kc : 1));
    const int nk = ((g.K + kstep - 1) / kstep) * g.nseg;
    long long stages = ((long long)MAX_DSMEM - (long long)fixed) / dp.stage_bytes;
    if (stages > MAX_DSTAGES) stages = MAX_DSTAGES;
    // two items' worth is plenty; FP8 (512 TMEM columns) keeps a full ring so
    // that one CTA holds an SM
    if (!fp8 && stages > 2 * nk) stages = 2 * nk;
    if (stages < 2) stages = 2;
    dp.stages = (int)stages;
    const size_t smem = fixed + (size_t)stages * dp.stage_bytes;
    if (smem > (size_t)MAX_DSMEM) {
        set_error("decode GEMM needs %zu bytes of shared memory", smem);
        return MOE_ERR_UNSUPPORTED;
    }
    CUtensorMap mx, mw, ms;
    if (dp.kc > 0) {
        if (!make_tensor_map_bf16_chunks(&mx, g.a, g.a_rows, g.a_cols, (unsigned)nb, (unsigned)dp.kc) ||
            (g.mode == kGemmSwiGLU
                 ? !make_tensor_map_glu_chunks(&mw, g.b, g.b_rows, g.b_cols, g.up_off, g.b_group_rows,
                                               (unsigned)DBM, (unsigned)dp.kc)
                 : !make_tensor_map_bf16_chunks(&mw, g.b, g.b_rows, g.b_cols, (unsigned)DBM, (unsigned)dp.kc)))
            return MOE_ERR_CUDA;
    } else if (!make_tensor_map_bf16(&mx, g.a, g.a_rows, g.a_cols, (unsigned)nb)) {
        return MOE_ERR_CUDA;
    }
    // code rows: K bytes (FP8) or K/2 bytes (NVFP4, two codes per byte)
    const long long code_cols = fp4 ? g.b_cols / 2 : g.b_cols;
    if (fp8 ? !make_tensor_map_u8_rows(&mw, g.b, g.b_rows, code_cols, code_cols, (unsigned)DBK8, (unsigned)DBM)
            : (dp.kc == 0 && !make_tensor_map_bf16(&mw, g.b, g.b_rows, g.b_cols, (unsigned)DBM)))
        return MOE_ERR_CUDA;
    if (fp4) {
        // block scales: K/16 bytes of each padded row, 16 per stage
        if (!make_tensor_map_u8_rows(&ms, g.bscale, g.b_rows, g.b_cols / 16, g.bscale_stride, 16u, (unsigned)DBM))
            return MOE_ERR_CUDA;
    } else {
        ms = mw;   // unused
    }
    cudaError_t e;
    if (fp4) {
        switch (g.mode) {
            case kGemmSwiGLU: e = launch_d<kGemmSwiGLU, kWeightNvfp4>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
            case kGemmReLU2: e = launch_d<kGemmReLU2, kWeightNvfp4>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
            default: e = launch_d<kGemmPlain, kWeightNvfp4>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
        }
    } else if (fp8) {
        switch (g.mode) {
            case kGemmSwiGLU: e = launch_d<kGemmSwiGLU, kWeightFp8E4M3>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
            case kGemmReLU2: e = launch_d<kGemmReLU2, kWeightFp8E4M3>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
            default: e = launch_d<kGemmPlain, kWeightFp8E4M3>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
        }
    } else {
        switch (g.mode) {
            case kGemmSwiGLU: e = launch_d<kGemmSwiGLU, kWeightBf16>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
            case kGemmReLU2: e = launch_d<kGemmReLU2, kWeightBf16>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
            case kGemmF32: e = launch_d<kGemmF32, kWeightBf16>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
            default: e = launch_d<kGemmPlain, kWeightBf16>(mx, mw, ms, dp, (unsigned)grid, smem, st); break;
        }
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
