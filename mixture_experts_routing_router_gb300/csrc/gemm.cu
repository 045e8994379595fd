// gemm.cu -- K4 / K5 / K7: the grouped expert GEMM on tcgen05 tensor cores.
//
// DeepSeek fleet REPORT.md (EXPERT_W13_SILU and EXPERT_W2 rows of the per-op
// table) and ONNX Runtime PR #33963 (Description: SwiGLU default, ReLU-square
// experts, BF16 store boundaries with FP32 accumulation).
//
// One persistent CTA per SM walks a tile list built on the device from the
// bucket bounds (offsets): group g (an expert) owns ceil(m_g / BMT) row tiles
// times ceil(N / BN) column tiles.  The counts never travel to the host, so
// the layer stays capturable in a CUDA graph.
//
// Roles:
//   warp 0     one thread issues TMA loads (128-byte swizzle, 64-column K
//              boxes) of the A rows and the 256-row B tile into a ring of
//              shared-memory stages;
//   warp 1     allocates all 512 TMEM columns; one thread issues tcgen05.mma
//              (M 128, N 256, K 16) per 16-wide K slice, committing each stage
//              back to the producer and each finished tile to the epilogue;
//   warps 2..  read the accumulator with tcgen05.ld (one TMEM lane = one row
//              per thread), apply the activation, round to BF16 and store,
//              masking rows past the bucket end and columns past N.
// Three tile shapes, chosen per launch:
//   * CTA pair (groups averaging >= 256 rows, e.g. the large layer's experts):
//     two SMs share a 256-row tile through tcgen05.mma.cta_group::2, each
//     loading its own A rows and half of B; a group's partial last tile runs
//     with the operands swapped -- see grouped_gemm_pair_kernel.
// Groups of at most a few dozen rows (decode) run the small-row kernel in
// gemm_decode.cu when its work fits in about two waves.
//   * single CTA, HALVES = 1 (fewer rows per group, K < 4096): 128-row tiles,
//     two 256-column accumulators in TMEM so the epilogue of one tile overlaps
//     the main loop of the next; 4 stages of 48 KiB; 4 epilogue warps.
//   * single CTA, HALVES = 2 (fewer rows per group, K >= 4096): 256-row tiles as
//     two 128-row halves sharing every B tile (two MMAs per K slice into the two
//     accumulators), which cuts the operand traffic per FLOP by a third; a tail
//     whose second half is empty loads and multiplies only the first.  3 stages
//     of 64 KiB; the epilogue (8 warps, one half each) is not overlapped.
// A 128-row accumulator with 64 rows or fewer in its tile uses M = 64 MMAs.
// In the single-CTA shapes a SwiGLU B tile is 128 gate rows and the matching
// 128 up rows, so gate and up land side by side in one accumulator and the
// epilogue computes silu(g) * u without a second pass (the pair kernel splits
// them as two [64 gate | 64 up] halves, one per CTA).
//
// Every wait is bounded; on a timeout the CTA stops issuing work, drains its
// in-flight tensor-core work, frees TMEM, raises MOE_ERR_TIMEOUT and returns.
#include "common.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace moe {
namespace {

constexpr int BM = 128;                      // rows per MMA / per accumulator
constexpr int BK = 64;                       // 64 BF16 = 128 B: one swizzle row
constexpr int BN_MMA = 256;
constexpr int A_BYTES = BM * BK * 2;         // 16 KiB
constexpr int B_HALF_BYTES = 128 * BK * 2;   // 16 KiB
constexpr int B_BYTES = BN_MMA * BK * 2;     // 32 KiB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN_MMA);
// A 128-row accumulator whose rows of this tile number 64 or fewer is computed
// with M = 64 MMAs (half the tensor work).  Their D rows sit in TMEM lanes
// 32q + i, i < 16, for row 16q + i (q = lane quarter).
constexpr uint32_t IDESC64 = idesc_bf16_f32(64, BN_MMA);
constexpr int kTailRows = 64;
// Dynamic shared memory ceiling set on the kernels: the stage ring plus the
// control block and the per-group tables of up to 1024 groups.  It stays below
// the 227 KiB opt-in limit minus the kernel's small static shared memory.
constexpr int MAX_DYN_SMEM = 216 * 1024;
// Reductions at least this long use the 256-row tile (HALVES = 2).
constexpr long long kLongK = 4096;
// Groups averaging at least this many rows use the CTA-pair kernel (compute
// bound: the halved operand traffic pays); fewer rows per group -- weight
// streaming at decode or at a few hundred tokens -- use the single-CTA shapes.
constexpr long long kPairRows = 256;

template <int HALVES>
struct Cfg {
    static constexpr int STAGES = HALVES == 1 ? 4 : 3;
    static constexpr int STAGE_BYTES = HALVES * A_BYTES + B_BYTES;   // 48 / 64 KiB
    static constexpr int NUM_ACC = HALVES == 1 ? 2 : 1;             // accumulator buffers
    static constexpr int EPI_WARPS = 4 * HALVES;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;             // 192 / 320
    static constexpr int BMT = BM * HALVES;                         // rows per tile
};

struct KParams {
    const int32_t* offsets;
    int groups, rows_all;
    int a_rows;                 // rows of A (bucket bounds are clamped to it)
    int K, nseg, a_seg_col, b_seg_row;
    int N, b_group_rows, up_off;
    void* out;                  // BF16, or FP32 for kGemmF32
    long long ldo;
    int out_group_col;
    WsHeader* hdr;
    int gated;                  // 1: no tiles when hdr->cap_exceeded (the layer's capacity verdict)
};

template <int HALVES>
struct SmemCtl {
    unsigned long long full[Cfg<HALVES>::STAGES];
    unsigned long long empty[Cfg<HALVES>::STAGES];
    unsigned long long tfull[Cfg<HALVES>::NUM_ACC];
    unsigned long long tempty[Cfg<HALVES>::NUM_ACC];
    unsigned long long drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// The four epilogue warps of a CTA (named barrier 1; __syncthreads uses 0).
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct Tile { int g, mt, nt, row0, mrows; };

// Tile order inside a group: bands of kRasterBand column tiles.  The up
// projection (long rows of A: K = hidden) walks the band's column tiles first,
// so the tiles running at the same time share a few A row blocks and each A
// row block is read from DRAM about once per band; the down projection (short
// A rows, wide N) walks row tiles first inside the band so a few weight tiles
// serve many row tiles.  Both orders measured faster than a plain row-major
// walk on the Zipf-skewed large layer.
constexpr int kRasterBand = 8;

// Group = largest g with prefix[g] <= tile (empty groups share their prefix value).
template <bool COLS_FIRST>
__device__ __forceinline__ Tile decode_tile(int tile, const int* prefix, const int* rstart, const int* rcount,
                                            const KParams& p, int ntn, int bmt) {
    int lo = 0, hi = p.groups;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= tile) lo = mid; else hi = mid;
    }
    Tile t;
    t.g = lo;
    const int local = tile - prefix[lo];
    const int mtiles = (rcount[lo] + bmt - 1) / bmt;
    const int band = local / (mtiles * kRasterBand);
    const int idx = local - band * mtiles * kRasterBand;
    if (COLS_FIRST) {
        const int nb = min(kRasterBand, ntn - band * kRasterBand);
        t.mt = idx / nb;
        t.nt = band * kRasterBand + idx % nb;
    } else {
        t.mt = idx % mtiles;
        t.nt = band * kRasterBand + idx / mtiles;
    }
    t.row0 = rstart[lo];
    t.mrows = rcount[lo];
    return t;
}

template <int MODE> struct OutOf { using T = __nv_bfloat16; };
template <> struct OutOf<kGemmF32> { using T = float; };

// Output row pointer of row `row` of group g (a valid row index is passed even
// for masked rows, so no pointer past the buffer is ever formed).
template <int MODE>
__device__ __forceinline__ typename OutOf<MODE>::T* out_row(const KParams& p, int row, int g) {
    return reinterpret_cast<typename OutOf<MODE>::T*>(p.out) + (size_t)row * p.ldo + (size_t)g * p.out_group_col;
}

// One 32-column chunk of the epilogue for this thread's row: read the
// accumulator columns at `tg` (and the matching up columns at `tu` for SwiGLU),
// apply the activation, round to BF16 and store output columns col0..col0+31
// (whole 16-byte groups below N; N is a multiple of 8).
template <int MODE>
__device__ __forceinline__ void epilogue_chunk(uint32_t tg, uint32_t tu, bool row_ok, typename OutOf<MODE>::T* orow,
                                               int col0, int N) {
    uint32_t gv[32], uv[32];
    tmem_ld_32cols(tg, gv);
    if (MODE == kGemmSwiGLU) tmem_ld_32cols(tu, uv);
    tmem_ld_wait();
    if (!row_ok) return;
    if constexpr (MODE == kGemmF32) {
        // FP32 accumulator as is: 16-byte stores where the row and N allow
        float* o = orow;
        const bool vec = ((reinterpret_cast<uintptr_t>(o) & 15u) == 0) && (N % 4 == 0);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const int c = col0 + v * 4;
            if (vec) {
                if (c < N)
                    *reinterpret_cast<float4*>(o + c) =
                        make_float4(__uint_as_float(gv[4 * v]), __uint_as_float(gv[4 * v + 1]),
                                    __uint_as_float(gv[4 * v + 2]), __uint_as_float(gv[4 * v + 3]));
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (c + i < N) o[c + i] = __uint_as_float(gv[4 * v + i]);
            }
        }
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            if (col0 + v * 8 < N) {
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float a[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float x = __uint_as_float(gv[v * 8 + 2 * i + h]);
                        if (MODE == kGemmSwiGLU) {
                            const float u = __uint_as_float(uv[v * 8 + 2 * i + h]);
                            a[h] = x / (1.0f + __expf(-x)) * u;
                        } else if (MODE == kGemmReLU2) {
                            a[h] = x > 0.f ? x * x : 0.f;
                        } else {
                            a[h] = x;
                        }
                    }
                    o[i] = pack2(a[0], a[1]);
                }
                *reinterpret_cast<uint4*>(orow + col0 + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// Epilogue of one 128-row accumulator of the single-CTA kernel: this warp's 32
// TMEM lanes at `tbase`, one row per thread.  SwiGLU accumulators hold 128 gate
// columns then the 128 matching up columns.
template <int MODE>
__device__ __forceinline__ void epilogue_rows(uint32_t tbase, bool row_ok, typename OutOf<MODE>::T* orow,
                                              int col_base, int N) {
    if (MODE == kGemmSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c)
            epilogue_chunk<MODE>(tbase + c * 32, tbase + 128 + c * 32, row_ok, orow, col_base + c * 32, N);
    } else {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) epilogue_chunk<MODE>(tbase + c * 32, 0, row_ok, orow, col_base + c * 32, N);
    }
}

template <int MODE, int HALVES>
__global__ void __launch_bounds__(Cfg<HALVES>::THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const KParams p) {
    using C = Cfg<HALVES>;
    constexpr int BN_OUT = (MODE == kGemmSwiGLU) ? 128 : 256;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB alignment for the 128-byte swizzle atoms
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    SmemCtl<HALVES>* ctl = reinterpret_cast<SmemCtl<HALVES>*>(smem + C::STAGES * C::STAGE_BYTES);
    int* prefix = reinterpret_cast<int*>(ctl + 1);          // [groups + 1] tiles before group g
    int* rstart = prefix + (p.groups + 1);                  // [groups] first row of group g
    int* rcount = rstart + p.groups;                        // [groups] rows of group g
    const uint32_t smem_base = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntn = (p.N + BN_OUT - 1) / BN_OUT;

    // ---- set-up: barriers, TMEM, tile prefix -------------------------------
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < C::NUM_ACC; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), C::EPI_WARPS);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    // After a capacity overflow in the same layer call no payload moved: leave
    // the outputs alone (no tiles).
    const bool skip = p.gated && p.hdr->cap_exceeded;
    // Group rows.  Each bucket is clamped to [0, a_rows] on its own, so even
    // malformed offsets keep every row access inside A and the output.
    for (int g = tid; g < p.groups; g += C::THREADS) {
        if (skip) {
            rstart[g] = 0;
            rcount[g] = 0;
        } else if (p.offsets) {
            int lo = p.offsets[g], hi = p.offsets[g + 1];
            lo = lo < 0 ? 0 : (lo > p.a_rows ? p.a_rows : lo);
            hi = hi < lo ? lo : (hi > p.a_rows ? p.a_rows : hi);
            rstart[g] = lo;
            rcount[g] = hi - lo;
        } else {
            rstart[g] = 0;
            rcount[g] = p.rows_all;
        }
    }
    __syncthreads();
    // exclusive scan of tiles per group -> prefix[0..groups]
    {
        const int n = p.groups;
        const int per = (n + C::THREADS - 1) / C::THREADS;
        const int g0 = tid * per;
        int loc = 0;
        for (int i = 0; i < per; ++i)
            if (g0 + i < n) loc += ((rcount[g0 + i] + C::BMT - 1) / C::BMT) * ntn;
        int inc = loc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        __shared__ int wtot[C::THREADS / 32];
        if (lane == 31) wtot[warp] = inc;
        __syncthreads();
        int run = inc - loc;
        for (int w = 0; w < warp; ++w) run += wtot[w];
        for (int i = 0; i < per; ++i) {
            if (g0 + i < n) {
                prefix[g0 + i] = run;
                run += ((rcount[g0 + i] + C::BMT - 1) / C::BMT) * ntn;
            }
        }
        if (tid == C::THREADS - 1) { prefix[n] = run; ctl->total_tiles = run; }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int total = ctl->total_tiles;
    volatile int* abort = &ctl->abort;
    const int nkb = (p.K + BK - 1) / BK;
    const int nk = nkb * p.nseg;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            long long armed = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p, ntn, C::BMT);
                const int a_row = t.row0 + t.mt * C::BMT;
                const bool second = HALVES == 2 && (t.mt * C::BMT + BM < t.mrows);
                const uint32_t bytes = (second ? 2 : 1) * A_BYTES + B_BYTES;
                const int n0 = t.nt * BN_OUT;
                const int b_lo = t.g * p.b_group_rows + n0;
                const int b_hi = (MODE == kGemmSwiGLU) ? b_lo + p.up_off : b_lo + 128;
                for (int i = 0; i < nk; ++i) {
                    const int seg = i / nkb, kb = i - seg * nkb;
                    if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort)) { ok = false; break; }
                    const uint32_t full = smem_u32(&ctl->full[stage]);
                    const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + HALVES * A_BYTES;
                    const int ax = seg * p.a_seg_col + kb * BK;
                    mbar_arrive_expect_tx(full, bytes);
                    tma_load_2d(sa, &tmA, full, ax, a_row);
                    if (second) tma_load_2d(sa + A_BYTES, &tmA, full, ax, a_row + BM);
                    tma_load_2d(sb, &tmB, full, kb * BK, b_lo + seg * p.b_seg_row);
                    tma_load_2d(sb + B_HALF_BYTES, &tmB, full, kb * BK, b_hi + seg * p.b_seg_row);
                    ++armed;
                    if (++stage == C::STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                if (!wait_armed_stages(smem_u32(&ctl->full[0]), C::STAGES, armed)) settle_delay();
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmProducer;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p, ntn, C::BMT);
                const int rows0 = t.mrows - t.mt * C::BMT;                  // rows from the first half on
                const bool second = HALVES == 2 && rows0 > BM;
                const uint32_t idesc0 = rows0 <= kTailRows ? IDESC64 : IDESC;
                const uint32_t idesc1 = rows0 - BM <= kTailRows ? IDESC64 : IDESC;
                if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)(acc * BN_MMA);
                for (int i = 0; i < nk; ++i) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), ph, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                    const uint64_t bd = sdesc_k_sw128(sa + HALVES * A_BYTES);
                    const uint64_t ad0 = sdesc_k_sw128(sa);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)   // +32 B along K inside the swizzle row
                        tc_mma_bf16(d0, ad0 + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc0,
                                    (i > 0 || kk > 0) ? 1u : 0u);
                    if (HALVES == 2 && second) {
                        const uint64_t ad1 = sdesc_k_sw128(sa + A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            tc_mma_bf16(d0 + BN_MMA, ad1 + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc1,
                                        (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&ctl->empty[stage]));
                    if (++stage == C::STAGES) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit(smem_u32(&ctl->tfull[acc]));
                if (++acc == C::NUM_ACC) { acc = 0; aph ^= 1u; }
            }
            // drain: wait until every MMA this thread issued has completed
            tc_commit(smem_u32(&ctl->drain));
            volatile int never = 0;
            const bool drained = mbar_wait_bounded(smem_u32(&ctl->drain), 0, &never);
            if (!ok || !drained) {
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmMma;
                *abort = 1;
            }
        }
    } else {
        // ---------------- epilogue (warps 2 .. 2 + EPI_WARPS - 1) ----------------
        const int q = warp & 3;                                   // TMEM lane quarter of this warp
        const int half = (HALVES == 2) ? (warp - 2) >> 2 : 0;     // which 128-row half
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p, ntn, C::BMT);
            if (!mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort)) {
                if (lane == 0) {
                    raise_status(p.hdr, MOE_ERR_TIMEOUT);
                    p.hdr->timeout_site = kSiteGemmEpilogue;
                }
                break;
            }
            tc_fence_after();
            const int hrow0 = t.mt * C::BMT + half * BM;                  // first row of this half
            const bool half_live = hrow0 < t.mrows;                       // warp-uniform
            if (half_live) {
                // M = 64 halves keep row 16q + i in lane 32q + i (i < 16)
                const bool m64 = t.mrows - hrow0 <= kTailRows;
                const int r = m64 ? hrow0 + q * 16 + lane : hrow0 + q * 32 + lane;
                const bool row_ok = (!m64 || lane < 16) && r < t.mrows;
                auto* orow = out_row<MODE>(p, t.row0 + (row_ok ? r : 0), t.g);
                const uint32_t tbase =
                    tmem_base + (uint32_t)((acc + half) * BN_MMA) + ((uint32_t)(q * 32) << 16);
                epilogue_rows<MODE>(tbase, row_ok, orow, t.nt * BN_OUT, p.N);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
            if (++acc == C::NUM_ACC) { acc = 0; aph ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// The CTA-pair shape.  A cluster of two CTAs (two SMs) owns a 256-row tile:
// each CTA TMA-loads its own 128 A rows and its half of the 256-row B tile
// (for SwiGLU, 64 gate rows and the matching 64 up rows per CTA), so a CTA
// moves 32 KiB per 64-wide K step instead of 48, and six stages fit.  The
// leader CTA's MMA thread issues tcgen05.mma.cta_group::2 (M 256, N 256)
// reading both CTAs' shared memory and writing both CTAs' TMEM; its commits
// arrive on the same barrier offsets in both CTAs.  A group's partial last
// tile swaps the operands (weights M 256, rows N = rows padded to 16).  Each CTA keeps two 256-column accumulators, so the epilogue of
// one tile overlaps the next tile's main loop.  Both CTAs' TMA loads count on
// the leader's stage barrier; both CTAs' epilogues release the leader's
// accumulator barrier.  No multicast load: each CTA reads only its own part.
// ---------------------------------------------------------------------------
constexpr int P_STAGES = 6;
constexpr int P_STAGE_BYTES = A_BYTES + B_HALF_BYTES;   // 32 KiB per CTA
constexpr int P_THREADS = 192;
constexpr int P_BMT = 256;
constexpr uint32_t P_IDESC_FULL = idesc_bf16_f32(256, BN_MMA);
// A group's last row tile with fewer than 256 rows is computed with the
// operands swapped (D^T = W * X^T): the pair's 256 weight rows (each CTA's B
// half) on the MMA's M side and the tile's rows, padded to 16, on its N side.
// A 5-row tile then costs 16 rows of tensor work instead of 128; under the
// power cap the saved tensor work is saved time.
constexpr int P_XG_FLOATS = 64 * 17;                    // SwiGLU gate exchange (64 rows x 16, padded)

struct PairCtl {
    unsigned long long full[P_STAGES];
    unsigned long long empty[P_STAGES];
    unsigned long long tfull[2];
    unsigned long long tempty[2];
    unsigned long long drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
};

template <int MODE>
__global__ void __launch_bounds__(P_THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const KParams p) {
    constexpr int BN_OUT = (MODE == kGemmSwiGLU) ? 128 : 256;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    PairCtl* ctl = reinterpret_cast<PairCtl*>(smem + P_STAGES * P_STAGE_BYTES);
    int* prefix = reinterpret_cast<int*>(ctl + 1);
    int* rstart = prefix + (p.groups + 1);
    int* rcount = rstart + p.groups;
    float* xg = reinterpret_cast<float*>(rcount + p.groups);        // [P_XG_FLOATS]
    const uint32_t smem_base = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();                 // 0: leader, 1: peer
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    const int ntn = (p.N + BN_OUT - 1) / BN_OUT;

    if (tid == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), 8);            // 4 epilogue warps x 2 CTAs
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    pdl_wait();
    pdl_trigger();
    const bool skip = p.gated && p.hdr->cap_exceeded;   // as in grouped_gemm_kernel
    for (int g = tid; g < p.groups; g += P_THREADS) {
        if (skip) {
            rstart[g] = 0;
            rcount[g] = 0;
        } else if (p.offsets) {
            int lo = p.offsets[g], hi = p.offsets[g + 1];
            lo = lo < 0 ? 0 : (lo > p.a_rows ? p.a_rows : lo);
            hi = hi < lo ? lo : (hi > p.a_rows ? p.a_rows : hi);
            rstart[g] = lo;
            rcount[g] = hi - lo;
        } else {
            rstart[g] = 0;
            rcount[g] = p.rows_all;
        }
    }
    __syncthreads();
    {
        const int n = p.groups;
        const int per = (n + P_THREADS - 1) / P_THREADS;
        const int g0 = tid * per;
        int loc = 0;
        for (int i = 0; i < per; ++i)
            if (g0 + i < n) loc += ((rcount[g0 + i] + P_BMT - 1) / P_BMT) * ntn;
        int inc = loc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        __shared__ int wtot[P_THREADS / 32];
        if (lane == 31) wtot[warp] = inc;
        __syncthreads();
        int run = inc - loc;
        for (int w = 0; w < warp; ++w) run += wtot[w];
        for (int i = 0; i < per; ++i) {
            if (g0 + i < n) {
                prefix[g0 + i] = run;
                run += ((rcount[g0 + i] + P_BMT - 1) / P_BMT) * ntn;
            }
        }
        if (tid == P_THREADS - 1) { prefix[n] = run; ctl->total_tiles = run; }
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before any cross-CTA arrive
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int total = ctl->total_tiles;
    volatile int* abort = &ctl->abort;
    const int nkb = (p.K + BK - 1) / BK;
    const int nk = nkb * p.nseg;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            long long armed = 0;
            for (int tile = pair; tile < total && ok; tile += npairs) {
                const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p, ntn, P_BMT);
                const int rows_t = t.mrows - t.mt * P_BMT;             // rows of this tile
                const bool swap = rows_t < P_BMT;
                const int npad = (rows_t + 15) & ~15;
                // this CTA's rows of the tile: all 256 rows split 128/128 (full), or the
                // padded rows split npad/2 each (swapped)
                const int a_row = t.row0 + t.mt * P_BMT + (int)rank * (swap ? npad / 2 : BM);
                const int n0 = t.nt * BN_OUT;
                // B half of this CTA: SwiGLU -- 64 gate rows and the matching 64 up
                // rows of output columns n0 + 64*rank ..; otherwise 128 rows
                const int b_row = t.g * p.b_group_rows + n0 + (int)rank * ((MODE == kGemmSwiGLU) ? 64 : 128);
                for (int i = 0; i < nk; ++i) {
                    const int seg = i / nkb, kb = i - seg * nkb;
                    if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort)) { ok = false; break; }
                    const uint32_t full_local = smem_u32(&ctl->full[stage]);
                    const uint32_t full_leader = mapa_shared(full_local, 0);
                    if (rank == 0) mbar_arrive_expect_tx(full_local, 2 * P_STAGE_BYTES);
                    const uint32_t sa = smem_base + stage * P_STAGE_BYTES;
                    // swapped: weights in the MMA's A slot, rows in its B slot (16 KiB each)
                    const uint32_t s_rows = swap ? sa + A_BYTES : sa;
                    const uint32_t s_w = swap ? sa : sa + A_BYTES;
                    tma_load_2d_pair(s_rows, &tmA, full_leader, seg * p.a_seg_col + kb * BK, a_row);
                    if (MODE == kGemmSwiGLU) {   // 64 gate rows, then the 64 up rows: one 4-D box
                        tma_load_4d_pair(s_w, &tmB, full_leader, kb * BK, n0 + (int)rank * 64, 0, t.g);
                    } else {
                        tma_load_2d_pair(s_w, &tmB, full_leader, kb * BK, b_row + seg * p.b_seg_row);
                    }
                    ++armed;
                    if (++stage == P_STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // Both CTAs' copies of a stage complete on the leader's full barrier,
                // armed for the pair's bytes: the leader waits for the phases it armed
                // (and the closing cluster barrier holds the peer until then); the
                // peer, which cannot wait on a remote barrier, adds the fixed delay.
                if (rank != 0 || !wait_armed_stages(smem_u32(&ctl->full[0]), P_STAGES, armed)) settle_delay();
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmProducer;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader CTA) ----------------
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true;
            for (int tile = pair; tile < total && ok; tile += npairs) {
                const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p, ntn, P_BMT);
                const int rows_t = t.mrows - t.mt * P_BMT;
                const uint32_t idesc = rows_t < P_BMT ? idesc_bf16_f32(256, (rows_t + 15) & ~15) : P_IDESC_FULL;
                if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN_MMA);
                for (int i = 0; i < nk; ++i) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), ph, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_base + stage * P_STAGE_BYTES;
                    const uint64_t ad = sdesc_k_sw128(sa);
                    const uint64_t bd = sdesc_k_sw128(sa + A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                                         (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit_pair_mc(smem_u32(&ctl->empty[stage]), (uint16_t)3);
                    if (++stage == P_STAGES) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair_mc(smem_u32(&ctl->tfull[acc]), (uint16_t)3);
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
            tc_commit_pair(smem_u32(&ctl->drain));
            volatile int never = 0;
            const bool drained = mbar_wait_bounded(smem_u32(&ctl->drain), 0, &never);
            if (!ok || !drained) {
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmMma;
                *abort = 1;
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int q = warp & 3;
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = pair; tile < total; tile += npairs) {
            const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p, ntn, P_BMT);
            if (!mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort)) {
                if (lane == 0) {
                    raise_status(p.hdr, MOE_ERR_TIMEOUT);
                    p.hdr->timeout_site = kSiteGemmEpilogue;
                }
                break;
            }
            tc_fence_after();
            const int rows_t = t.mrows - t.mt * P_BMT;
            if (rows_t < P_BMT) {
                // Swapped: TMEM lane = this CTA's weight row i (its B half), column j =
                // row j of the tile.  SwiGLU: lanes 0..63 gate, 64..127 up of output
                // columns n0 + 64*rank + (i mod 64); the gate values cross to the up
                // warps through shared memory, 16 rows at a time.
                const int i = q * 32 + lane;
                const int n0 = t.nt * BN_OUT;
                const bool gate = MODE == kGemmSwiGLU && q < 2;
                const int col = (MODE == kGemmSwiGLU) ? n0 + 64 * (int)rank + (i & 63) : n0 + 128 * (int)rank + i;
                const bool col_ok = col < p.N;
                const uint32_t tl = tmem_base + (uint32_t)(acc * BN_MMA) + ((uint32_t)(q * 32) << 16);
                const int npad = (rows_t + 15) & ~15;
                for (int c = 0; c < npad; c += 16) {
                    uint32_t v[16];
                    tmem_ld_16cols(tl + (uint32_t)c, v);
                    tmem_ld_wait();
                    if (MODE == kGemmSwiGLU) {
                        if (gate) {
#pragma unroll
                            for (int u = 0; u < 16; ++u) xg[i * 17 + u] = __uint_as_float(v[u]);
                        }
                        epi_bar_sync();
                        if (!gate && col_ok) {
#pragma unroll
                            for (int u = 0; u < 16; ++u) {
                                const int row = c + u;
                                if (row < rows_t) {
                                    const float g = xg[(i - 64) * 17 + u];
                                    out_row<MODE>(p, t.row0 + t.mt * P_BMT + row, t.g)[col] =
                                        __float2bfloat16_rn(g / (1.0f + __expf(-g)) * __uint_as_float(v[u]));
                                }
                            }
                        }
                        epi_bar_sync();
                    } else if (col_ok) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int row = c + u;
                            if (row < rows_t) {
                                const float x = __uint_as_float(v[u]);
                                auto* o = out_row<MODE>(p, t.row0 + t.mt * P_BMT + row, t.g) + col;
                                if constexpr (MODE == kGemmF32) *o = x;
                                else *o = __float2bfloat16_rn(MODE == kGemmReLU2 ? (x > 0.f ? x * x : 0.f) : x);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[acc]), 0));
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
                continue;
            }
            {
                // Full tile (M 256): lane = this CTA's row 128*rank + 32q + lane, all
                // 256 columns; D columns 0..127 come from CTA 0's B half, 128..255
                // from CTA 1's.
                const int r = t.mt * P_BMT + (int)rank * BM + q * 32 + lane;
                auto* orow = out_row<MODE>(p, t.row0 + r, t.g);
                const uint32_t tl = tmem_base + (uint32_t)(acc * BN_MMA) + ((uint32_t)(q * 32) << 16);
                const int n0 = t.nt * BN_OUT;
                if (MODE == kGemmSwiGLU) {
                    // each 128-column block is [64 gate | 64 up] of output columns 64 * block ..
#pragma unroll 1
                    for (int b = 0; b < 2; ++b)
#pragma unroll 1
                        for (int i0 = 0; i0 < 64; i0 += 32)
                            epilogue_chunk<MODE>(tl + b * 128 + i0, tl + b * 128 + 64 + i0, true, orow,
                                                 n0 + 64 * b + i0, p.N);
                } else {
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) epilogue_chunk<MODE>(tl + c * 32, 0, true, orow, n0 + c * 32, p.N);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[acc]), 0));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    // the leader's MMAs have drained before either CTA frees its TMEM
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Quantized expert weights at prefill sizes (ONNX Runtime PR #33963: weight-only
// quantized FC1/FC2 with BF16 activations; here FP8 E4M3 with a scale per weight
// row, or NVFP4 with an E4M3 scale per 16 elements and a scale per row).
// The single-CTA tile of the BF16 kernel -- 128 activation rows (A) by 256
// weight rows (B) per tile, tcgen05.mma M128 N256 K16 into TMEM -- with B read
// as codes: the TMA ring carries the A box and two 128-row code boxes per 64-wide
// K step (16 or 8 KiB of codes instead of 32 KiB of BF16), and eight converter
// warps decode each step's codes exactly to BF16 (the decoders of the small-row
// kernel) into a separate ring of swizzled B tiles, which the MMA reads from
// shared memory.  Each weight tile is converted once per 128-row activation tile,
// however many rows the group holds.  The row scales multiply the accumulator in
// the epilogue (NVFP4 tiles are converted at 2^-8 of their value and undone there).
// A ring stage is released by the converters (codes read) and the MMA (A read).
// ---------------------------------------------------------------------------
constexpr int Q_STAGES = 5;                               // the most any geometry uses
constexpr int Q_CSLOTS = 2;
constexpr int Q_CONV_WARPS = 8;
constexpr int Q_SLOT_BYTES = B_BYTES;                     // 256 rows x 64 BF16, 128-byte swizzled

template <int WF>
struct QCfg {
    static constexpr int CODE_ROW = WF == kWeightNvfp4 ? 32 : 64;   // code bytes per weight row per K step
    static constexpr int CODE_BOX = 128 * CODE_ROW;                 // one 128-row code box
    // NVFP4: 16 bytes of block scales per weight row (the 16-byte group holding this
    // K step's four), one box per 128 rows
    static constexpr int SCALE_BOX = WF == kWeightNvfp4 ? 128 * 16 : 0;
};
// Tile geometry: 128 activation rows per tile, a ring of QParams::stages TMA
// stages (four, or five of the smaller NVFP4 stages where they fit), two
// converted B tiles, double-buffered accumulators; warps: producer, MMA, four
// epilogue warps, eight converter warps.
template <int WF>
struct QGeo {
    static constexpr int S_PART = A_BYTES + 2 * QCfg<WF>::CODE_BOX;        // NVFP4 block-scale boxes
    static constexpr int STAGE_BYTES = S_PART + 2 * QCfg<WF>::SCALE_BOX;
    static constexpr int CONV_W0 = 6;                                     // first converter warp
    static constexpr int THREADS = 32 * CONV_W0 + 32 * Q_CONV_WARPS;
};

struct QParams {
    KParams k;
    const float* wscale;        // FP32 scale per weight row
    int stages;                 // TMA ring stages (at most Q_STAGES)
};

struct QCtl {
    float scl[4][256];          // per epilogue warp: the weight-row scales of its tile's 256 B rows
    unsigned long long full[Q_STAGES];
    unsigned long long empty[Q_STAGES];
    unsigned long long cfull[Q_CSLOTS];
    unsigned long long cempty[Q_CSLOTS];
    unsigned long long tfull[2];
    unsigned long long tempty[2];
    unsigned long long drain;
    uint32_t tmem_base;
    int abort;
    int total_tiles;
};

// The epilogue chunk with the weight rows' scales: output column col0 + c of the
// tile takes scale sg[c] (and su[c] for the matching up row), from shared memory.
template <int MODE>
__device__ __forceinline__ void epilogue_chunk_q(uint32_t tg, uint32_t tu, bool row_ok, __nv_bfloat16* orow,
                                                 int col0, int N, const float* sg, const float* su) {
    uint32_t gv[32], uv[32];
    tmem_ld_32cols(tg, gv);
    if (MODE == kGemmSwiGLU) tmem_ld_32cols(tu, uv);
    tmem_ld_wait();
    if (!row_ok) return;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int c0 = col0 + v * 8;
        if (c0 < N) {                       // N is a multiple of 8: the whole group of 8 is inside
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float a[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = v * 8 + 2 * i + h;
                    const float x = __uint_as_float(gv[j]) * sg[j];
                    if (MODE == kGemmSwiGLU) {
                        const float u = __uint_as_float(uv[j]) * su[j];
                        a[h] = x / (1.0f + __expf(-x)) * u;
                    } else if (MODE == kGemmReLU2) {
                        a[h] = x > 0.f ? x * x : 0.f;
                    } else {
                        a[h] = x;
                    }
                }
                o[i] = pack2(a[0], a[1]);
            }
            *reinterpret_cast<uint4*>(orow + c0) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

template <int MODE, int WF>
__global__ void __launch_bounds__(QGeo<WF>::THREADS, 1)
grouped_gemm_q_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmS, const QParams qp) {
    using QC = QCfg<WF>;
    using QG = QGeo<WF>;
    constexpr bool FP4W = WF == kWeightNvfp4;
    constexpr int BN_OUT = (MODE == kGemmSwiGLU) ? 128 : 256;
    const KParams& p = qp.k;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    const int nst = qp.stages;
    uint8_t* slots = smem + nst * QG::STAGE_BYTES;          // converted B tiles
    QCtl* ctl = reinterpret_cast<QCtl*>(slots + Q_CSLOTS * Q_SLOT_BYTES);
    int* prefix = reinterpret_cast<int*>(ctl + 1);
    int* rstart = prefix + (p.groups + 1);
    int* rcount = rstart + p.groups;
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t slot_base = smem_u32(slots);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntn = (p.N + BN_OUT - 1) / BN_OUT;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1 + Q_CONV_WARPS);      // MMA commit + converter warps
        }
        for (int c = 0; c < Q_CSLOTS; ++c) {
            mbar_init(smem_u32(&ctl->cfull[c]), Q_CONV_WARPS);
            mbar_init(smem_u32(&ctl->cempty[c]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), 4);                 // the 4 epilogue warps
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (FP4W) tma_prefetch_desc(&tmS);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    // after a capacity overflow in the same layer call no payload moved: no tiles
    const bool skip = p.gated && p.hdr->cap_exceeded;
    for (int g = tid; g < p.groups; g += QG::THREADS) {
        if (skip) {
            rstart[g] = 0;
            rcount[g] = 0;
        } else if (p.offsets) {
            int lo = p.offsets[g], hi = p.offsets[g + 1];
            lo = lo < 0 ? 0 : (lo > p.a_rows ? p.a_rows : lo);
            hi = hi < lo ? lo : (hi > p.a_rows ? p.a_rows : hi);
            rstart[g] = lo;
            rcount[g] = hi - lo;
        } else {
            rstart[g] = 0;
            rcount[g] = p.rows_all;
        }
    }
    __syncthreads();
    if (tid == 0) {             // exclusive scan of tiles per group (at most 1024 groups)
        int run = 0;
        for (int g = 0; g < p.groups; ++g) {
            prefix[g] = run;
            run += ((rcount[g] + BM - 1) / BM) * ntn;
        }
        prefix[p.groups] = run;
        ctl->total_tiles = run;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int total = ctl->total_tiles;
    volatile int* abort = &ctl->abort;
    const int nk = (p.K + BK - 1) / BK;

    if (warp == 0) {
        // ---------------- TMA producer: A box + two code boxes per K step ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            long long armed = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p,
                                                                                     ntn, BM);
                const int a_row = t.row0 + t.mt * BM;
                const uint32_t bytes = (uint32_t)QG::STAGE_BYTES;
                const int b_lo = t.g * p.b_group_rows + t.nt * BN_OUT;
                const int b_hi = (MODE == kGemmSwiGLU) ? b_lo + p.up_off : b_lo + 128;
                for (int i = 0; i < nk; ++i) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort)) { ok = false; break; }
                    const uint32_t full = smem_u32(&ctl->full[stage]);
                    const uint32_t sa = smem_base + stage * QG::STAGE_BYTES;
                    mbar_arrive_expect_tx(full, bytes);
                    tma_load_2d(sa, &tmA, full, i * BK, a_row);
                    tma_load_2d(sa + A_BYTES, &tmB, full, i * QC::CODE_ROW, b_lo);
                    tma_load_2d(sa + A_BYTES + QC::CODE_BOX, &tmB, full, i * QC::CODE_ROW, b_hi);
                    if (FP4W) {     // the 16-byte group of block scales holding step i's four
                        tma_load_2d(sa + QG::S_PART, &tmS, full, (i * (BK / 16)) & ~15, b_lo);
                        tma_load_2d(sa + QG::S_PART + QC::SCALE_BOX, &tmS, full, (i * (BK / 16)) & ~15, b_hi);
                    }
                    ++armed;
                    if (++stage == nst) { stage = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                if (!wait_armed_stages(smem_u32(&ctl->full[0]), nst, armed)) settle_delay();
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmProducer;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: A from the ring, B from the converted tiles ----------------
        if (lane == 0) {
            int stage = 0, acc = 0, cs = 0;
            uint32_t ph = 0, aph = 0, cph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p,
                                                                                     ntn, BM);
                const uint32_t idesc = t.mrows - t.mt * BM <= kTailRows ? IDESC64 : IDESC;
                if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)(acc * BN_MMA);
                for (int i = 0; i < nk; ++i) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), ph, abort) ||
                        !mbar_wait_bounded(smem_u32(&ctl->cfull[cs]), cph, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = sdesc_k_sw128(smem_base + stage * QG::STAGE_BYTES);
                    const uint64_t bd = sdesc_k_sw128(slot_base + cs * Q_SLOT_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_bf16(d0, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                                    (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(smem_u32(&ctl->empty[stage]));
                    tc_commit(smem_u32(&ctl->cempty[cs]));
                    if (++stage == nst) { stage = 0; ph ^= 1u; }
                    if (++cs == Q_CSLOTS) { cs = 0; cph ^= 1u; }
                }
                if (!ok) break;
                tc_commit(smem_u32(&ctl->tfull[acc]));
                if (++acc == 2) { acc = 0; aph ^= 1u; }
            }
            tc_commit(smem_u32(&ctl->drain));
            volatile int never = 0;
            const bool drained = mbar_wait_bounded(smem_u32(&ctl->drain), 0, &never);
            if (!ok || !drained) {
                raise_status(p.hdr, MOE_ERR_TIMEOUT);
                p.hdr->timeout_site = kSiteGemmMma;
                *abort = 1;
            }
        }
    } else if (warp >= QG::CONV_W0) {
        // ---------------- converters (the last 8 warps): codes -> swizzled BF16 B tile ----------------
        // Thread ct takes, in four passes, weight row r = 64*pass + ct/4 of the
        // 256-row tile and its 16-element quarter qd = ct%4 of the 64-wide K step:
        // reads 16 codes (FP8: 16 bytes; NVFP4: 8 bytes and the block's scale),
        // writes 16 BF16 as two 16-byte chunks of the row at chunk (2qd + h) ^ (r%8).
        const int ct = tid - 32 * QG::CONV_W0;
        const int qd = ct & 3;
        int stage = 0, cs = 0;
        uint32_t ph = 0, cph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            for (int i = 0; i < nk; ++i) {
                if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), ph, abort) ||
                    !mbar_wait_bounded(smem_u32(&ctl->cempty[cs]), cph ^ 1u, abort)) { ok = false; break; }
                const uint8_t* codes = smem + stage * QG::STAGE_BYTES + A_BYTES;
                // NVFP4: this quarter's block scale of each pass, from the stage (0x100
                // marks a block past K: zeros; rows past the weights arrive as scale 0)
                uint32_t s_cur[4] = {0u, 0u, 0u, 0u};
                if (FP4W) {
                    const uint8_t* sc = smem + stage * QG::STAGE_BYTES + QG::S_PART + (i & 3) * 4 + qd;
                    const bool in_k = i * BK + qd * 16 < p.K;
#pragma unroll
                    for (int pass = 0; pass < 4; ++pass) {
                        const int r = pass * 64 + (ct >> 2);
                        s_cur[pass] = in_k ? (uint32_t)sc[(r >> 7) * QC::SCALE_BOX + (r & 127) * 16] : 0x100u;
                    }
                }
                uint8_t* dst = slots + cs * Q_SLOT_BYTES;
#pragma unroll
                for (int pass = 0; pass < 4; ++pass) {
                    const int r = pass * 64 + (ct >> 2);
                    const uint8_t* src = codes + (r >> 7) * QC::CODE_BOX + (r & 127) * QC::CODE_ROW;
                    uint32_t v[8];
                    if constexpr (FP4W) {
                        // this quarter is one 16-element block: its E4M3 scale, at 2^-8
                        // (0x100 marks a block past K: zeros)
                        uint32_t m = 0u;
                        if (s_cur[pass] != 0x100u) {
                            constexpr uint32_t kTwo118 = 0x7A807A80u;       // (2^118, 2^118) in BF16
                            uint32_t lo, hi;
                            e4m3x4_to_bf16x4(s_cur[pass], lo, hi);
                            asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(lo), "r"(kTwo118));
                            asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(m) : "r"(lo));
                        }
                        const uint2 w = *reinterpret_cast<const uint2*>(src + qd * 8);
                        e2m1x8_to_bf16x8(w.x, m, &v[0]);
                        e2m1x8_to_bf16x8(w.y, m, &v[4]);
                    } else {
                        const uint4 w = *reinterpret_cast<const uint4*>(src + qd * 16);
                        e4m3x4_to_bf16x4(w.x, v[0], v[1]);
                        e4m3x4_to_bf16x4(w.y, v[2], v[3]);
                        e4m3x4_to_bf16x4(w.z, v[4], v[5]);
                        e4m3x4_to_bf16x4(w.w, v[6], v[7]);
                    }
                    uint8_t* drow = dst + r * 128;
                    *reinterpret_cast<uint4*>(drow + (((2 * qd) ^ (r & 7)) << 4)) = make_uint4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<uint4*>(drow + (((2 * qd + 1) ^ (r & 7)) << 4)) =
                        make_uint4(v[4], v[5], v[6], v[7]);
                }
                // the BF16 tile is read by the tensor core (async proxy); the codes
                // have been read: release both
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&ctl->cfull[cs]));
                    mbar_arrive(smem_u32(&ctl->empty[stage]));
                }
                if (++stage == nst) { stage = 0; ph ^= 1u; }
                if (++cs == Q_CSLOTS) { cs = 0; cph ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5): scales, activation, BF16 stores ----------------
        // warp w: TMEM lane quarter w % 4 (the warps a warp may read)
        const int q = warp & 3;
        const float undo = FP4W ? 256.f : 1.f;
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode_tile<MODE == kGemmSwiGLU || MODE == kGemmReLU2>(tile, prefix, rstart, rcount, p,
                                                                                 ntn, BM);
            const int n0 = t.nt * BN_OUT;
            // the tile's 256 weight-row scales into this warp's shared slice while
            // the accumulator fills (SwiGLU: 128 gate rows, then the 128 up rows);
            // warp-local, so a warp that gives up leaves no other warp waiting
            float* scl = ctl->scl[warp - 2];
#pragma unroll
            for (int j = lane; j < 256; j += 32) {
                const int col = n0 + (MODE == kGemmSwiGLU ? (j & 127) : j);
                const long long row = (long long)t.g * p.b_group_rows + col +
                                      ((MODE == kGemmSwiGLU && j >= 128) ? p.up_off : 0);
                scl[j] = col < p.N ? __ldg(qp.wscale + row) * undo : 0.f;
            }
            __syncwarp();
            if (!mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort)) {
                if (lane == 0) {
                    raise_status(p.hdr, MOE_ERR_TIMEOUT);
                    p.hdr->timeout_site = kSiteGemmEpilogue;
                }
                break;
            }
            tc_fence_after();
            // M = 64 tiles keep row 16q + i in lane 32q + i (i < 16)
            const int row0 = t.mt * BM;
            const bool m64 = t.mrows - row0 <= kTailRows;
            const int r = m64 ? row0 + q * 16 + lane : row0 + q * 32 + lane;
            const bool row_ok = (!m64 || lane < 16) && r < t.mrows;
            __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(out_row<MODE>(p, t.row0 + (row_ok ? r : 0), t.g));
            const uint32_t tbase = tmem_base + (uint32_t)(acc * BN_MMA) + ((uint32_t)(q * 32) << 16);
            if (MODE == kGemmSwiGLU) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c)
                    epilogue_chunk_q<MODE>(tbase + c * 32, tbase + 128 + c * 32, row_ok, orow, n0 + c * 32, p.N,
                                           scl + c * 32, scl + 128 + c * 32);
            } else {
#pragma unroll 1
                for (int c = 0; c < 8; ++c)
                    epilogue_chunk_q<MODE>(tbase + c * 32, 0, row_ok, orow, n0 + c * 32, p.N, scl + c * 32,
                                           scl + c * 32);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
            if (++acc == 2) { acc = 0; aph ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- host side ---------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Row-major [rows, cols] BF16, 64-column x box_rows boxes, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols, unsigned box_rows = 128) {
    auto enc = encode_fn();
    if (!enc) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d) for a [%lld, %lld] bf16 tensor at %p", (int)r, rows,
                  cols, base);
        return false;
    }
    return true;
}

// SwiGLU weights [groups x (gate rows | up rows), cols] BF16 seen as 4-D
// (cols, row in half, half, group): one box brings box_rows gate rows and the
// up rows of the same output columns, gate first -- in shared memory exactly
// the two box_rows-row boxes of the 2-D map, one after the other, in one copy
// instead of two.  Rows past the half's end read zeros.
bool make_map_glu(CUtensorMap* m, const void* base, long long rows, long long cols, long long half_rows,
                  long long group_rows, unsigned box_rows) {
    auto enc = encode_fn();
    if (!enc) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    if (half_rows < 1 || group_rows != 2 * half_rows || rows % group_rows != 0) {
        set_error("SwiGLU weight map: %lld rows in groups of %lld, half %lld", rows, group_rows, half_rows);
        return false;
    }
    cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)half_rows, 2u, (cuuint64_t)(rows / group_rows)};
    cuuint64_t strides[3] = {(cuuint64_t)cols * 2, (cuuint64_t)(half_rows * cols * 2), (cuuint64_t)(group_rows * cols * 2)};
    cuuint32_t box[4] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 2u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d) for SwiGLU weights [%lld, %lld] at %p", (int)r, rows,
                  cols, base);
        return false;
    }
    return true;
}

template <int MODE, int HALVES>
cudaError_t launch_mode(const CUtensorMap& ma, const CUtensorMap& mb, const KParams& kp, size_t smem,
                        cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, HALVES>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM);
    });
    if (attr_err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(max dynamic smem %d): %s", MAX_DYN_SMEM, cudaGetErrorString(attr_err));
        return attr_err;
    }
    const cudaError_t e = launch_kernel(grouped_gemm_kernel<MODE, HALVES>, dim3((unsigned)device_sm_count()),
                                        dim3(Cfg<HALVES>::THREADS), smem, st, 1, kUsePdl, ma, mb, kp);
    if (e != cudaSuccess) set_error("grouped GEMM launch (smem %zu): %s", smem, cudaGetErrorString(e));
    return e;
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const KParams& kp, size_t smem,
                        cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(grouped_gemm_pair_kernel<MODE>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM);
    });
    if (attr_err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(max dynamic smem %d): %s", MAX_DYN_SMEM, cudaGetErrorString(attr_err));
        return attr_err;
    }
    const cudaError_t e = launch_kernel(grouped_gemm_pair_kernel<MODE>, dim3((unsigned)(device_sm_count() & ~1)),
                                        dim3(P_THREADS), smem, st, 2, kUsePdl, ma, mb, kp);
    if (e != cudaSuccess) set_error("grouped GEMM pair launch (smem %zu): %s", smem, cudaGetErrorString(e));
    return e;
}

template <int MODE, int WF>
cudaError_t launch_q(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ms, const QParams& qp,
                     size_t smem, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(grouped_gemm_q_kernel<MODE, WF>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_DYN_SMEM);
    });
    if (attr_err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(max dynamic smem %d): %s", MAX_DYN_SMEM, cudaGetErrorString(attr_err));
        return attr_err;
    }
    const cudaError_t e = launch_kernel(grouped_gemm_q_kernel<MODE, WF>, dim3((unsigned)device_sm_count()),
                                        dim3(QGeo<WF>::THREADS), smem, st, 1, kUsePdl, ma, mb, ms, qp);
    if (e != cudaSuccess) set_error("quantized grouped GEMM launch (smem %zu): %s", smem, cudaGetErrorString(e));
    return e;
}

template <int WF>
size_t q_smem_bytes(int groups, int stages) {
    return 1024 + (size_t)stages * QGeo<WF>::STAGE_BYTES + (size_t)Q_CSLOTS * Q_SLOT_BYTES +
           sizeof(QCtl) +
           3 * (size_t)(groups + 1) * 4;
}

size_t pair_smem_bytes(int groups) {
    return 1024 + (size_t)P_STAGES * P_STAGE_BYTES + sizeof(PairCtl) + 3 * (size_t)(groups + 1) * 4 +
           (size_t)P_XG_FLOATS * 4;
}

template <int HALVES>
size_t smem_bytes(int groups) {
    return 1024 + (size_t)Cfg<HALVES>::STAGES * Cfg<HALVES>::STAGE_BYTES + sizeof(SmemCtl<HALVES>) +
           3 * (size_t)(groups + 1) * 4;
}

}  // namespace

bool make_tensor_map_bf16_chunks(CUtensorMap* m, const void* base, long long rows, long long cols, unsigned box_rows,
                                 unsigned chunks) {
    auto enc = encode_fn();
    if (!enc) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    if (cols % BK != 0) {
        set_error("chunked tensor map: %lld columns are not whole 64-column chunks", cols);
        return false;
    }
    cuuint64_t dims[3] = {(cuuint64_t)BK, (cuuint64_t)rows, (cuuint64_t)(cols / BK)};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)BK * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, (cuuint32_t)chunks};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d) for a chunked [%lld, %lld] bf16 tensor at %p", (int)r,
                  rows, cols, base);
        return false;
    }
    return true;
}

bool make_tensor_map_glu_chunks(CUtensorMap* m, const void* base, long long rows, long long cols, long long half_rows,
                                long long group_rows, unsigned box_rows, unsigned chunks) {
    auto enc = encode_fn();
    if (!enc) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    if (cols % BK != 0 || half_rows < 1 || group_rows != 2 * half_rows || rows % group_rows != 0) {
        set_error("chunked SwiGLU weight map: [%lld, %lld] in groups of %lld, half %lld", rows, cols, group_rows,
                  half_rows);
        return false;
    }
    cuuint64_t dims[5] = {(cuuint64_t)BK, (cuuint64_t)half_rows, 2u, (cuuint64_t)(rows / group_rows),
                          (cuuint64_t)(cols / BK)};
    cuuint64_t strides[4] = {(cuuint64_t)cols * 2, (cuuint64_t)(half_rows * cols * 2),
                             (cuuint64_t)(group_rows * cols * 2), (cuuint64_t)BK * 2};
    cuuint32_t box[5] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 2u, 1u, (cuuint32_t)chunks};
    cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d) for chunked SwiGLU weights [%lld, %lld] at %p",
                  (int)r, rows, cols, base);
        return false;
    }
    return true;
}

bool make_tensor_map_bf16(CUtensorMap* m, const void* base, long long rows, long long cols, unsigned box_rows) {
    return make_map(m, base, rows, cols, box_rows);
}

bool make_tensor_map_u8_rows(CUtensorMap* m, const void* base, long long rows, long long cols, long long stride,
                             unsigned box_cols, unsigned box_rows) {
    // 128-byte rows are 128-byte swizzled (the converter reads them conflict-free)
    auto enc = encode_fn();
    if (!enc) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)stride};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d) for a [%lld, %lld] byte tensor at %p", (int)r, rows,
                  cols, base);
        return false;
    }
    return true;
}

moe_status launch_grouped_gemm(const GemmProblem& g, WsHeader* hdr, cudaStream_t st) {
    if (g.groups < 1 || g.groups > 1024 || g.K < 1 || g.N < 1) {
        set_error("grouped GEMM: unsupported problem (groups %d, K %d, N %d)", g.groups, g.K, g.N);
        return MOE_ERR_UNSUPPORTED;
    }
    // A bound on the rows of any group: a few dozen rows make the GEMM a weight
    // stream.  When its work items (non-empty groups x 128-row weight blocks)
    // fit in about two waves the small-row kernel spreads them over more SMs and
    // starts sooner; with many more items the tile kernels' larger tiles
    // stream a few percent better (measured at 1 to 16 tokens over 240 experts).
    const long long row_bound = g.offsets ? (g.max_group_rows > 0 ? g.max_group_rows : g.a_rows) : g.rows_all;
    if (g.wfmt != kWeightBf16) {
        if (g.nseg != 1) {
            set_error("grouped GEMM: quantized weights take one K segment");
            return MOE_ERR_UNSUPPORTED;
        }
        // Groups of up to 64 rows (decode): the small-row kernel, weights on the
        // MMA's M side, converted into tensor memory.  Larger groups (prefill):
        // the tile kernel with converted B tiles, each weight tile converted once
        // per 128 activation rows instead of re-streamed per 64-row chunk.
        if (row_bound <= kDecodeRows || g.mode == kGemmF32) {
            const int nb = row_bound >= kDecodeRows ? kDecodeRows
                                                    : (row_bound < 16 ? 16 : (int)((row_bound + 15) / 16 * 16));
            return launch_decode_gemm(g, nb, hdr, st);
        }
        const bool fp4 = g.wfmt == kWeightNvfp4;
        if (fp4 && (!g.bscale || g.K % 32 != 0 || g.bscale_stride % 16 != 0 || g.bscale_stride * 16 < g.K)) {
            set_error("grouped GEMM: NVFP4 weights need K %% 32 == 0 and 16-byte block-scale rows covering K");
            return MOE_ERR_UNSUPPORTED;
        }
        if (!g.wscale) {
            set_error("grouped GEMM: quantized weights need a scale per weight row");
            return MOE_ERR_UNSUPPORTED;
        }
        // five of the smaller NVFP4 stages where the group list leaves room, else four
        const int qst = fp4 && q_smem_bytes<kWeightNvfp4>(g.groups, Q_STAGES) <= (size_t)MAX_DYN_SMEM ? Q_STAGES : 4;
        const size_t smem = fp4 ? q_smem_bytes<kWeightNvfp4>(g.groups, qst) : q_smem_bytes<kWeightFp8E4M3>(g.groups, qst);
        if (smem > (size_t)MAX_DYN_SMEM) {
            set_error("quantized grouped GEMM needs %zu bytes of shared memory", smem);
            return MOE_ERR_UNSUPPORTED;
        }
        CUtensorMap ma, mb;
        if (!make_map(&ma, g.a, g.a_rows, g.a_cols)) return MOE_ERR_CUDA;
        const long long code_cols = fp4 ? g.b_cols / 2 : g.b_cols;
        if (!make_tensor_map_u8_rows(&mb, g.b, g.b_rows, code_cols, code_cols,
                                     (unsigned)(fp4 ? QCfg<kWeightNvfp4>::CODE_ROW : QCfg<kWeightFp8E4M3>::CODE_ROW),
                                     128u))
            return MOE_ERR_CUDA;
        // NVFP4 block scales: 16-byte groups of 128 weight rows
        CUtensorMap ms = mb;
        if (fp4 && !make_tensor_map_u8_rows(&ms, g.bscale, g.b_rows, g.bscale_stride, g.bscale_stride, 16u, 128u))
            return MOE_ERR_CUDA;
        QParams qp;
        qp.k.offsets = g.offsets;
        qp.k.groups = g.groups;
        qp.k.rows_all = g.rows_all;
        qp.k.a_rows = (int)g.a_rows;
        qp.k.K = g.K;
        qp.k.nseg = 1;
        qp.k.a_seg_col = 0;
        qp.k.b_seg_row = 0;
        qp.k.N = g.N;
        qp.k.b_group_rows = g.b_group_rows;
        qp.k.up_off = g.up_off;
        qp.k.out = g.out;
        qp.k.ldo = g.ldo;
        qp.k.out_group_col = g.out_group_col;
        qp.k.hdr = hdr;
        qp.k.gated = g.gated;
        qp.wscale = g.wscale;
        qp.stages = qst;
        cudaError_t e;
        if (fp4) {
            switch (g.mode) {
                case kGemmSwiGLU: e = launch_q<kGemmSwiGLU, kWeightNvfp4>(ma, mb, ms, qp, smem, st); break;
                case kGemmReLU2: e = launch_q<kGemmReLU2, kWeightNvfp4>(ma, mb, ms, qp, smem, st); break;
                default: e = launch_q<kGemmPlain, kWeightNvfp4>(ma, mb, ms, qp, smem, st); break;
            }
        } else {
            switch (g.mode) {
                case kGemmSwiGLU: e = launch_q<kGemmSwiGLU, kWeightFp8E4M3>(ma, mb, ms, qp, smem, st); break;
                case kGemmReLU2: e = launch_q<kGemmReLU2, kWeightFp8E4M3>(ma, mb, ms, qp, smem, st); break;
                default: e = launch_q<kGemmPlain, kWeightFp8E4M3>(ma, mb, ms, qp, smem, st); break;
            }
        }
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    if (row_bound <= kDecodeRows) {
        const long long slots = g.offsets ? (g.a_rows < g.groups ? g.a_rows : g.groups) : g.groups;
        if (slots * ((g.N + 127) / 128) <= 2LL * device_sm_count())
            return launch_decode_gemm(g, row_bound < 16 ? 16 : (int)((row_bound + 15) / 16 * 16), hdr, st);
    }
    const long long avg_rows = g.offsets ? g.a_rows / g.groups : g.rows_all;
    const bool pairs = avg_rows >= kPairRows && device_sm_count() >= 2;
    CUtensorMap ma, mb;
    if (!make_map(&ma, g.a, g.a_rows, g.a_cols)) return MOE_ERR_CUDA;
    // the pair kernel loads a SwiGLU B half as 64 gate rows + 64 up rows (one 4-D box)
    if (pairs && g.mode == kGemmSwiGLU) {
        if (g.nseg != 1) {
            set_error("grouped GEMM: SwiGLU over %d K segments", g.nseg);
            return MOE_ERR_UNSUPPORTED;
        }
        if (!make_map_glu(&mb, g.b, g.b_rows, g.b_cols, g.up_off, g.b_group_rows, 64u)) return MOE_ERR_CUDA;
    } else if (!make_map(&mb, g.b, g.b_rows, g.b_cols, 128u)) {
        return MOE_ERR_CUDA;
    }
    KParams kp;
    kp.offsets = g.offsets;
    kp.groups = g.groups;
    kp.rows_all = g.rows_all;
    kp.a_rows = (int)g.a_rows;
    kp.K = g.K;
    kp.nseg = g.nseg;
    kp.a_seg_col = g.a_seg_col;
    kp.b_seg_row = g.b_seg_row;
    kp.N = g.N;
    kp.b_group_rows = g.b_group_rows;
    kp.up_off = g.up_off;
    kp.out = g.out;
    kp.ldo = g.ldo;
    kp.out_group_col = g.out_group_col;
    kp.hdr = hdr;
    kp.gated = g.gated;
    if (pairs) {
        const size_t smem = pair_smem_bytes(g.groups);
        if (smem > (size_t)MAX_DYN_SMEM) {
            set_error("grouped GEMM needs %zu bytes of shared memory", smem);
            return MOE_ERR_UNSUPPORTED;
        }
        cudaError_t e;
        switch (g.mode) {
            case kGemmSwiGLU: e = launch_pair<kGemmSwiGLU>(ma, mb, kp, smem, st); break;
            case kGemmReLU2: e = launch_pair<kGemmReLU2>(ma, mb, kp, smem, st); break;
            case kGemmF32: e = launch_pair<kGemmF32>(ma, mb, kp, smem, st); break;
            default: e = launch_pair<kGemmPlain>(ma, mb, kp, smem, st); break;
        }
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    // Long reductions amortise the un-overlapped epilogue of the 256-row
    // tile; short ones keep the double-buffered 128-row tile.
    const int halves = (long long)g.K * g.nseg >= kLongK ? 2 : 1;
    const size_t smem = halves == 2 ? smem_bytes<2>(g.groups) : smem_bytes<1>(g.groups);
    if (smem > (size_t)MAX_DYN_SMEM) {
        set_error("grouped GEMM needs %zu bytes of shared memory", smem);
        return MOE_ERR_UNSUPPORTED;
    }
    cudaError_t e;
    if (halves == 2) {
        switch (g.mode) {
            case kGemmSwiGLU: e = launch_mode<kGemmSwiGLU, 2>(ma, mb, kp, smem, st); break;
            case kGemmReLU2: e = launch_mode<kGemmReLU2, 2>(ma, mb, kp, smem, st); break;
            case kGemmF32: e = launch_mode<kGemmF32, 2>(ma, mb, kp, smem, st); break;
            default: e = launch_mode<kGemmPlain, 2>(ma, mb, kp, smem, st); break;
        }
    } else {
        switch (g.mode) {
            case kGemmSwiGLU: e = launch_mode<kGemmSwiGLU, 1>(ma, mb, kp, smem, st); break;
            case kGemmReLU2: e = launch_mode<kGemmReLU2, 1>(ma, mb, kp, smem, st); break;
            case kGemmF32: e = launch_mode<kGemmF32, 1>(ma, mb, kp, smem, st); break;
            default: e = launch_mode<kGemmPlain, 1>(ma, mb, kp, smem, st); break;
        }
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
