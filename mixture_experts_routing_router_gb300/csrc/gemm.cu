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
// Two shapes of the same kernel (HALVES):
//   1: 128-row tiles, two 256-column accumulators in TMEM so the epilogue of
//      one tile overlaps the main loop of the next; 4 stages of 48 KiB;
//      4 epilogue warps.  For short K (the down projection).
//   2: 256-row tiles as two 128-row halves sharing every B tile (two MMAs per
//      K slice into the two 256-column accumulators), which cuts the operand
//      traffic per FLOP by a third; a tail whose second half is empty loads
//      and multiplies only the first.  3 stages of 64 KiB; the epilogue (8
//      warps, one half each) is not overlapped.  For long K (the up projection).
// SwiGLU tiles load 128 gate rows and the matching 128 up rows as the two
// halves of the 256-row B tile, so gate and up land side by side in one
// accumulator and the epilogue computes silu(g) * u without a second pass.
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
constexpr int MAX_DYN_SMEM = 212 * 1024;
// Reductions at least this long use the 256-row tile (HALVES = 2).
constexpr long long kLongK = 4096;

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
    __nv_bfloat16* out;
    long long ldo;
    int out_group_col;
    WsHeader* hdr;
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

struct Tile { int g, mt, nt, row0, mrows; };

// Largest g with prefix[g] <= tile (empty groups share their prefix value).
__device__ __forceinline__ Tile decode_tile(int tile, const int* prefix, const int* rstart, const int* rcount,
                                            const KParams& p, int ntn) {
    int lo = 0, hi = p.groups;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= tile) lo = mid; else hi = mid;
    }
    Tile t;
    t.g = lo;
    const int local = tile - prefix[lo];
    t.mt = local / ntn;
    t.nt = local - t.mt * ntn;
    t.row0 = rstart[lo];
    t.mrows = rcount[lo];
    return t;
}

// Epilogue of one 128-row accumulator: this warp's 32 TMEM lanes at `tbase`,
// one row per thread; writes the tile's BN_OUT output columns from col_base.
template <int MODE>
__device__ __forceinline__ void epilogue_rows(uint32_t tbase, bool row_ok, __nv_bfloat16* orow, int col_base,
                                              int N) {
    if (MODE == kGemmSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t gv[32], uv[32];
            tmem_ld_32cols(tbase + c * 32, gv);
            tmem_ld_32cols(tbase + 128 + c * 32, uv);
            tmem_ld_wait();
            const int col0 = col_base + c * 32;
            if (row_ok) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    if (col0 + v * 8 < N) {
                        uint32_t o[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float hv[2];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const float g = __uint_as_float(gv[v * 8 + 2 * i + h]);
                                const float u = __uint_as_float(uv[v * 8 + 2 * i + h]);
                                hv[h] = g / (1.0f + __expf(-g)) * u;
                            }
                            o[i] = pack2(hv[0], hv[1]);
                        }
                        *reinterpret_cast<uint4*>(orow + col0 + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            uint32_t av[32];
            tmem_ld_32cols(tbase + c * 32, av);
            tmem_ld_wait();
            const int col0 = col_base + c * 32;
            if (row_ok) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    if (col0 + v * 8 < N) {
                        uint32_t o[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float a0 = __uint_as_float(av[v * 8 + 2 * i]);
                            float a1 = __uint_as_float(av[v * 8 + 2 * i + 1]);
                            if (MODE == kGemmReLU2) {
                                a0 = a0 > 0.f ? a0 * a0 : 0.f;
                                a1 = a1 > 0.f ? a1 * a1 : 0.f;
                            }
                            o[i] = pack2(a0, a1);
                        }
                        *reinterpret_cast<uint4*>(orow + col0 + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
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
    // Group rows.  Each bucket is clamped to [0, a_rows] on its own, so even
    // malformed offsets keep every row access inside A and the output.
    for (int g = tid; g < p.groups; g += C::THREADS) {
        if (p.offsets) {
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
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const Tile t = decode_tile(tile, prefix, rstart, rcount, p, ntn);
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
                    if (++stage == C::STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let copies already issued land before the CTA exits
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 1000000ull) { }
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
                const Tile t = decode_tile(tile, prefix, rstart, rcount, p, ntn);
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
            const Tile t = decode_tile(tile, prefix, rstart, rcount, p, ntn);
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
                __nv_bfloat16* orow = p.out + (size_t)(t.row0 + (row_ok ? r : 0)) * p.ldo +
                                      (size_t)t.g * p.out_group_col;
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

// Row-major [rows, cols] BF16, 64 x 128 boxes, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols) {
    auto enc = encode_fn();
    if (!enc) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, 128u};
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
    grouped_gemm_kernel<MODE, HALVES><<<device_sm_count(), Cfg<HALVES>::THREADS, smem, st>>>(ma, mb, kp);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) set_error("grouped GEMM launch (smem %zu): %s", smem, cudaGetErrorString(e));
    return e;
}

template <int HALVES>
size_t smem_bytes(int groups) {
    return 1024 + (size_t)Cfg<HALVES>::STAGES * Cfg<HALVES>::STAGE_BYTES + sizeof(SmemCtl<HALVES>) +
           3 * (size_t)(groups + 1) * 4;
}

}  // namespace

moe_status launch_grouped_gemm(const GemmProblem& g, WsHeader* hdr, cudaStream_t st) {
    if (g.groups < 1 || g.groups > 1024 || g.K < 1 || g.N < 1) {
        set_error("grouped GEMM: unsupported problem (groups %d, K %d, N %d)", g.groups, g.K, g.N);
        return MOE_ERR_UNSUPPORTED;
    }
    CUtensorMap ma, mb;
    if (!make_map(&ma, g.a, g.a_rows, g.a_cols)) return MOE_ERR_CUDA;
    if (!make_map(&mb, g.b, g.b_rows, g.b_cols)) return MOE_ERR_CUDA;
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
    kp.out = reinterpret_cast<__nv_bfloat16*>(g.out);
    kp.ldo = g.ldo;
    kp.out_group_col = g.out_group_col;
    kp.hdr = hdr;
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
            default: e = launch_mode<kGemmPlain, 2>(ma, mb, kp, smem, st); break;
        }
    } else {
        switch (g.mode) {
            case kGemmSwiGLU: e = launch_mode<kGemmSwiGLU, 1>(ma, mb, kp, smem, st); break;
            case kGemmReLU2: e = launch_mode<kGemmReLU2, 1>(ma, mb, kp, smem, st); break;
            default: e = launch_mode<kGemmPlain, 1>(ma, mb, kp, smem, st); break;
        }
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
