// dispatch.cu -- K2 (count + scan) and K3 (stable scatter): count-first dispatch.
//
// afdEP-comm count-first validation record (.change, and the fault patches P3
// "count puts" and P4 "FFN publishes prefix sums"): the per-expert counts and
// their prefix sums are known before any payload row moves, so every row is
// written once, straight into its expert-contiguous slot, and a capacity
// overflow is caught before the payload moves.
//
// K2 splits the R = T*k pairs into tiles of kCountChunk pairs (one block each,
// tile ids taken in launch order from a counter, so every predecessor tile is
// already running).  A block
//   1. validates its pairs (0 <= id < E, no duplicate earlier in the token),
//   2. ranks every valid pair among the earlier same-expert pairs of the tile
//      (warp __match_any_sync + popc, warps taken in order: stable in p),
//   3. publishes its E-vector of counts and runs a decoupled look-back over the
//      preceding tiles' published vectors (aggregate / inclusive flags packed
//      with the value in one 64-bit word), so each pair's rank inside its
//      expert = look-back prefix + in-tile rank,
//   4. if it is the last tile, holds the totals: writes counts, the exclusive
//      scan offsets[0..E], and the capacity verdict.
// K3 then places pair p at dest[p] = offsets[e] + rank[p] and copies the token
// row with 16-byte vectors: one read of x[t], k writes.
#include "common.cuh"

#include <mutex>

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kFlagAgg = 1ull << 32;
constexpr unsigned long long kFlagIncl = 2ull << 32;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Fresh look-back state for a dispatch: flags "not ready", tile counter 0 (a
// kernel rather than memsets, so the layer stays one chain of kernels).
__global__ void __launch_bounds__(256)
clear_lookback_kernel(unsigned long long* flags, long long n, WsHeader* hdr) {
    pdl_wait();
    pdl_trigger();
    const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (long long i = i0; i < n; i += (long long)gridDim.x * blockDim.x) flags[i] = 0ull;
    // normally 0; a test may start the ids at 1 (moe_workspace_set_wait)
    if (i0 == 0) hdr->tile_counter = hdr->count_tile_skip == 1 ? 1u : 0u;
}

// The test controls of a workspace's look-back wait, written in stream order.
__global__ void set_wait_kernel(WsHeader* hdr, unsigned long long lookback_wait_ns, int count_tile_skip) {
    pdl_wait();
    pdl_trigger();
    hdr->lookback_wait_ns = lookback_wait_ns;
    hdr->count_tile_skip = count_tile_skip;
}

__global__ void __launch_bounds__(kCountThreads)
count_kernel(long long R, int k, int E, int capacity, const int32_t* __restrict__ ids,
             int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ rank,
             unsigned long long* flags, int ntiles, WsHeader* hdr) {
    extern __shared__ int smem_i[];
    int* hist = smem_i;         // [E] in-tile counts
    int* excl = smem_i + E;     // [E] look-back prefix
    __shared__ unsigned tile_s;
    __shared__ int warp_tot[kCountThreads / 32];
    constexpr int kItems = kCountChunk / kCountThreads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_wait();
    pdl_trigger();
    // one tile: no look-back, so neither the counter nor the flags are read
    if (tid == 0) tile_s = ntiles == 1 ? 0u : atomicAdd(&hdr->tile_counter, 1u);
    for (int e = tid; e < E; e += kCountThreads) hist[e] = 0;
    __syncthreads();
    const unsigned tile = tile_s;
    if (tile >= (unsigned)ntiles) return;            // only with a skipped first tile
    const unsigned long long wait_ns = hdr->lookback_wait_ns ? hdr->lookback_wait_ns : kWaitLimitNs;
    const long long p0 = (long long)tile * kCountChunk;

    int item_e[kItems], item_r[kItems];
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const long long p = p0 + (long long)it * kCountThreads + tid;
        int e = -1;
        if (p < R) {
            const int id = ids[p];
            const long long t = p / k;
            const int j = (int)(p - t * k);
            bool ok = (id >= 0 && id < E);
            for (int jj = 0; jj < j && ok; ++jj)
                if (ids[t * k + jj] == id) ok = false;
            if (ok) e = id;
            else raise_status(hdr, MOE_ERR_INVALID_ROUTE);
        }
        const unsigned grp = __match_any_sync(kFull, e);
        const int lrank = __popc(grp & lanemask_lt());
        const bool leader = (lane == 31 - __clz(grp));
        int r = 0;
        // warps in order, so ranks follow p inside the tile
        for (int w = 0; w < kCountThreads / 32; ++w) {
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

    // publish this tile's counts: inclusive right away for tile 0, else aggregate
    unsigned long long* mine = flags + (size_t)tile * E;
    for (int e = tid; e < E; e += kCountThreads)
        st_release_u64(mine + e, (tile == 0 ? kFlagIncl : kFlagAgg) | (unsigned)hist[e]);

    // decoupled look-back, one expert column per thread
    for (int e = tid; e < E; e += kCountThreads) {
        int ex = 0;
        if (tile > 0) {
            long long j = (long long)tile - 1;
            unsigned long long t0 = 0;
            unsigned spins = 0;
            while (j >= 0) {
                const unsigned long long f = ld_acquire_u64(flags + (size_t)j * E + e);
                const unsigned long long st = f & 0xffffffff00000000ull;
                if (st == 0) {
                    if (++spins == 64) t0 = globaltimer_ns();
                    if (spins > 64 && (spins & 63u) == 0 && globaltimer_ns() - t0 > wait_ns) {
                        raise_status(hdr, MOE_ERR_TIMEOUT);
                        hdr->timeout_site = kSiteLookback;
                        break;
                    }
                    continue;
                }
                ex += (int)(unsigned)(f & 0xffffffffull);
                if (st == kFlagIncl) break;
                --j;
            }
            st_release_u64(mine + e, kFlagIncl | (unsigned)(ex + hist[e]));
        }
        excl[e] = ex;
    }
    __syncthreads();

#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const long long p = p0 + (long long)it * kCountThreads + tid;
        if (p < R) rank[p] = (item_e[it] >= 0) ? excl[item_e[it]] + item_r[it] : -1;
    }

    if (tile != (unsigned)ntiles - 1) return;
    // the last tile holds the totals: counts, offsets (exclusive scan), capacity
    const int per = (E + kCountThreads - 1) / kCountThreads;
    const int e0 = tid * per;
    int loc = 0;
    for (int i = 0; i < per; ++i)
        if (e0 + i < E) loc += excl[e0 + i] + hist[e0 + i];
    int inc = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(kFull, inc, off);
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
            const int c = excl[e] + hist[e];
            counts[e] = c;
            offsets[e] = run;
            if (c > capacity) over = 1;
            run += c;
        }
    }
    if (tid == kCountThreads - 1) offsets[E] = run;
    const int any_over = __syncthreads_or(over);
    if (tid == 0) {
        hdr->cap_exceeded = any_over;
        if (any_over) raise_status(hdr, MOE_ERR_CAPACITY);
    }
}

// One block per token row (grid-stride over tokens).  Threads < k place the
// pairs; every thread copies up to 4 16-byte chunks of the row per pass and
// stores each to the k destinations.
__global__ void __launch_bounds__(256)
scatter_kernel(int T, int HV, int k, int E, const uint4* __restrict__ x, const int32_t* __restrict__ ids,
               const int32_t* __restrict__ offsets, const int32_t* __restrict__ rank,
               int32_t* __restrict__ dest, int32_t* __restrict__ sorted_pair, uint4* __restrict__ x_perm,
               const WsHeader* hdr) {
    pdl_wait();
    pdl_trigger();
    if (hdr->cap_exceeded) return;                 // over capacity: no payload moves
    __shared__ int dsh[32];
    const long long R = (long long)T * k;
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (tid < k) {
            const long long p = (long long)t * k + tid;
            const int e = ids[p];
            const int r = rank[p];
            int d = -1;
            if (r >= 0 && e >= 0 && e < E) {
                const long long dd = (long long)offsets[e] + r;
                if (dd >= 0 && dd < R) d = (int)dd;
            }
            dest[p] = d;
            if (d >= 0) sorted_pair[d] = (int)p;
            dsh[tid] = d;
        }
        __syncthreads();
        const uint4* src = x + (size_t)t * HV;
        for (int c0 = tid; c0 < HV; c0 += 4 * nt) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * nt;
                if (c < HV) v[u] = __ldcs(src + c);
            }
            for (int j = 0; j < k; ++j) {
                const int d = dsh[j];
                if (d < 0) continue;
                uint4* dst = x_perm + (size_t)d * HV;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + u * nt;
                    if (c < HV) dst[c] = v[u];
                }
            }
        }
        __syncthreads();
    }
}

int row_threads(int HV) {
    int t = 32;
    while (t < 256 && t < HV) t *= 2;
    return t;
}

}  // namespace

cudaError_t launch_count(const moe_shape& s, const int32_t* ids, int32_t* counts, int32_t* offsets,
                         int32_t* rank, unsigned long long* flags, int count_tiles, WsHeader* hdr,
                         cudaStream_t st) {
    const long long R = (long long)s.tokens * s.top_k;
    // fresh look-back state: flags "not ready", tile counter 0 (a single tile
    // reads neither)
    if (count_tiles > 1) {
        const long long nflags = (long long)count_tiles * s.experts;
        long long cblocks = (nflags + 255) / 256;
        if (cblocks > device_sm_count()) cblocks = device_sm_count();
        const cudaError_t err = launch_kernel(clear_lookback_kernel, dim3((unsigned)cblocks), dim3(256), 0, st, 1,
                                              kUsePdl, flags, nflags, hdr);
        if (err != cudaSuccess) return err;
    }
    const size_t smem = (size_t)2 * s.experts * sizeof(int);
    return launch_kernel(count_kernel, dim3((unsigned)count_tiles), dim3(kCountThreads), smem, st, 1, kUsePdl, R,
                         s.top_k, s.experts, s.capacity, ids, counts, offsets, rank, flags, count_tiles, hdr);
}

cudaError_t launch_set_wait(WsHeader* hdr, unsigned long long lookback_wait_ns, int count_tile_skip, cudaStream_t st) {
    return launch_kernel(set_wait_kernel, dim3(1), dim3(1), 0, st, 1, kUsePdl, hdr, lookback_wait_ns, count_tile_skip);
}

cudaError_t launch_scatter(const moe_shape& s, const uint16_t* x, const int32_t* ids, const int32_t* offsets,
                           const int32_t* rank, int32_t* dest, int32_t* sorted_pair, uint16_t* x_perm,
                           WsHeader* hdr, cudaStream_t st) {
    const int HV = s.hidden / 8;
    const int threads = row_threads(HV);
    long long blocks = s.tokens;
    const long long cap = (long long)device_sm_count() * (2048 / threads);
    if (blocks > cap) blocks = cap;
    return launch_kernel(scatter_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, 1, kUsePdl, s.tokens, HV,
                         s.top_k, s.experts, reinterpret_cast<const uint4*>(x), ids, offsets, rank, dest, sorted_pair,
                         reinterpret_cast<uint4*>(x_perm), static_cast<const WsHeader*>(hdr));
}

}  // namespace moe

// ---------------------------------------------------------------------------
// moe_dispatch_noalloc: the same count-first dispatch for callers that cannot
// allocate device memory.  Its scratch -- the status header, the per-pair
// ranks and the look-back flags that moe_dispatch keeps in the caller's
// workspace -- lives in one file-scope device array of fixed size instead.
// Every GPU that loads this library holds that array until the process exits.
// ---------------------------------------------------------------------------
namespace moe {
namespace {
constexpr long long kNoAllocMaxPairs = 131072;                      // T * k limit
constexpr int kNoAllocMaxExperts = 1024;
constexpr size_t kNoAllocHdrBytes = 4096;
constexpr size_t kNoAllocRankBytes = (size_t)kNoAllocMaxPairs * 4;  // 512 KiB
constexpr size_t kNoAllocFlagBytes =                                // 1 MiB
    (size_t)((kNoAllocMaxPairs + kCountChunk - 1) / kCountChunk) * kNoAllocMaxExperts * 8;
constexpr size_t kNoAllocBytes = kNoAllocHdrBytes + kNoAllocRankBytes + kNoAllocFlagBytes;
}  // namespace
}  // namespace moe

static __device__ __align__(256) unsigned char g_noalloc_scratch[moe::kNoAllocBytes];

namespace moe {
namespace {
// Device address of g_noalloc_scratch per device, looked up once per device
// with that device current (the host-side name is only a stand-in).
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[64] = {nullptr};

moe_status noalloc_scratch(unsigned char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        set_error("moe_dispatch_noalloc: no usable current CUDA device");
        return MOE_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            set_error("moe_dispatch_noalloc: cudaGetSymbolAddress of the static scratch failed: %s",
                      cudaGetErrorString(e));
            return MOE_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace
}  // namespace moe

extern "C" moe_status moe_dispatch_noalloc(const moe_shape* shape, const uint16_t* x, const int32_t* topk_ids,
                                           int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* sorted_pair,
                                           uint16_t* x_perm, int32_t* device_status, void* stream) {
    using namespace moe;
    clear_error();
    moe_status r = validate_shape(shape);
    if (r != MOE_OK) return r;
    if (!al16(x) || !al16(topk_ids) || !al16(counts) || !al16(offsets) || !al16(dest) || !al16(sorted_pair) ||
        !al16(x_perm) || (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)))
        return MOE_ERR_INVALID_ARG;
    const long long R = (long long)shape->tokens * shape->top_k;
    if (R > kNoAllocMaxPairs) {
        set_error("moe_dispatch_noalloc: %lld pairs (tokens x top_k) exceed the static scratch limit of %lld",
                  R, kNoAllocMaxPairs);
        return MOE_ERR_UNSUPPORTED;
    }
    unsigned char* base = nullptr;
    if ((r = noalloc_scratch(&base)) != MOE_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(base);
    int32_t* rank = reinterpret_cast<int32_t*>(base + kNoAllocHdrBytes);
    unsigned long long* flags = reinterpret_cast<unsigned long long*>(base + kNoAllocHdrBytes + kNoAllocRankBytes);
    const int tiles = (int)((R + kCountChunk - 1) / kCountChunk);
    // the array keeps the previous call's contents: start from a clear header
    // (status, timeout site, tile counter, capacity verdict); launch_count
    // clears the look-back flags it uses
    cudaError_t e = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st);
    if (e == cudaSuccess) e = launch_count(*shape, topk_ids, counts, offsets, rank, flags, tiles, hdr, st);
    if (e == cudaSuccess) e = launch_scatter(*shape, x, topk_ids, offsets, rank, dest, sorted_pair, x_perm, hdr, st);
    if (e == cudaSuccess && device_status)
        e = cudaMemcpyAsync(device_status, &hdr->status, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) {
        set_error("moe_dispatch_noalloc: %s", cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
