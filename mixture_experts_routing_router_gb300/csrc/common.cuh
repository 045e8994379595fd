// common.cuh -- shared definitions of the libmoe.so CUDA sources (sm_103a only):
// the workspace layout, the device status word, bounded waits, and thin inline-PTX
// wrappers for mbarrier, TMA (cp.async.bulk.tensor) and tcgen05 (MMA / TMEM).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/moe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libmoe targets sm_103a (Blackwell tcgen05/TMEM); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace moe {

// ---------------------------------------------------------------------------
// Workspace.  A caller-owned device buffer; regions are 1 KiB aligned.
// The first 4 KiB hold the header below; the count kernel's look-back flags,
// the per-pair ranks and the shared-expert activations follow (needed by the
// stage calls); the whole-layer intermediates come last (moe_layer only).
// ---------------------------------------------------------------------------
struct WsHeader {
    int status;             // sticky: atomicMax of every device-raised moe_status
    int timeout_site;       // which bounded wait gave up (diagnostic)
    unsigned tile_counter;  // dynamic tile ids of the count kernel (reset per dispatch)
    int cap_exceeded;       // this dispatch's capacity verdict (written by the count kernel)
    // test controls (moe_workspace_set_wait); zero = normal operation
    unsigned long long lookback_wait_ns;   // look-back give-up time; 0 = kWaitLimitNs
    int count_tile_skip;                   // first tile id the count kernel hands out (0 or 1)
    unsigned route_ready;                  // moe_layer: 1 once the fused dispatch has written the bucket
                                           // bounds and the capacity verdict; 0 again after the combine
};

constexpr int kCountChunk = 1024;      // pairs per count tile (one 256-thread block)
constexpr int kCountThreads = 256;
constexpr size_t kAlign = 1024;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct WsLayout {
    size_t hdr, flags, rank, h_shared;        // stage regions
    size_t stage_end;                         // bytes the stage calls need
    size_t counts, offsets, ids, w, dest, sorted_pair, x_perm, h, y_perm, y_shared;
    size_t sync;                              // moe_layer's fused decode FFN: its counters
    size_t total;                             // bytes moe_layer needs
    int count_tiles;
};

inline WsLayout ws_layout(const moe_shape& s) {
    WsLayout L{};
    const size_t T = (size_t)s.tokens, H = (size_t)s.hidden, E = (size_t)s.experts;
    const size_t R = T * (size_t)s.top_k, I = (size_t)s.inter;
    L.count_tiles = (int)((R + kCountChunk - 1) / kCountChunk);
    size_t o = 0;
    L.hdr = o;          o = align_up(o + 4096, kAlign);
    L.flags = o;        o = align_up(o + (size_t)L.count_tiles * E * 8, kAlign);
    L.rank = o;         o = align_up(o + R * 4, kAlign);
    L.h_shared = o;     o = align_up(o + T * (size_t)s.shared * (size_t)s.shared_inter * 2, kAlign);
    L.stage_end = o;
    L.counts = o;       o = align_up(o + E * 4, kAlign);
    L.offsets = o;      o = align_up(o + (E + 1) * 4, kAlign);
    L.ids = o;          o = align_up(o + R * 4, kAlign);
    L.w = o;            o = align_up(o + R * 4, kAlign);
    L.dest = o;         o = align_up(o + R * 4, kAlign);
    L.sorted_pair = o;  o = align_up(o + R * 4, kAlign);
    L.x_perm = o;       o = align_up(o + R * H * 2, kAlign);
    L.h = o;            o = align_up(o + R * I * 2, kAlign);
    L.y_perm = o;       o = align_up(o + R * H * 2, kAlign);
    L.y_shared = o;     o = align_up(o + (s.shared > 0 ? T * H * 2 : 0), kAlign);
    L.sync = o;         o = align_up(o + (E + 4 * ((H + 127) / 128) + 1) * 4, kAlign);
    L.total = o;
    return L;
}

// Bounded waits give up after this long and raise MOE_ERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s
// How long the up projection looks for the fused dispatch's published bucket
// bounds before it falls back to the programmatic wait (not an error).
constexpr unsigned long long kEarlyWaitNs = 200000ull;       // 200 us

// Where a bounded wait gave up (WsHeader::timeout_site).
enum TimeoutSite : int {
    kSiteNone = 0, kSiteLookback = 1, kSiteGemmProducer = 2, kSiteGemmMma = 3, kSiteGemmEpilogue = 4,
    kSiteGemmDecode = 5, kSiteDecodeFfn = 6,
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_status(WsHeader* h, int code) { atomicMax(&h->status, code); }

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 64-bit release store / acquire load at GPU scope (the look-back flags).
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Wait until the phase with parity `parity` of barrier `bar` has completed.
// Gives up (returns false) when *abort is set by another role of the CTA, or
// after kWaitLimitNs, in which case it sets *abort itself.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) { *abort = 1; return false; }
        }
    }
}

// After a TMA producer gave up: wait (bounded, on a never-set abort flag of its
// own) for the full-barrier phases of the last stages it armed, so that no bulk
// copy it issued is still writing this CTA's shared memory when the CTA exits.
// `armed` counts the stages armed since the kernel began; the ring has `stages`
// slots whose full barriers are 8 bytes apart from `full0`.  Returns false if
// some phase did not complete within the limit.
__device__ __forceinline__ bool wait_armed_stages(uint32_t full0, int stages, long long armed) {
    volatile int never = 0;
    bool all = true;
    for (long long j = armed > stages ? armed - stages : 0; j < armed; ++j) {
        const uint32_t bar = full0 + 8u * (uint32_t)(j % stages);
        if (!mbar_wait_bounded(bar, (uint32_t)((j / stages) & 1), &never)) all = false;
    }
    return all;
}

// Last resort after wait_armed_stages failed: a fixed 1 ms delay.
__device__ __forceinline__ void settle_delay() {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) { }
}

// ---- programmatic dependent launch ----------------------------------------------
// Every kernel of the library runs: a prologue that touches no memory another
// kernel writes (barrier init, TMEM allocation, descriptor prefetch), then
// pdl_wait() -- which returns once the preceding kernel in the stream has
// completed and its writes are visible -- then pdl_trigger(), which lets the
// next kernel's CTAs start their own prologue as SMs free up.  No kernel
// triggers before its wait returns, so when a kernel passes its wait every
// earlier kernel of the stream has completed.  Without a programmatic
// dependency (or launched plainly) both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- TMA --------------------------------------------------------------------
// 2-D tiled bulk tensor load global -> shared, completion counted on `bar`.
// (x, y) = (inner element index, row index); x * 2 bytes is a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y) : "memory");
}
// 3-D / 5-D tiled loads: coordinates innermost first.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z, int w,
                                            int v) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v)
        : "memory");
}
// 4-D tiled load: coordinates (x, y, z, w), innermost first.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---- tcgen05 / TMEM -----------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, BF16 inputs, FP32 accumulator.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// 32 consecutive FP32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 16 consecutive FP32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- CTA pairs (cluster of 2) ------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on an mbarrier that may live in the peer CTA (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (the leader's, for the pair MMA).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, uint32_t bar_cluster, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const void* tmap, uint32_t bar_cluster, int x, int y,
                                                 int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}
// Pair-wide TMEM allocation: one warp of each CTA of the pair executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T, issued by the leader CTA.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive once on the mbarrier at offset `bar` in every CTA of `mask` when the
// pair MMAs issued so far by this thread are done.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(bar), "h"(mask) : "memory");
}
// Local (non-multicast) commit of the pair MMAs issued so far by this thread.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 64 BF16 (128 B), 8-row swizzle atoms of 1 KiB stacked densely
// (stride byte offset 1 KiB); the tile starts on a 1 KiB boundary.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);       // bits  0-13: start address >> 4
    d |= (uint64_t)1u << 16;                        // bits 16-29: leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;              // bits 32-45: stride byte offset >> 4
    d |= (uint64_t)1u << 46;                        // bits 46-47: descriptor version 1
    d |= (uint64_t)2u << 61;                        // bits 61-63: 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: BF16 A and B (both K-major), FP32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                               // D format: F32
         | (1u << 7)                               // A format: BF16
         | (1u << 10)                              // B format: BF16
         | ((uint32_t)(N >> 3) << 17)              // N >> 3
         | ((uint32_t)(M >> 4) << 24);             // M >> 4
}

// ---- weight decoders (FP8 E4M3, NVFP4 E2M1) to BF16 ---------------------------
// Four E4M3 codes (bytes 0..3 of w) -> four BF16 values, exact, in integer and
// one BF16 multiply per pair: prmt spreads two codes into 16-bit halves with
// the sign byte replicated above each ([S|b]); shifting left 4 and masking
// with 0x87F0 per half leaves the sign at bit 15 and the code's 7 exponent and
// mantissa bits at bits 4..10 -- a BF16 whose exponent field is the E4M3
// exponent field (bias 127 instead of 7) -- and multiplying by 2^120 rebiases
// it.  An E4M3 subnormal (exponent field 0) is then a BF16 subnormal m*2^-129,
// and the same multiply gives m*2^-9 exactly.  Out: lo = (b0, b1), hi = (b2, b3),
// low half first.  The E4M3 NaN codes (S.1111.111) are not valid weights; they
// decode to +-480 here.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    constexpr uint32_t kTwo120 = 0x7B807B80u;                 // (2^120, 2^120) in BF16
    uint32_t t0, t1;
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w));  // [S1 b1 S0 b0]
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w));  // [S3 b3 S2 b2]
    t0 = (t0 << 4) & 0x87F087F0u;
    t1 = (t1 << 4) & 0x87F087F0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(t0), "r"(kTwo120));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(t1), "r"(kTwo120));
}

// Eight E2M1 codes (the nibbles of w, element 0 in the low nibble) times a
// block scale -> four BF16 pairs (elements 2j, 2j+1 in out[j], low half
// first), exact.  The codes are split into even and odd elements, one per
// byte; prmt places element 2j in the low and 2j+1 in the high 16-bit half
// (zero bytes from the sign-replicate selector on a byte below 0x80), and the
// multiply by 0x1040 adds the copies shifted by 6 and by 12 (disjoint bits),
// so the mask keeps the code's exponent and mantissa bits at bits 6..8 and
// its sign at bit 15 of each half: the BF16 number e2m1 * 2^-126 (subnormal
// for exponent field 0, where E2M1 is 0 or 0.5, exactly as E2M1 defines it).
// m = (s, s) with s = block scale * 2^126 * 2^-8 finishes the value in one
// BF16 multiply: at most 2 + 4 significant bits, within the normal range.
__device__ __forceinline__ void e2m1x8_to_bf16x8(uint32_t w, uint32_t m, uint32_t* out) {
    const uint32_t ev = w & 0x0F0F0F0Fu;                      // elements 0, 2, 4, 6
    const uint32_t od = (w >> 4) & 0x0F0F0F0Fu;               // elements 1, 3, 5, 7
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t t;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(ev), "r"(od), "r"(0x8480u + 0x0101u * (uint32_t)j));
        t = (t * 0x1040u) & 0x81C081C0u;
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out[j]) : "r"(t), "r"(m));
    }
}

// ---------------------------------------------------------------------------
// Host-side launchers (one per translation unit); all return cudaError_t of the launch.
// ---------------------------------------------------------------------------
cudaError_t launch_route(const moe_shape& s, const float* logits, int32_t* ids, float* w,
                         WsHeader* hdr, cudaStream_t st);
cudaError_t launch_route_sigmoid(const moe_shape& s, const float* logits, const float* bias, float scale,
                                 int32_t* ids, float* w, WsHeader* hdr, cudaStream_t st);
cudaError_t launch_count(const moe_shape& s, const int32_t* ids, int32_t* counts, int32_t* offsets,
                         int32_t* rank, unsigned long long* flags, int count_tiles,
                         WsHeader* hdr, cudaStream_t st);
cudaError_t launch_scatter(const moe_shape& s, const uint16_t* x, const int32_t* ids,
                           const int32_t* offsets, const int32_t* rank, int32_t* dest,
                           int32_t* sorted_pair, uint16_t* x_perm, WsHeader* hdr, cudaStream_t st);
// Route (when logits is not null; else take ids_in), count and scatter in one
// kernel for batches of at most kSmallDispatchTokens tokens; results bitwise
// those of launch_route + launch_count + launch_scatter.  `sync` (nsync
// words, or null): counters of the fused decode FFN that follows, zeroed
// before the bucket bounds are published.
constexpr int kSmallDispatchTokens = 16;
cudaError_t launch_small_dispatch(const moe_shape& s, const float* logits, const int32_t* ids_in, int32_t* ids_out,
                                  float* w_out, const uint16_t* x, int32_t* counts, int32_t* offsets, int32_t* dest,
                                  int32_t* sorted_pair, uint16_t* x_perm, WsHeader* hdr, unsigned* sync, int nsync,
                                  cudaStream_t st);
// moe_layer at decode: the expert FFN (up, down) and the weighted combine in
// one persistent launch after the fused dispatch (decode_ffn.cu), for shapes
// decode_ffn_fits accepts; `sync` is the workspace's counter region
// (decode_ffn_sync_words words), zeroed by that dispatch.
bool decode_ffn_fits(const moe_shape& s);
size_t decode_ffn_sync_words(const moe_shape& s);
moe_status launch_decode_ffn(const moe_shape& s, const uint16_t* x_perm, const int32_t* offsets,
                             const uint16_t* w13, const uint16_t* w2, uint16_t* h, uint16_t* y_perm,
                             const int32_t* dest, const float* topk_w, const uint16_t* residual, uint16_t* out,
                             unsigned* sync, WsHeader* hdr, cudaStream_t st);
// gate: NULL, or (inside moe_layer) the workspace header whose capacity verdict,
// when set, makes the kernel leave `out` untouched; the kernel also puts the
// header's route_ready back to 0 for the next layer call.
cudaError_t launch_combine(const moe_shape& s, const uint16_t* y_perm, const int32_t* dest,
                           const float* w, const uint16_t* y_shared, const uint16_t* residual, uint16_t* out,
                           WsHeader* gate, cudaStream_t st);
// The test controls of the look-back wait (moe_workspace_set_wait).
cudaError_t launch_set_wait(WsHeader* hdr, unsigned long long lookback_wait_ns, int count_tile_skip,
                            cudaStream_t st);

// Launch with programmatic stream serialization (the kernel may start while
// the preceding kernel of the stream finishes; it waits in pdl_wait), and an
// optional cluster of `cluster_x` CTAs.
constexpr bool kUsePdl = true;
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          unsigned cluster_x, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Grouped GEMM problem (one launch): for every group g and row r of the group,
// out[row0(g) + r, g*out_group_col + n] = epilogue( sum_seg sum_k A[row0(g)+r, seg*a_seg_col + k]
//                                                   * B[g*b_group_rows + seg*b_seg_row + n', k] )
// SwiGLU / ReLU^2 / plain store BF16; F32 stores the FP32 accumulator (router logits).
enum GemmMode : int { kGemmSwiGLU = 0, kGemmReLU2 = 1, kGemmPlain = 2, kGemmF32 = 3 };
struct GemmProblem {
    int mode;
    const void* a; long long a_rows; long long a_cols;    // A [a_rows, a_cols] bf16
    const void* b; long long b_rows; long long b_cols;    // B [b_rows, b_cols] bf16
    const int32_t* offsets;                               // [G+1] row bounds, or null
    int groups;
    int rows_all;                                         // rows per group when offsets == null
    int K, nseg, a_seg_col, b_seg_row;
    int N;                                                // output columns per group
    int b_group_rows;
    int up_off;                                           // SwiGLU: rows from gate to up half
    void* out; long long ldo; int out_group_col;
    int max_group_rows;                                   // host bound on rows per group (0: a_rows)
    int wfmt;                                             // B's format: kWeightBf16 / Fp8E4M3 / Nvfp4
    const float* wscale;                                  // FP8, NVFP4: FP32 scale per B row
    const uint8_t* bscale;                                // NVFP4: E4M3 scale per 16 K elements
    long long bscale_stride;                              // NVFP4: bytes per B row of bscale
    int gated;                                            // 1: do nothing if this layer's dispatch
                                                          //    exceeded the capacity (hdr->cap_exceeded)
    // Small-row kernel only (moe_layer): 1 = the bucket bounds are final when the
    // kernel starts (the down projection); 2 = the fused dispatch publishes them
    // in hdr->route_ready (the up projection after it); 0 = neither (any caller).
    int early;
};
constexpr int kWeightBf16 = 0;
constexpr int kWeightFp8E4M3 = 1;   // one E4M3 code per element (b_cols bytes per row)
constexpr int kWeightNvfp4 = 2;     // two E2M1 codes per byte, low nibble first (b_cols / 2 bytes per row)
// Returns MOE_OK, MOE_ERR_CUDA (tensor map / launch) or MOE_ERR_UNSUPPORTED.
// Problems whose groups hold at most kDecodeRows rows and whose work fits in
// about two waves run the small-row kernel (launch_decode_gemm); the rest the
// tile kernels.
moe_status launch_grouped_gemm(const GemmProblem& p, WsHeader* hdr, cudaStream_t st);

// Small-row form: weights on the MMA's M side, nb (16..kDecodeRows, a
// multiple of 16) activation rows per chunk on its N side.
constexpr int kDecodeRows = 64;
moe_status launch_decode_gemm(const GemmProblem& p, int nb, WsHeader* hdr, cudaStream_t st);

// Tensor map of a row-major [rows, cols] BF16 matrix, 128-byte swizzle, boxes
// of 64 columns x box_rows rows (records the failure for moe_last_error_message).
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, long long rows, long long cols, unsigned box_rows);
// [rows, cols] BF16 with cols a multiple of 64, as (column in chunk, row, chunk):
// a box of `chunks` 64-column chunks of box_rows rows lands as that many
// 128-byte swizzled [box_rows x 64] tiles, one after the other; chunks past the
// last read zeros.
bool make_tensor_map_bf16_chunks(CUtensorMap* m, const void* base, long long rows, long long cols, unsigned box_rows,
                                 unsigned chunks);
// SwiGLU weights [groups x (half_rows gate | half_rows up), cols] as (column in
// chunk, row in half, half, group, chunk): per chunk a box lands as box_rows
// gate rows, then the up rows of the same output columns.
bool make_tensor_map_glu_chunks(CUtensorMap* m, const void* base, long long rows, long long cols, long long half_rows,
                                long long group_rows, unsigned box_rows, unsigned chunks);
// Tensor map of a [rows, cols] byte matrix with row stride `stride` bytes (a
// multiple of 16; FP8 / NVFP4 codes, NVFP4 block scales), boxes of box_cols
// bytes x box_rows rows; 128-byte boxes are 128-byte swizzled, others not.
bool make_tensor_map_u8_rows(CUtensorMap* m, const void* base, long long rows, long long cols, long long stride,
                             unsigned box_cols, unsigned box_rows);

int device_sm_count();

// The host-side shape checks every entry point applies (MOE_OK when valid).
moe_status validate_shape(const moe_shape* s);

// Record a host-side failure description for moe_last_error_message (this thread).
void set_error(const char* fmt, ...);
void clear_error();

}  // namespace moe
