// api.cu -- the extern "C" entry points of libmoe.so declared in include/moe.h:
// host-side validation (errors returned at once, nothing launched), workspace
// carving, and the kernel sequence of each call on the caller's stream.
#include "common.cuh"

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

namespace moe {

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (dev < 0 || dev >= 64) dev = 0;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 152;
    }
    return cache[dev];
}

namespace {
thread_local char g_last_error[512] = "";
}  // namespace

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

void clear_error() { g_last_error[0] = 0; }

namespace {

bool aligned(const void* p, uintptr_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool aligned_or_null(const void* p, uintptr_t a) { return p == nullptr || aligned(p, a); }

moe_status check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->tokens < 1 || s->hidden < 8 || s->hidden % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (s->experts < 1 || s->experts > 1024) return MOE_ERR_INVALID_ARG;
    if (s->top_k < 1 || s->top_k > 32 || s->top_k > s->experts) return MOE_ERR_INVALID_ARG;
    if (s->inter < 8 || s->inter % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (s->shared < 0 || s->shared > 64) return MOE_ERR_INVALID_ARG;
    if (s->shared > 0 && (s->shared_inter < 8 || s->shared_inter % 8 != 0)) return MOE_ERR_INVALID_ARG;
    if (s->capacity < 1) return MOE_ERR_INVALID_ARG;
    if (s->act != MOE_ACT_SWIGLU && s->act != MOE_ACT_RELU2) return MOE_ERR_INVALID_ARG;
    // every row / slot index must fit in int32
    const long long R = (long long)s->tokens * s->top_k;
    const long long up = (s->act == MOE_ACT_SWIGLU ? 2LL : 1LL) * s->inter;
    if (R > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if ((long long)s->experts * up > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if ((long long)s->experts * s->hidden > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (s->shared > 0 && (long long)s->shared * s->hidden > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status check_ws(const moe_shape* s, const void* ws, size_t ws_bytes, bool whole_layer) {
    if (!aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*s);
    if (ws_bytes < (whole_layer ? L.total : L.stage_end)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

moe_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    if (g_last_error[0] == 0) set_error("%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

int up_rows(const moe_shape& s, int inter) { return (s.act == MOE_ACT_SWIGLU ? 2 : 1) * inter; }

// A layer call that failed to launch a kernel after its fused dispatch never
// reaches the combine that puts route_ready back to 0: do it here, so the next
// call's up projection cannot take this call's published bucket bounds.
void reset_route_ready(void* ws, cudaStream_t st) {
    cudaMemsetAsync(&at<WsHeader>(ws, 0)->route_ready, 0, sizeof(unsigned), st);
}

// ---- the stage bodies (arguments already validated) --------------------------
moe_status do_route(const moe_shape& s, const float* logits, int32_t* ids, float* w, void* ws, cudaStream_t st) {
    return from_cuda(launch_route(s, logits, ids, w, at<WsHeader>(ws, 0), st));
}

moe_status do_dispatch(const moe_shape& s, const uint16_t* x, const int32_t* ids, int32_t* counts, int32_t* offsets,
                       int32_t* dest, int32_t* sorted_pair, uint16_t* x_perm, void* ws, cudaStream_t st) {
    const WsLayout L = ws_layout(s);
    WsHeader* hdr = at<WsHeader>(ws, 0);
    int32_t* rank = at<int32_t>(ws, L.rank);
    cudaError_t e = launch_count(s, ids, counts, offsets, rank, at<unsigned long long>(ws, L.flags), L.count_tiles,
                                 hdr, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(launch_scatter(s, x, ids, offsets, rank, dest, sorted_pair, x_perm, hdr, st));
}

// `gated` (moe_layer): the GEMMs and the combine skip their work when this
// call's dispatch found a bucket over capacity, so no output is touched.
moe_status do_up(const moe_shape& s, const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w13,
                 const uint16_t* x, const uint16_t* ws13, uint16_t* h, void* ws, cudaStream_t st,
                 bool gated = false, int early = 0) {
    const WsLayout L = ws_layout(s);
    WsHeader* hdr = at<WsHeader>(ws, 0);
    const long long R = (long long)s.tokens * s.top_k;
    const int mode = s.act == MOE_ACT_SWIGLU ? kGemmSwiGLU : kGemmReLU2;
    GemmProblem g{};
    g.mode = mode;
    g.a = x_perm; g.a_rows = R; g.a_cols = s.hidden;
    g.b = w13; g.b_rows = (long long)s.experts * up_rows(s, s.inter); g.b_cols = s.hidden;
    g.offsets = offsets; g.groups = s.experts; g.rows_all = 0;
    g.K = s.hidden; g.nseg = 1; g.a_seg_col = 0; g.b_seg_row = 0;
    g.N = s.inter; g.b_group_rows = up_rows(s, s.inter); g.up_off = s.inter;
    g.out = h; g.ldo = s.inter; g.out_group_col = 0;
    g.max_group_rows = s.tokens;   // a token's k experts are distinct
    g.gated = gated;
    g.early = early;
    moe_status r = launch_grouped_gemm(g, hdr, st);
    if (r != MOE_OK || s.shared == 0) return r;
    GemmProblem q{};
    const int Is = s.shared_inter;
    q.mode = mode;
    q.a = x; q.a_rows = s.tokens; q.a_cols = s.hidden;
    q.b = ws13; q.b_rows = (long long)s.shared * up_rows(s, Is); q.b_cols = s.hidden;
    q.offsets = nullptr; q.groups = s.shared; q.rows_all = s.tokens;
    q.K = s.hidden; q.nseg = 1; q.a_seg_col = 0; q.b_seg_row = 0;
    q.N = Is; q.b_group_rows = up_rows(s, Is); q.up_off = Is;
    q.out = at<uint16_t>(ws, L.h_shared); q.ldo = (long long)s.shared * Is; q.out_group_col = Is;
    q.gated = gated;
    return launch_grouped_gemm(q, hdr, st);
}

moe_status do_down(const moe_shape& s, const uint16_t* h, const int32_t* offsets, const uint16_t* w2,
                   const uint16_t* ws2, uint16_t* y_perm, uint16_t* y_shared, void* ws, cudaStream_t st,
                   bool gated = false, int early = 0) {
    const WsLayout L = ws_layout(s);
    WsHeader* hdr = at<WsHeader>(ws, 0);
    const long long R = (long long)s.tokens * s.top_k;
    GemmProblem g{};
    g.mode = kGemmPlain;
    g.a = h; g.a_rows = R; g.a_cols = s.inter;
    g.b = w2; g.b_rows = (long long)s.experts * s.hidden; g.b_cols = s.inter;
    g.offsets = offsets; g.groups = s.experts; g.rows_all = 0;
    g.K = s.inter; g.nseg = 1; g.a_seg_col = 0; g.b_seg_row = 0;
    g.N = s.hidden; g.b_group_rows = s.hidden; g.up_off = 0;
    g.out = y_perm; g.ldo = s.hidden; g.out_group_col = 0;
    g.max_group_rows = s.tokens;
    g.gated = gated;
    g.early = early;
    moe_status r = launch_grouped_gemm(g, hdr, st);
    if (r != MOE_OK || s.shared == 0) return r;
    // all shared experts in one accumulation: K runs over (s, n), so their sum
    // is rounded to BF16 once
    const int Is = s.shared_inter;
    GemmProblem q{};
    q.mode = kGemmPlain;
    q.a = at<uint16_t>(ws, L.h_shared); q.a_rows = s.tokens; q.a_cols = (long long)s.shared * Is;
    q.b = ws2; q.b_rows = (long long)s.shared * s.hidden; q.b_cols = Is;
    q.offsets = nullptr; q.groups = 1; q.rows_all = s.tokens;
    q.K = Is; q.nseg = s.shared; q.a_seg_col = Is; q.b_seg_row = s.hidden;
    q.N = s.hidden; q.b_group_rows = 0; q.up_off = 0;
    q.out = y_shared; q.ldo = s.hidden; q.out_group_col = 0;
    q.gated = gated;
    return launch_grouped_gemm(q, hdr, st);
}

// FP8 E4M3 or NVFP4 expert weights (no shared experts): one FP32 scale per
// weight row; NVFP4 adds the E4M3 block scales (16 bytes per 256 elements of a row).
size_t nvfp4_bscale_stride(int K) { return 16 * (size_t)((K + 255) / 256); }

moe_status do_up_q(const moe_shape& s, const uint16_t* x_perm, const int32_t* offsets, const uint8_t* w13,
                   const uint8_t* b13, const float* s13, int wfmt, uint16_t* h, void* ws, cudaStream_t st,
                   bool gated = false, int early = 0) {
    const long long R = (long long)s.tokens * s.top_k;
    GemmProblem g{};
    g.mode = s.act == MOE_ACT_SWIGLU ? kGemmSwiGLU : kGemmReLU2;
    g.a = x_perm; g.a_rows = R; g.a_cols = s.hidden;
    g.b = w13; g.b_rows = (long long)s.experts * up_rows(s, s.inter); g.b_cols = s.hidden;
    g.offsets = offsets; g.groups = s.experts; g.rows_all = 0;
    g.K = s.hidden; g.nseg = 1; g.a_seg_col = 0; g.b_seg_row = 0;
    g.N = s.inter; g.b_group_rows = up_rows(s, s.inter); g.up_off = s.inter;
    g.out = h; g.ldo = s.inter; g.out_group_col = 0;
    g.max_group_rows = s.tokens;
    g.wfmt = wfmt; g.wscale = s13;
    g.bscale = b13; g.bscale_stride = (long long)nvfp4_bscale_stride(s.hidden);
    g.gated = gated;
    g.early = early;
    return launch_grouped_gemm(g, at<WsHeader>(ws, 0), st);
}

moe_status do_down_q(const moe_shape& s, const uint16_t* h, const int32_t* offsets, const uint8_t* w2,
                     const uint8_t* b2, const float* s2, int wfmt, uint16_t* y_perm, void* ws, cudaStream_t st,
                     bool gated = false, int early = 0) {
    const long long R = (long long)s.tokens * s.top_k;
    GemmProblem g{};
    g.mode = kGemmPlain;
    g.a = h; g.a_rows = R; g.a_cols = s.inter;
    g.b = w2; g.b_rows = (long long)s.experts * s.hidden; g.b_cols = s.inter;
    g.offsets = offsets; g.groups = s.experts; g.rows_all = 0;
    g.K = s.inter; g.nseg = 1; g.a_seg_col = 0; g.b_seg_row = 0;
    g.N = s.hidden; g.b_group_rows = s.hidden; g.up_off = 0;
    g.out = y_perm; g.ldo = s.hidden; g.out_group_col = 0;
    g.max_group_rows = s.tokens;
    g.wfmt = wfmt; g.wscale = s2;
    g.bscale = b2; g.bscale_stride = (long long)nvfp4_bscale_stride(s.inter);
    g.gated = gated;
    g.early = early;
    return launch_grouped_gemm(g, at<WsHeader>(ws, 0), st);
}

// Quantized weight rows are TMA-loaded: their byte stride (H or I for FP8,
// half that for NVFP4) must be a multiple of 16; shared experts are not part
// of the quantized entry points.
moe_status check_quant_shape(const moe_shape* s, int wfmt) {
    const char* name = wfmt == kWeightNvfp4 ? "NVFP4" : "FP8";
    const int mult = wfmt == kWeightNvfp4 ? 32 : 16;
    if (s->shared > 0) {
        set_error("%s expert weights: shared experts are not supported (shape.shared must be 0)", name);
        return MOE_ERR_UNSUPPORTED;
    }
    if (s->hidden % mult != 0 || s->inter % mult != 0) {
        set_error("%s expert weights: hidden and inter must be multiples of %d (got %d, %d)", name, mult, s->hidden,
                  s->inter);
        return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

moe_status do_combine(const moe_shape& s, const uint16_t* y_perm, const int32_t* dest, const float* w,
                      const uint16_t* y_shared, const uint16_t* residual, uint16_t* out, cudaStream_t st,
                      WsHeader* gate = nullptr) {
    return from_cuda(launch_combine(s, y_perm, dest, w, y_shared, residual, out, gate, st));
}

moe_status expert_up_q(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets, const uint8_t* w13,
                       const uint8_t* w13_bscale, const float* w13_scale, int wfmt, uint16_t* h, void* ws,
                       size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_quant_shape(shape, wfmt)) != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(x_perm, 16) || !aligned(offsets, 16) || !aligned(w13, 16) || !aligned(w13_scale, 16) ||
        !aligned(h, 16) || (wfmt == kWeightNvfp4 && !aligned(w13_bscale, 16)))
        return MOE_ERR_INVALID_ARG;
    return do_up_q(*shape, x_perm, offsets, w13, w13_bscale, w13_scale, wfmt, h, ws,
                   static_cast<cudaStream_t>(stream));
}

moe_status expert_down_q(const moe_shape* shape, const uint16_t* h, const int32_t* offsets, const uint8_t* w2,
                         const uint8_t* w2_bscale, const float* w2_scale, int wfmt, uint16_t* y_perm, void* ws,
                         size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_quant_shape(shape, wfmt)) != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(h, 16) || !aligned(offsets, 16) || !aligned(w2, 16) || !aligned(w2_scale, 16) ||
        !aligned(y_perm, 16) || (wfmt == kWeightNvfp4 && !aligned(w2_bscale, 16)))
        return MOE_ERR_INVALID_ARG;
    return do_down_q(*shape, h, offsets, w2, w2_bscale, w2_scale, wfmt, y_perm, ws,
                     static_cast<cudaStream_t>(stream));
}

moe_status layer_q(const moe_shape* shape, const float* logits, const int32_t* ids_in, const float* w_in,
                   const uint16_t* x, const uint8_t* w13, const uint8_t* w13_bscale, const float* w13_scale,
                   const uint8_t* w2, const uint8_t* w2_bscale, const float* w2_scale, int wfmt,
                   const uint16_t* residual, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_quant_shape(shape, wfmt)) != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, true)) != MOE_OK) return r;
    if (logits ? !aligned(logits, 16) : (!aligned(ids_in, 16) || !aligned(w_in, 16))) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(w13_scale, 16) || !aligned(w2, 16) ||
        !aligned(w2_scale, 16) || !aligned(out, 16) || !aligned_or_null(residual, 16))
        return MOE_ERR_INVALID_ARG;
    if (wfmt == kWeightNvfp4 && (!aligned(w13_bscale, 16) || !aligned(w2_bscale, 16))) return MOE_ERR_INVALID_ARG;
    const moe_shape& s = *shape;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const WsLayout L = ws_layout(s);
    const int32_t* ids = ids_in;
    const float* w = w_in;
    const bool small = s.tokens <= kSmallDispatchTokens;   // one fused route + dispatch kernel
    if (logits) {
        int32_t* ids_ws = at<int32_t>(ws, L.ids);
        float* w_ws = at<float>(ws, L.w);
        if (!small && (r = do_route(s, logits, ids_ws, w_ws, ws, st)) != MOE_OK) return r;
        ids = ids_ws;
        w = w_ws;
    }
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* dest = at<int32_t>(ws, L.dest);
    uint16_t* x_perm = at<uint16_t>(ws, L.x_perm);
    uint16_t* h = at<uint16_t>(ws, L.h);
    uint16_t* y_perm = at<uint16_t>(ws, L.y_perm);
    if (small) {
        if ((r = from_cuda(launch_small_dispatch(s, logits, ids_in, at<int32_t>(ws, L.ids), at<float>(ws, L.w), x,
                                                 at<int32_t>(ws, L.counts), offsets, dest,
                                                 at<int32_t>(ws, L.sorted_pair), x_perm, at<WsHeader>(ws, 0),
                                                 nullptr, 0, st))) !=
            MOE_OK)
            return r;
    } else if ((r = do_dispatch(s, x, ids, at<int32_t>(ws, L.counts), offsets, dest, at<int32_t>(ws, L.sorted_pair),
                                x_perm, ws, st)) != MOE_OK) {
        return r;
    }
    // the up projection may start its weight loads once the fused dispatch has
    // published the bucket bounds; the down projection at once (they are final)
    if ((r = do_up_q(s, x_perm, offsets, w13, w13_bscale, w13_scale, wfmt, h, ws, st, true, small ? 2 : 0)) ==
            MOE_OK &&
        (r = do_down_q(s, h, offsets, w2, w2_bscale, w2_scale, wfmt, y_perm, ws, st, true, 1)) == MOE_OK)
        r = do_combine(s, y_perm, dest, w, nullptr, residual, out, st, at<WsHeader>(ws, 0));
    if (r != MOE_OK) reset_route_ready(ws, st);
    return r;
}

}  // namespace

moe_status validate_shape(const moe_shape* s) { return check_shape(s); }

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(*shape).total;
    return MOE_OK;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!aligned(ws, 256) || ws_bytes < 4096) return MOE_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(ws, 0, 4096, static_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const moe_shape* shape, const float* logits, int32_t* topk_ids, float* topk_w, void* ws,
                     size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(logits, 16) || !aligned(topk_ids, 16) || !aligned(topk_w, 16)) return MOE_ERR_INVALID_ARG;
    return do_route(*shape, logits, topk_ids, topk_w, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_gate(const moe_shape* shape, const uint16_t* x, const uint16_t* w_gate, float* logits, void* ws,
                    size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(x, 16) || !aligned(w_gate, 16) || !aligned(logits, 16)) return MOE_ERR_INVALID_ARG;
    const moe_shape& s = *shape;
    GemmProblem g{};
    g.mode = kGemmF32;
    g.a = x; g.a_rows = s.tokens; g.a_cols = s.hidden;
    g.b = w_gate; g.b_rows = s.experts; g.b_cols = s.hidden;
    g.offsets = nullptr; g.groups = 1; g.rows_all = s.tokens;
    g.K = s.hidden; g.nseg = 1; g.a_seg_col = 0; g.b_seg_row = 0;
    g.N = s.experts; g.b_group_rows = 0; g.up_off = 0;
    g.out = logits; g.ldo = s.experts; g.out_group_col = 0;
    return launch_grouped_gemm(g, at<WsHeader>(ws, 0), static_cast<cudaStream_t>(stream));
}

moe_status moe_route_sigmoid(const moe_shape* shape, const float* logits, const float* bias, float route_scale,
                             int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(logits, 16) || !aligned(topk_ids, 16) || !aligned(topk_w, 16) || !aligned_or_null(bias, 4))
        return MOE_ERR_INVALID_ARG;
    if (!(route_scale == route_scale) || route_scale == INFINITY || route_scale == -INFINITY)
        return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_route_sigmoid(*shape, logits, bias, route_scale, topk_ids, topk_w, at<WsHeader>(ws, 0),
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* topk_ids, int32_t* counts,
                        int32_t* offsets, int32_t* dest, int32_t* sorted_pair, uint16_t* x_perm, void* ws,
                        size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(x, 16) || !aligned(topk_ids, 16) || !aligned(counts, 16) || !aligned(offsets, 16) ||
        !aligned(dest, 16) || !aligned(sorted_pair, 16) || !aligned(x_perm, 16))
        return MOE_ERR_INVALID_ARG;
    return do_dispatch(*shape, x, topk_ids, counts, offsets, dest, sorted_pair, x_perm, ws,
                       static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_up(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w13,
                         const uint16_t* x, const uint16_t* ws13, uint16_t* h, void* ws, size_t ws_bytes,
                         void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(x_perm, 16) || !aligned(offsets, 16) || !aligned(w13, 16) || !aligned(h, 16))
        return MOE_ERR_INVALID_ARG;
    if (shape->shared > 0 && (!aligned(x, 16) || !aligned(ws13, 16))) return MOE_ERR_INVALID_ARG;
    return do_up(*shape, x_perm, offsets, w13, x, ws13, h, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_down(const moe_shape* shape, const uint16_t* h, const int32_t* offsets, const uint16_t* w2,
                           const uint16_t* ws2, uint16_t* y_perm, uint16_t* y_shared, void* ws, size_t ws_bytes,
                           void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(h, 16) || !aligned(offsets, 16) || !aligned(w2, 16) || !aligned(y_perm, 16))
        return MOE_ERR_INVALID_ARG;
    if (shape->shared > 0 && (!aligned(ws2, 16) || !aligned(y_shared, 16))) return MOE_ERR_INVALID_ARG;
    return do_down(*shape, h, offsets, w2, ws2, y_perm, y_shared, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets,
                          const uint16_t* w13, const uint16_t* w2, const uint16_t* x, const uint16_t* ws13,
                          const uint16_t* ws2, uint16_t* h, uint16_t* y_perm, uint16_t* y_shared, void* ws,
                          size_t ws_bytes, void* stream) {
    moe_status r = moe_expert_up(shape, x_perm, offsets, w13, x, ws13, h, ws, ws_bytes, stream);
    if (r != MOE_OK) return r;
    return moe_expert_down(shape, h, offsets, w2, ws2, y_perm, y_shared, ws, ws_bytes, stream);
}

moe_status moe_combine(const moe_shape* shape, const uint16_t* y_perm, const int32_t* dest, const float* topk_w,
                       const uint16_t* y_shared, const uint16_t* residual, uint16_t* out, void* ws,
                       size_t ws_bytes, void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, false)) != MOE_OK) return r;
    if (!aligned(y_perm, 16) || !aligned(dest, 16) || !aligned(topk_w, 16) || !aligned(out, 16) ||
        !aligned_or_null(y_shared, 16) || !aligned_or_null(residual, 16))
        return MOE_ERR_INVALID_ARG;
    return do_combine(*shape, y_perm, dest, topk_w, y_shared, residual, out, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer(const moe_shape* shape, const float* logits, const int32_t* ids_in, const float* w_in,
                     const uint16_t* x, const uint16_t* w13, const uint16_t* w2, const uint16_t* ws13,
                     const uint16_t* ws2, const uint16_t* residual, uint16_t* out, void* ws, size_t ws_bytes,
                     void* stream) {
    clear_error();
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((r = check_ws(shape, ws, ws_bytes, true)) != MOE_OK) return r;
    if (logits ? !aligned(logits, 16) : (!aligned(ids_in, 16) || !aligned(w_in, 16))) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) ||
        !aligned_or_null(residual, 16))
        return MOE_ERR_INVALID_ARG;
    if (shape->shared > 0 && (!aligned(ws13, 16) || !aligned(ws2, 16))) return MOE_ERR_INVALID_ARG;
    const moe_shape& s = *shape;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const WsLayout L = ws_layout(s);
    const int32_t* ids = ids_in;
    const float* w = w_in;
    const bool small = s.tokens <= kSmallDispatchTokens;   // one fused route + dispatch kernel
    if (logits) {
        int32_t* ids_ws = at<int32_t>(ws, L.ids);
        float* w_ws = at<float>(ws, L.w);
        if (!small && (r = do_route(s, logits, ids_ws, w_ws, ws, st)) != MOE_OK) return r;
        ids = ids_ws;
        w = w_ws;
    }
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* dest = at<int32_t>(ws, L.dest);
    uint16_t* x_perm = at<uint16_t>(ws, L.x_perm);
    uint16_t* h = at<uint16_t>(ws, L.h);
    uint16_t* y_perm = at<uint16_t>(ws, L.y_perm);
    uint16_t* y_shared = s.shared > 0 ? at<uint16_t>(ws, L.y_shared) : nullptr;
    // decode: the expert FFN and the combine in one launch after the fused dispatch
    const bool fused = small && decode_ffn_fits(s);
    unsigned* sync = at<unsigned>(ws, L.sync);
    if (small) {
        if ((r = from_cuda(launch_small_dispatch(s, logits, ids_in, at<int32_t>(ws, L.ids), at<float>(ws, L.w), x,
                                                 at<int32_t>(ws, L.counts), offsets, dest,
                                                 at<int32_t>(ws, L.sorted_pair), x_perm, at<WsHeader>(ws, 0),
                                                 fused ? sync : nullptr, (int)decode_ffn_sync_words(s), st))) !=
            MOE_OK)
            return r;
        if (fused) {
            r = launch_decode_ffn(s, x_perm, offsets, w13, w2, h, y_perm, dest, w, residual, out, sync,
                                  at<WsHeader>(ws, 0), st);
            if (r != MOE_OK) reset_route_ready(ws, st);
            return r;
        }
    } else if ((r = do_dispatch(s, x, ids, at<int32_t>(ws, L.counts), offsets, dest, at<int32_t>(ws, L.sorted_pair),
                                x_perm, ws, st)) != MOE_OK) {
        return r;
    }
    // the up projection may start its weight loads once the fused dispatch has
    // published the bucket bounds; the down projection at once (they are final)
    if ((r = do_up(s, x_perm, offsets, w13, x, ws13, h, ws, st, true, small ? 2 : 0)) == MOE_OK &&
        (r = do_down(s, h, offsets, w2, ws2, y_perm, y_shared, ws, st, true, 1)) == MOE_OK)
        r = do_combine(s, y_perm, dest, w, y_shared, residual, out, st, at<WsHeader>(ws, 0));
    if (r != MOE_OK) reset_route_ready(ws, st);
    return r;
}

moe_status moe_expert_up_fp8(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets,
                             const uint8_t* w13, const float* w13_scale, uint16_t* h, void* ws, size_t ws_bytes,
                             void* stream) {
    return expert_up_q(shape, x_perm, offsets, w13, nullptr, w13_scale, kWeightFp8E4M3, h, ws, ws_bytes, stream);
}

moe_status moe_expert_down_fp8(const moe_shape* shape, const uint16_t* h, const int32_t* offsets, const uint8_t* w2,
                               const float* w2_scale, uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream) {
    return expert_down_q(shape, h, offsets, w2, nullptr, w2_scale, kWeightFp8E4M3, y_perm, ws, ws_bytes, stream);
}

moe_status moe_layer_fp8(const moe_shape* shape, const float* logits, const int32_t* ids_in, const float* w_in,
                         const uint16_t* x, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                         const float* w2_scale, const uint16_t* residual, uint16_t* out, void* ws, size_t ws_bytes,
                         void* stream) {
    return layer_q(shape, logits, ids_in, w_in, x, w13, nullptr, w13_scale, w2, nullptr, w2_scale, kWeightFp8E4M3,
                   residual, out, ws, ws_bytes, stream);
}

moe_status moe_expert_up_nvfp4(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets,
                               const uint8_t* w13, const uint8_t* w13_bscale, const float* w13_scale, uint16_t* h,
                               void* ws, size_t ws_bytes, void* stream) {
    return expert_up_q(shape, x_perm, offsets, w13, w13_bscale, w13_scale, kWeightNvfp4, h, ws, ws_bytes, stream);
}

moe_status moe_expert_down_nvfp4(const moe_shape* shape, const uint16_t* h, const int32_t* offsets,
                                 const uint8_t* w2, const uint8_t* w2_bscale, const float* w2_scale,
                                 uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream) {
    return expert_down_q(shape, h, offsets, w2, w2_bscale, w2_scale, kWeightNvfp4, y_perm, ws, ws_bytes, stream);
}

moe_status moe_layer_nvfp4(const moe_shape* shape, const float* logits, const int32_t* ids_in, const float* w_in,
                           const uint16_t* x, const uint8_t* w13, const uint8_t* w13_bscale, const float* w13_scale,
                           const uint8_t* w2, const uint8_t* w2_bscale, const float* w2_scale,
                           const uint16_t* residual, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
    return layer_q(shape, logits, ids_in, w_in, x, w13, w13_bscale, w13_scale, w2, w2_bscale, w2_scale,
                   kWeightNvfp4, residual, out, ws, ws_bytes, stream);
}

moe_status moe_workspace_set_wait(void* ws, size_t ws_bytes, uint64_t lookback_wait_ns, int32_t count_tile_skip,
                                  void* stream) {
    clear_error();
    if (!aligned(ws, 256) || ws_bytes < 4096) return MOE_ERR_INVALID_ARG;
    if (count_tile_skip != 0 && count_tile_skip != 1) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_set_wait(at<WsHeader>(ws, 0), (unsigned long long)lookback_wait_ns, count_tile_skip,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status moe_timeout_site_read(void* ws, void* stream, int32_t* site) {
    if (!aligned(ws, 256) || !site) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader h;
    if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    *site = h.timeout_site;
    return MOE_OK;
}

moe_status moe_status_read(void* ws, void* stream, moe_status* device_status) {
    if (!aligned(ws, 256) || !device_status) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader h;
    if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    *device_status = static_cast<moe_status>(h.status);
    // clear the sticky status and the timeout site
    if (cudaMemsetAsync(ws, 0, 2 * sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

const char* moe_last_error_message(void) { return g_last_error; }

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_INVALID_ROUTE: return "invalid route (expert id out of range or duplicated in a token)";
        case MOE_ERR_CAPACITY: return "an expert received more pairs than the capacity";
        case MOE_ERR_NONFINITE: return "non-finite router logit";
        case MOE_ERR_TIMEOUT: return "a bounded device wait timed out";
        case MOE_ERR_CUDA: return "CUDA runtime or driver error";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_INTERNAL: return "internal error";
    }
    return "unknown status";
}

}  // extern "C"
