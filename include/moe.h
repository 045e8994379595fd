/*
 * moe.h -- C ABI of libmoe.so, the single-GPU MoE layer hot path for GB300 (sm_103a).
 *
 * The layer (ONNX Runtime PR #33963 "Extend MoEPacked for Bolt ReLU-square routing
 * and BF16 IQ2 precision", Description and "Measured CUDA kernel latency"): router
 * logits -> softmax top-k routing (or caller-preselected expert ids with FP32
 * weights) -> count-first dispatch of token rows into expert-contiguous buckets
 * (afdEP-comm count-first validation record, keys .change and .setup) -> the
 * grouped expert FFN with SwiGLU (the default) or ReLU-square experts in BF16 with
 * FP32 accumulation -> the weighted combine back to token order (DeepSeek fleet
 * megakernel REPORT.md, MOE_GATE_TOPK / EXPERT_W13_SILU / EXPERT_W2 /
 * MOE_COMBINE_RESIDUAL rows of the per-op table).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers named "device" must be device memory of the current CUDA device;
 *    the caller owns every buffer.  The library never allocates or frees memory.
 *  - BF16 tensors are passed as uint16_t bit patterns.  All tensors are
 *    row-major and contiguous: a row of x, x_perm, y_perm, y_shared and out has
 *    `hidden` elements, a row of h has `inter` elements.
 *  - Device pointers must be 16-byte aligned; the workspace 256-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    only enqueues work on it: no host synchronisation, no allocation, so a
 *    sequence of calls can be captured in a CUDA graph.  The one exception is
 *    moe_status_read, which synchronises the stream.
 *  - Errors come in two tiers.  (1) Host-detectable errors (bad shape, null or
 *    misaligned pointers, small workspace) are returned at once and nothing is
 *    launched.  (2) Errors only the device can see -- an invalid route, a
 *    bucket over capacity, non-finite logits, a bounded wait that ran out --
 *    are folded into a status word in the workspace with an atomic max of the
 *    code and read back by moe_status_read.  After a device-side error the
 *    call's outputs are unspecified, but no kernel ever reads or writes outside
 *    the buffers described here.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* host: bad shape, null/misaligned pointer, small workspace */
    MOE_ERR_INVALID_ROUTE = 2,  /* device: an id < 0, an id >= experts, or a duplicate id inside a token */
    MOE_ERR_CAPACITY = 3,       /* device: some expert received more than `capacity` pairs */
    MOE_ERR_NONFINITE = 4,      /* device: a NaN or infinite router logit */
    MOE_ERR_TIMEOUT = 5,        /* device: a bounded wait inside a kernel gave up */
    MOE_ERR_CUDA = 6,           /* host: a CUDA runtime/driver call failed (launch, tensor map) */
    MOE_ERR_UNSUPPORTED = 7,    /* host: a shape this build does not handle */
    MOE_ERR_INTERNAL = 8
} moe_status;

typedef enum moe_act {
    MOE_ACT_SWIGLU = 0,  /* h = silu(x W_gate^T) * (x W_up^T); W13 rows [0,I) gate, [I,2I) up */
    MOE_ACT_RELU2 = 1    /* h = max(x W1^T, 0)^2; W13 has I rows */
} moe_act;

/* Shape of one layer call.
 *   tokens T >= 1; hidden H, multiple of 8; experts E in [1, 1024];
 *   top_k k in [1, min(E, 32)]; inter I, multiple of 8 (expert intermediate);
 *   shared S >= 0 always-on shared experts of intermediate shared_inter
 *   (multiple of 8 when S > 0); capacity >= 1: the most pairs one expert may
 *   receive (a receive-buffer bound, as "capacity 2048" in the afdEP-comm
 *   record's .setup; it is not a drop policy); act: a moe_act value.
 * Derived: R = T*k routed pairs; up = 2I (SwiGLU) or I (ReLU^2). */
typedef struct moe_shape {
    int32_t tokens;
    int32_t hidden;
    int32_t experts;
    int32_t top_k;
    int32_t inter;
    int32_t shared;
    int32_t shared_inter;
    int32_t capacity;
    int32_t act;
} moe_shape;

/* Bytes of device workspace that every call below needs for this shape (the
 * moe_layer figure, which covers the others).  Host only, synchronous. */
MOE_API moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes);

/* Zero the workspace's status word and counters.  Call once after allocating
 * a workspace (or allocate it zero-filled).  Enqueued on `stream`. */
MOE_API moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Routing (ONNX Runtime PR #33963, "Measured CUDA kernel latency": internal
 * softmax routing over router logits).
 *   logits   device f32 [T, E]  router logits
 *   topk_ids device i32 [T, k]  out: the k experts with the largest logits,
 *                               in descending logit order; equal logits
 *                               (-0 == +0 included) go to the lower index
 *   topk_w   device f32 [T, k]  out: softmax over the k selected logits
 *                               (sums to 1; the +16/-16 case gives 1/9 each)
 * Device error: MOE_ERR_NONFINITE if any logit is NaN or infinite. */
MOE_API moe_status moe_route(const moe_shape* shape, const float* logits, int32_t* topk_ids,
                     float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* Router projection in front of the routing (ONNX Runtime PR #33963,
 * Description: "projected" routing; DeepSeek fleet REPORT.md, MOE_GATE_TOPK
 * fuses this projection with the top-k):
 *   logits[t][e] = sum_h x[t][h] * w_gate[e][h], FP32 accumulation, FP32 out.
 *   x      device bf16 [T, H];  w_gate device bf16 [E, H] (nn.Linear [out, in])
 *   logits device f32  [T, E]  out
 * Runs on the grouped GEMM kernels (one group, FP32 epilogue). */
MOE_API moe_status moe_gate(const moe_shape* shape, const uint16_t* x, const uint16_t* w_gate, float* logits,
                            void* ws, size_t ws_bytes, void* stream);

/* Sigmoid routing with a selection-only correction bias (ONNX Runtime PR
 * #33963, Description bullet 2: fused sigmoid routing with FP32 correction
 * bias, mixture weights from the unbiased scores).  Per token: s_e =
 * sigmoid(logit_e), taken in double and rounded once to FP32; the k experts
 * with the largest FP32 keys s_e + bias[e] are selected (ties to the lower
 * index), in descending key order; topk_w[t,j] = route_scale * s / (sum of the
 * selected s), FP32.
 *   logits device f32 [T, E]; bias device f32 [E] or NULL (no bias);
 *   topk_ids device i32 [T, k] out; topk_w device f32 [T, k] out.
 * Device error: MOE_ERR_NONFINITE if any logit is NaN or infinite. */
MOE_API moe_status moe_route_sigmoid(const moe_shape* shape, const float* logits, const float* bias,
                                     float route_scale, int32_t* topk_ids, float* topk_w, void* ws,
                                     size_t ws_bytes, void* stream);

/* Count-first dispatch (afdEP-comm count-first record, .change: per-expert
 * counts and their prefix sums come before the payload rows move).
 *   x           device bf16 [T, H]
 *   topk_ids    device i32 [T, k]   expert of pair p = t*k + j
 *   counts      device i32 [E]      out: valid pairs per expert
 *   offsets     device i32 [E+1]    out: exclusive scan of counts; offsets[E] = valid pairs
 *   dest        device i32 [T*k]    out: slot of pair p in the expert-contiguous order
 *                                   (-1 for an invalid pair); stable: inside a bucket,
 *                                   pairs keep ascending p
 *   sorted_pair device i32 [T*k]    out: sorted_pair[dest[p]] = p
 *   x_perm      device bf16 [T*k, H] out: x_perm[dest[p]] = x[p / k]
 * A pair is invalid when its id is < 0 or >= E, or equals an id earlier in the
 * same token (afdEP-comm runner: negative / wide / duplicate / dummy routes);
 * invalid pairs are neither counted nor written and raise MOE_ERR_INVALID_ROUTE.
 * If a count exceeds `capacity`, counts and offsets are still written,
 * MOE_ERR_CAPACITY is raised and no payload (dest, sorted_pair, x_perm) moves. */
MOE_API moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* topk_ids,
                        int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* sorted_pair,
                        uint16_t* x_perm, void* ws, size_t ws_bytes, void* stream);

/* Expert up projection with the fused activation (DeepSeek fleet REPORT.md,
 * EXPERT_W13_SILU; ONNX Runtime PR #33963, ReLU-square experts).
 *   x_perm  device bf16 [T*k, H]  rows [offsets[e], offsets[e+1]) belong to expert e
 *   offsets device i32 [E+1]      as written by moe_dispatch
 *   w13     device bf16 [E, up, H]  (nn.Linear [out, in] layout per expert)
 *   h       device bf16 [T*k, I]  out: h = bf16(act(x_perm W13[e]^T)), FP32 accumulation;
 *                                 rows past offsets[E] are not written
 *   x, ws13 device bf16 [T, H], [S, shared_up, H]: shared experts (NULL when S == 0);
 *           their activations go to the workspace for moe_expert_down. */
MOE_API moe_status moe_expert_up(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets,
                         const uint16_t* w13, const uint16_t* x, const uint16_t* ws13,
                         uint16_t* h, void* ws, size_t ws_bytes, void* stream);

/* Expert down projection (DeepSeek fleet REPORT.md, EXPERT_W2).
 *   h        device bf16 [T*k, I]   from moe_expert_up
 *   w2       device bf16 [E, H, I]
 *   y_perm   device bf16 [T*k, H]   out: y_perm[r] = bf16(h[r] W2[e]^T), FP32 accumulation
 *   ws2      device bf16 [S, H, shared_inter] (NULL when S == 0)
 *   y_shared device bf16 [T, H]     out (S > 0): bf16(sum_s h_s W2s[s]^T), summed over s
 *                                   in FP32 and rounded once; NULL when S == 0.
 * moe_expert_up must have run on the same workspace first when S > 0. */
MOE_API moe_status moe_expert_down(const moe_shape* shape, const uint16_t* h, const int32_t* offsets,
                           const uint16_t* w2, const uint16_t* ws2, uint16_t* y_perm,
                           uint16_t* y_shared, void* ws, size_t ws_bytes, void* stream);

/* moe_expert_up followed by moe_expert_down. */
MOE_API moe_status moe_expert_ffn(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets,
                          const uint16_t* w13, const uint16_t* w2,
                          const uint16_t* x, const uint16_t* ws13, const uint16_t* ws2,
                          uint16_t* h, uint16_t* y_perm, uint16_t* y_shared,
                          void* ws, size_t ws_bytes, void* stream);

/* Weighted combine back to token order (DeepSeek fleet REPORT.md,
 * MOE_COMBINE_RESIDUAL: the combine with the block's residual add fused;
 * ONNX Runtime PR #33963, "FP32 final routing/reduction"):
 *   out[t] = bf16( sum_{j<k} topk_w[t,j] * y_perm[dest[t*k+j]] + y_shared[t] + residual[t] )
 * summed in FP32 in j order, then the shared term, then the residual; pairs
 * with dest < 0 are skipped.
 *   y_perm device bf16 [T*k, H]; dest device i32 [T*k]; topk_w device f32 [T, k];
 *   y_shared device bf16 [T, H] or NULL; residual device bf16 [T, H] or NULL
 *   (out may alias residual: each element is read before it is written);
 *   out device bf16 [T, H]. */
MOE_API moe_status moe_combine(const moe_shape* shape, const uint16_t* y_perm, const int32_t* dest,
                               const float* topk_w, const uint16_t* y_shared, const uint16_t* residual,
                               uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* The whole layer: route (when logits != NULL) or take preselected ids_in /
 * w_in (device i32 [T,k] / f32 [T,k], used when logits == NULL), then dispatch,
 * expert FFN and combine (adding residual [T, H] when it is not NULL), with
 * every intermediate in the workspace.  Given the ids and weights moe_route
 * returns, the output is bitwise the same either way (ONNX Runtime PR #33963:
 * internal and preselected routing give bitwise-equal outputs).
 * out: device bf16 [T, H] (may alias residual).
 * Device errors are those of the stages.  When a bucket exceeds `capacity`
 * (MOE_ERR_CAPACITY) no payload moves and the expert GEMMs and the combine do
 * nothing: out (and so an aliased residual) keeps its contents. */
MOE_API moe_status moe_layer(const moe_shape* shape, const float* logits, const int32_t* ids_in,
                             const float* w_in, const uint16_t* x, const uint16_t* w13,
                             const uint16_t* w2, const uint16_t* ws13, const uint16_t* ws2,
                             const uint16_t* residual, uint16_t* out, void* ws, size_t ws_bytes,
                             void* stream);

/* Quantized expert weights: FP8 E4M3 (ONNX Runtime PR #33963: weight-only
 * quantized FC1/FC2 experts with BF16 activations, BF16 store boundaries and
 * FP32 accumulation; the codec here is FP8 E4M3 -- the afdEP-comm record's
 * fp8 payload type -- in place of the page's IQ2_XXS).
 *   w13       device u8  [E, up, H]  E4M3 codes (OCP: bias 7, subnormals, no
 *                                    infinities); row layout as moe_expert_up.  The
 *                                    NaN codes S.1111.111 are not valid weights
 *                                    (the kernels decode them as +-480)
 *   w13_scale device f32 [E, up]     one scale per weight row
 *   w2        device u8  [E, H, I]   E4M3 codes; w2_scale device f32 [E, H]
 * A weight is decode(code) * scale of its row; the kernels decode the codes to
 * BF16 in tensor memory (exactly), multiply in BF16 with FP32 accumulation and
 * apply the row scale to the accumulator:
 *   SwiGLU: h[r][n] = bf16( silu(g) * u ), g = (x_r . dec(W13[e][n])) * s13[e][n],
 *           u = (x_r . dec(W13[e][I+n])) * s13[e][I+n];  ReLU^2 likewise with one row;
 *   y_perm[r][c] = bf16( (h_r . dec(W2[e][c])) * s2[e][c] ).
 * Host errors: MOE_ERR_UNSUPPORTED when shape->shared > 0 (no shared experts
 * here); MOE_ERR_INVALID_ARG when hidden or inter is not a multiple of 16 or a
 * pointer is not 16-byte aligned.  The other arguments, the workspace and the
 * device errors are those of moe_expert_up / moe_expert_down / moe_layer.
 * These run on the small-row kernel at any size: efficient when groups hold
 * up to 64 rows (decode); larger groups are taken in 64-row chunks. */
MOE_API moe_status moe_expert_up_fp8(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets,
                                     const uint8_t* w13, const float* w13_scale, uint16_t* h, void* ws,
                                     size_t ws_bytes, void* stream);
MOE_API moe_status moe_expert_down_fp8(const moe_shape* shape, const uint16_t* h, const int32_t* offsets,
                                       const uint8_t* w2, const float* w2_scale, uint16_t* y_perm, void* ws,
                                       size_t ws_bytes, void* stream);
MOE_API moe_status moe_layer_fp8(const moe_shape* shape, const float* logits, const int32_t* ids_in,
                                 const float* w_in, const uint16_t* x, const uint8_t* w13,
                                 const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                 const uint16_t* residual, uint16_t* out, void* ws, size_t ws_bytes,
                                 void* stream);

/* Quantized expert weights: NVFP4 (ONNX Runtime PR #33963, section "Current
 * source and CI repair": the NVFP4 guard and the BF16/FP16 NVFP4
 * scale-before-cast cases; the page names the format, this is the standard
 * NVFP4 layout).  Activations stay BF16; every weight row of K elements
 * (K = H for w13, I for w2) is
 *   codes  u8 [K/2]               E2M1 codes, two per byte, element 2j in the
 *                                 low nibble of byte j (1 sign bit, 2 exponent
 *                                 bits with bias 1, 1 mantissa bit: magnitudes
 *                                 0, 0.5, 1, 1.5, 2, 3, 4, 6)
 *   bscale u8 [16*ceil(K/256)]    byte j (j < K/16): the E4M3 scale of elements
 *                                 16j..16j+15; the padding bytes are never read
 *   scale  f32                    one scale per row
 * so that weight[c] = e2m1(code c) * e4m3(bscale[c/16]) * scale:
 *   w13 device u8 [E, up, H/2], w13_bscale device u8 [E, up, 16*ceil(H/256)],
 *   w13_scale device f32 [E, up]; w2 device u8 [E, H, I/2],
 *   w2_bscale device u8 [E, H, 16*ceil(I/256)], w2_scale device f32 [E, H].
 * The kernels form e2m1 * block scale (exact in BF16: the scale is applied
 * before the cast), multiply in BF16 with FP32 accumulation and apply the row
 * scale to the accumulator, with the output formulas of the FP8 calls.  The
 * E4M3 NaN codes are not valid block scales (decoded as +-480).
 * Host errors: MOE_ERR_UNSUPPORTED when shape->shared > 0; MOE_ERR_INVALID_ARG
 * when hidden or inter is not a multiple of 32 or a pointer is not 16-byte
 * aligned.  The rest is as for the FP8 calls (small-row kernel at any size). */
MOE_API moe_status moe_expert_up_nvfp4(const moe_shape* shape, const uint16_t* x_perm, const int32_t* offsets,
                                       const uint8_t* w13, const uint8_t* w13_bscale, const float* w13_scale,
                                       uint16_t* h, void* ws, size_t ws_bytes, void* stream);
MOE_API moe_status moe_expert_down_nvfp4(const moe_shape* shape, const uint16_t* h, const int32_t* offsets,
                                         const uint8_t* w2, const uint8_t* w2_bscale, const float* w2_scale,
                                         uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream);
MOE_API moe_status moe_layer_nvfp4(const moe_shape* shape, const float* logits, const int32_t* ids_in,
                                   const float* w_in, const uint16_t* x, const uint8_t* w13,
                                   const uint8_t* w13_bscale, const float* w13_scale, const uint8_t* w2,
                                   const uint8_t* w2_bscale, const float* w2_scale, const uint16_t* residual,
                                   uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* moe_dispatch for callers that cannot allocate device memory, and so cannot
 * provide the workspace the other calls take: code that runs where cudaMalloc
 * is not allowed or not safe (while a CUDA graph is being captured, inside a
 * custom allocator's own callbacks, on a teardown path), or a host whose device
 * memory is all handed out by a fixed arena with nothing spare for scratch.
 * The paper has no counterpart: this is a deployment convenience, not a step
 * of the method.
 * Arguments and results are those of moe_dispatch without the workspace; the
 * device status of this call (0 or a moe_status code) is written to
 * *device_status (device i32, 4-byte aligned; NULL skips it).
 * The scratch moe_dispatch keeps in the workspace (status header, per-pair
 * ranks, look-back flags) lives instead in one static device array of about
 * 1.5 MiB inside this library; every GPU that loads the library holds its own
 * copy until the process exits.  Limit: tokens * top_k <= 131072 pairs (with
 * the usual experts <= 1024); larger calls return MOE_ERR_UNSUPPORTED and say
 * why in moe_last_error_message, before anything is launched.
 * The first call on a device looks up the array's device address for that
 * device, a host-side step: make that first call before any stream capture.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).  All calls on a device share its one array, and each call clears
 * what must start at zero; calls that overlap on the same GPU (for example on
 * two concurrent streams) therefore race and must be serialised. */
MOE_API moe_status moe_dispatch_noalloc(const moe_shape* shape, const uint16_t* x, const int32_t* topk_ids,
                                        int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* sorted_pair,
                                        uint16_t* x_perm, int32_t* device_status, void* stream);

/* The plan of the expert-parallel count-first exchange (afdEP-comm count-first
 * validation record, .change and .setup: with the experts split over the ranks
 * of a node, the per-expert counts travel first -- E*G int32 in all -- so that
 * before any payload row moves every rank knows where each of its rows lands
 * in the owner's expert-contiguous receive buffer, and whether a receive
 * buffer would overflow; the combine returns along the same segments).
 * Host only: no device memory, nothing enqueued.
 * The E experts are split over `world` ranks in contiguous balanced blocks:
 * rank g owns experts [first(g), first(g+1)), first(g) = (g * E) / world, and
 * el = first(rank+1) - first(rank) of them belong to `rank`.
 *   counts_all   host i32 [world, E]  row s: rank s's per-expert counts (the
 *                                     counts its moe_dispatch wrote)
 *   send_offsets host i32 [E+1] out   where this rank's rows of expert e start
 *                                     in its own x_perm (the exclusive scan of
 *                                     its counts)
 *   recv_offsets host i32 [el+1] out  the receive buffer's bucket bounds for
 *                                     the el local experts (the offsets the
 *                                     local expert FFN takes)
 *   recv_slot    host i32 [world, el] out  first receive row of the rows that
 *                                     source s sends for local expert j; inside a
 *                                     bucket the sources come in rank order, each
 *                                     in its own token order
 *   peer_send, peer_recv host i32 [world] out  rows sent to / received from
 *                                     each rank
 * Rows for one (source, expert) pair travel as one segment, sender and
 * receiver taking the segments of a peer in ascending expert order.
 * Returns MOE_ERR_CAPACITY (with every output written) when some expert of some
 * rank would receive more than `capacity` rows -- every rank reaches the same
 * verdict from the same counts, so all skip the payload together -- and
 * MOE_ERR_INVALID_ARG for bad sizes, null pointers or a negative count. */
MOE_API moe_status moe_ep_plan(int32_t experts, int32_t world, int32_t rank, int32_t capacity,
                               const int32_t* counts_all, int32_t* send_offsets, int32_t* recv_offsets,
                               int32_t* recv_slot, int32_t* peer_send, int32_t* peer_recv);

/* Synchronise `stream`, return in *device_status the largest status code raised
 * by kernels on this workspace since the last read, and clear it (together
 * with the timeout site below). */
MOE_API moe_status moe_status_read(void* ws, void* stream, moe_status* device_status);

/* Test controls of the count kernel's bounded look-back wait, modelled on the
 * afdEP-comm count-first record's bounded timeout_while spins and its must-fail
 * case of counts that never arrive (.faults_shipped), injected from the host:
 * nothing here faults, traps or hangs a GPU.
 *   lookback_wait_ns  how long a count tile waits for a predecessor tile's
 *                     published counts before it gives up, raising
 *                     MOE_ERR_TIMEOUT (site 1); 0 restores the default 2 s.
 *   count_tile_skip   0 (normal) or 1.  With 1 the count kernel hands out tile
 *                     ids from 1, so no block ever publishes tile 0's counts:
 *                     on a dispatch of more than one count tile (T*k > 1024
 *                     pairs) the look-back waits for a flag that nothing sets
 *                     and gives up after lookback_wait_ns.  The dispatch's
 *                     outputs are then unspecified; every access stays inside
 *                     the buffers.  A single-tile dispatch is unaffected.
 * Both settings stay in the workspace header until changed (moe_workspace_init
 * resets them to 0) and apply to moe_dispatch and moe_layer calls on it.  The
 * GEMM kernels' waits keep their fixed 2 s limit.  Enqueued on `stream`.
 * Host error: MOE_ERR_INVALID_ARG for a bad workspace or count_tile_skip. */
MOE_API moe_status moe_workspace_set_wait(void* ws, size_t ws_bytes, uint64_t lookback_wait_ns,
                                          int32_t count_tile_skip, void* stream);

/* Synchronise `stream` and return in *site where the last bounded wait that
 * ran out on this workspace gave up: 0 none, 1 the count kernel's look-back,
 * 2 a GEMM TMA producer, 3 a GEMM MMA issuer, 4 a GEMM epilogue, 5 the
 * small-row GEMM, 6 moe_layer's fused decode FFN.  Read it before
 * moe_status_read, which clears it. */
MOE_API moe_status moe_timeout_site_read(void* ws, void* stream, int32_t* site);

/* A static, human-readable name for a status code. */
MOE_API const char* moe_status_string(moe_status status);

/* A description of the last host-side failure (MOE_ERR_CUDA, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_INVALID_ARG) raised by a call on this host thread, e.g. the CUDA error
 * name of a failed launch; "" when none.  The pointer stays valid until the next
 * call on the same thread. */
MOE_API const char* moe_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
