/*
 * moe_decode.h — C ABI of a single-GPU (GB300, sm_103a) mixture-of-experts
 * decode layer for 1..64 rows.
 *
 * The layer (one call of moe_decode_forward) is, for every row b of x:
 *   router      logits = x_b . W_r^T; s = sigmoid(logits); the top_k experts
 *               by s + bias (ties to the lower index); combine weights
 *               w = routed_scale * s_sel / sum(s_sel)
 *   routed      for each selected expert e: h = silu(W_gate,e x_b) * (W_up,e x_b),
 *               y_e = W_down,e h; y_routed = sum_j w_j y_{e_j}
 *               (expert weights are MXFP4: E2M1 nibbles, one E8M0 scale per
 *               32 contiguous K elements)
 *   shared      y_shared = W_sd (silu(W_sg x_b) * (W_su x_b)), bf16 weights
 *   tail        z = residual_b + y_routed + y_shared; residual_b <- bf16(z);
 *               out_b = bf16(z / sqrt(mean(z^2) + eps) * gamma)
 *
 * Sources: "Kimi K3 on GB300: 13 kernels a layer, and what 842 and 423 tokens
 * a second measure" — section "What one decode step of Kimi K3 does" (16 of
 * 896 experts per token, 17,547,264-byte MXFP4 experts), section "Why batch 1
 * on a rack is not only a bandwidth problem" (packed FP4 expert weights),
 * section "What the fused path changes" (router/MoE front, shared expert on a
 * side stream, one persistent routed-expert kernel for FC1 and FC2, a tail that
 * folds the down-projection reduction and the next norm together, L2 prefetch
 * of upcoming weights on a third stream; here the prefetch is issued by the
 * tail kernel).  The pages give the structure only;
 * the formulas above are the plainest reading of that structure.  Element and
 * scale encodings: OCP Microscaling Formats (MX) Specification v1.0.
 *
 * Conventions for every call:
 *  - Pointers marked "device" are CUDA device pointers on the device that was
 *    current at moe_layer_create; "host" pointers are ordinary host memory.
 *    The caller owns every buffer it passes; the library borrows weight
 *    pointers for the handle's lifetime and never frees them.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Forward calls are asynchronous on that stream, allocate nothing and never
 *    synchronise the host, so they may be captured into a CUDA graph.
 *  - Every call returns a moe_status (0 = MOE_OK).  Nothing aborts or throws
 *    across the ABI.  A handle must not be used from two streams at once.
 *  - bf16 tensors are row-major uint16 bit patterns (torch.bfloat16 layout).
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size or dims */
  MOE_ERR_UNSUPPORTED = 2,   /* B outside [1, max_batch], device is not sm_103, misaligned
                                pointer: the caller should use another implementation */
  MOE_ERR_CUDA = 3,          /* a CUDA runtime call failed (the error is kept for
                                moe_last_cuda_error) */
  MOE_ERR_ALLOC = 4,         /* workspace allocation failed at create time */
  MOE_ERR_TIMEOUT = 5        /* a device-side bounded wait expired (see moe_layer_status) */
} moe_status;

typedef struct moe_layer* moe_layer_t;

/* Layer dimensions.  d % 256 == 0 and d <= 7680; f % 256 == 0 and f <= 3072;
 * f_shared % 256 == 0 and f_shared <= 4096; 1 <= top_k <= 32; top_k <= n_experts
 * <= 1024; 1 <= max_batch <= 64 (INVALID_ARG otherwise).
 *
 * expert_path picks how the routed experts run.  1: mma.sync tensor cores
 * with the weights converted to f16 in registers (the GEMV regime; the
 * kernels read the tiled layouts, FC1 matrices in layout 2 and FC2 matrices in
 * layout 1), the shared expert and the router on the CUDA cores.  2: tcgen05
 * tensor cores, block-scaled MXFP4 MMAs with tensor-memory accumulators (the
 * UMMA layouts, FC1 in layout 4 and FC2 in layout 3); the shared expert (and,
 * from 25 rows, the router) as bf16 MMAs on the same tensor cores, from bf16
 * copies of those weights in 128-row tiles that the handle owns (2 * (3 * d *
 * f_shared + 128 * ceil(E / 128) * d) bytes of extra device memory).  0
 * (default): the layer keeps both and takes path 1 for B = 1 and path 2 for
 * B >= 2, or only path 1 when max_batch is 1 (one copy of the expert bytes
 * instead of two).  Path 1's kernels hold a ring of shared-memory stages
 * sized for the dims; where it does not fit (large d with large f, or
 * f_shared above 3072, for example), path 1 returns UNSUPPORTED and path 0
 * keeps path 2 alone.  All give results within the same tolerance of the
 * exact layer.
 *
 * mxfp4_layout says how the caller's expert weights are laid out: 0
 * (canonical), 1 (tiled: FC1 layout 2, FC2 layout 1) or 3 (UMMA: FC1 layout 4,
 * FC2 layout 3); see mxfp4_pack.  Weights already in a kept path's layouts
 * are used in place; for every other kept path moe_layer_create relays them
 * into a copy the handle owns (E * 3 * d * f * 17/32 bytes of extra device
 * memory each). */
typedef struct {
  int32_t d;              /* hidden size */
  int32_t f;              /* routed-expert intermediate size */
  int32_t n_experts;      /* E */
  int32_t top_k;          /* k */
  int32_t f_shared;       /* shared-expert intermediate size */
  int32_t max_batch;      /* largest B forward will be called with */
  float routed_scale;     /* combine weights sum to this (2.5 for the Kimi-style router) */
  float rms_eps;          /* RMSNorm epsilon (1e-6) */
  int32_t mxfp4_layout;   /* 0: canonical, 1: tiled, 3: UMMA expert weights (see above) */
  int32_t expert_path;    /* 0: both (by batch), 1: mma.sync, 2: tcgen05 (see above) */
} moe_dims_t;

/* Device pointers to the layer's weights (borrowed, never freed).
 * Expert e's FC1 rows 0..f-1 are the gate projection and rows f..2f-1 the up
 * projection; row i of the gate pairs with row i of the up projection. */
typedef struct {
  const void* router_w;        /* device bf16 [E][d] */
  const float* router_bias;    /* device fp32 [E], used for selection only */
  const uint8_t* w_gu_q;       /* device [E][2f][d/2]  E2M1 nibbles (layout 0, 2 or 4) */
  const uint8_t* w_gu_s;       /* device [E][2f][d/32] E8M0 scale bytes (layout 0, 2 or 4) */
  const uint8_t* w_d_q;        /* device [E][d][f/2]  (layout 0, 1 or 3) */
  const uint8_t* w_d_s;        /* device [E][d][f/32] (layout 0, 1 or 3) */
  const void* shared_gu;       /* device bf16 [2 f_shared][d] (gate rows, then up rows) */
  const void* shared_d;        /* device bf16 [d][f_shared] */
  const void* rms_gamma;       /* device bf16 [d] */
} moe_weights_t;

/* Validate dims, device (must be sm_103) and pointer alignment (16 bytes),
 * allocate the workspace (routing tables, intermediates, timing events) on
 * the current device and return a handle in *out.
 * Errors: INVALID_ARG (null or bad dims), UNSUPPORTED (device/alignment),
 * ALLOC (workspace), CUDA. */
int moe_layer_create(const moe_dims_t* dims, const moe_weights_t* weights, moe_layer_t* out);

/* Free the workspace (synchronises the device first).  NULL is accepted. */
int moe_layer_destroy(moe_layer_t layer);

/* Router only: x device bf16 [B][d] -> idx device int32 [B][k] (descending by
 * score + bias, ties to the lower index) and w device fp32 [B][k] (combine
 * weights).  Same kernel as the first step of moe_decode_forward.
 * Errors: INVALID_ARG, UNSUPPORTED (B), CUDA. */
int moe_router_topk(moe_layer_t layer, void* stream, const void* x, int B, int32_t* idx, float* w);

/* The whole layer.  x device bf16 [B][d] (read only); residual device bf16
 * [B][d], read and overwritten with bf16(z); out device bf16 [B][d].  x, out
 * and residual must not overlap.  Asynchronous, allocation-free. */
int moe_decode_forward(moe_layer_t layer, void* stream, const void* x, int B, void* residual,
                       void* out);

/* The same layer with HOST buffers: copies x and residual host -> device on
 * `stream`, runs moe_decode_forward on the handle's own device staging
 * buffers, copies residual and out back, and synchronises `stream` before
 * returning.  x_host, residual_host, out_host: host bf16 [B][d] (pinned memory
 * gives asynchronous copies; pageable memory works but copies synchronously).
 * With pinned buffers and a stream other than the legacy default stream, the
 * first call captures the copies and the kernels as one CUDA graph, which
 * later calls with the same buffers, B and stream replay (one launch per call;
 * changing any of them captures again).  Overlapping calls on one layer race,
 * as for moe_decode_forward. */
int moe_decode_forward_host(moe_layer_t layer, void* stream, const void* x_host, int B,
                            void* residual_host, void* out_host);

/* moe_decode_forward that also exports intermediates (any may be NULL):
 * y_routed device fp32 [B][d], y_shared device fp32 [B][d],
 * h device fp32 [B][k][f] (h[b][j] belongs to expert idx[b][j]),
 * z device fp32 [B][d] (residual + y_routed + y_shared before bf16 rounding),
 * out_f32 device fp32 [B][d] (the normalised output before bf16 rounding). */
int moe_decode_forward_debug(moe_layer_t layer, void* stream, const void* x, int B, void* residual,
                             void* out, float* y_routed, float* y_shared, float* h, float* z,
                             float* out_f32);

/* Dequantise one expert matrix on the GPU from the handle's tiled copy, with
 * the kernels' element decode (cvt.rn.f16x2.e2m1x2) and the exact scale value:
 * which = 0 -> FC1 [2f][d], which = 1 -> FC2 [d][f], canonical row order;
 * out device fp32.  (The matmul kernels read scale code 0, 2^-127, as 0: the
 * products it scales are below 6 * 2^-127 * |activation|.) */
int moe_debug_dequant(moe_layer_t layer, void* stream, int expert, int which, float* out);

/* Activation format of the routed experts' products (the pages' routed-expert
 * kernel multiplies FP4 weights by MXFP8 activations: "Kimi K3 on GB300: 13
 * kernels a layer", "Why batch 1 on a rack is not only a bandwidth problem").
 * fmt 0 (default): x (bf16) and h (fp32) as they are, the exact layer within
 * the stated tolerance.  fmt 1: x and h rounded to MXFP8 (OCP MX v1.0: E4M3
 * elements, nearest with ties to even and saturation at 448, one E8M0 scale
 * 2^(floor(log2 max|v|) - 8) per 32 contiguous elements) before they meet the
 * MXFP4 weights; the router, shared expert and tail are unchanged.  The
 * one-row mma.sync kernel carries the rounded values exactly in its f16
 * operands; the tensor-core path builds its activation planes (E2M1 digits,
 * block-scaled MMAs) from them.  fmt 1 runs on the tensor-core path at any B
 * and on the mma.sync path at B = 1; a forward of B > 1 rows on the mma.sync
 * path returns MOE_ERR_UNSUPPORTED.  Errors: INVALID_ARG. */
int moe_set_act_format(moe_layer_t layer, int fmt);

/* Chain layers: this layer's tail kernel, whose CTAs start while the expert
 * kernels finish, issues L2 prefetches (prefetch.global.L2::evict_last) of
 * `next`'s router weights before it waits for them, so the next layer's
 * router, the first kernel of the next forward, finds them in L2.  No extra
 * launch or stream.  next may be NULL to switch it off.  Both handles must
 * live on the same device. */
int moe_set_prefetch_next(moe_layer_t layer, moe_layer_t next);

/* Synchronise the layer's streams and report the device status word
 * (0 = ok, else a moe_status such as MOE_ERR_TIMEOUT); clears it. */
int moe_layer_status(moe_layer_t layer, int* device_status);

/* Failure-detection test hook (the pages have no counterpart; it exists so a
 * test can watch a device-side wait expire without faulting anything).
 * fault = 1: in later forwards of one row on the mma.sync path (FC1 and FC2
 * in one launch, whose CTAs meet at a grid-wide barrier between the two
 * steps), CTA 0 does not count itself at that barrier, and every CTA's wait
 * there is limited to wait_ns nanoseconds (0: the default 2 s).  The waits
 * expire, FC2 runs on the FC1 results that are already written, the forward
 * completes, and moe_layer_status then reports MOE_ERR_TIMEOUT.  fault = 0
 * restores normal operation.
 * Nothing on the GPU traps, faults or hangs.  Errors: INVALID_ARG. */
int moe_debug_set_fault(moe_layer_t layer, int fault, unsigned long long wait_ns);

/* Per-phase timing of forward calls (CUDA events on the launching stream;
 * under stream capture they become event-record nodes of the graph).
 * enable != 0 records events around each phase from the next forward on.
 * moe_get_timing synchronises and writes up to n floats (microseconds) for
 * the last forward: [0] router + top-k, [1] FC1 (shared then routed gate/up),
 * [2] FC2 (shared then routed down), [3] always 0 (the shared expert has no
 * phase of its own), [4] tail, [5] whole layer. */
int moe_set_timing(moe_layer_t layer, int enable);
int moe_get_timing(moe_layer_t layer, float* us, int n);

/* Device-side kernel trace.  enable != 0 makes every later forward record,
 * per kernel, the earliest CTA start and the latest CTA end (globaltimer,
 * nanoseconds).  moe_get_trace synchronises the device and writes up to n
 * values: [start, end] of router, top-k, FC1, FC2, tail, in that order (ten
 * values); a kernel that did not run reports start > end. */
int moe_set_trace(moe_layer_t layer, int enable);
int moe_get_trace(moe_layer_t layer, unsigned long long* ns, int n);

/* Number of kernel launches one forward makes for batch B. */
int moe_launches_per_forward(moe_layer_t layer, int B);

/* ---- MXFP4 packing (OCP MX v1.0: E2M1 elements, E8M0 scale per 32 K) ---- */
/* Canonical layout 0: row-major; byte j of a row holds elements 2j (low
 * nibble) and 2j+1 (high nibble); scale byte b of a row covers elements
 * 32b..32b+31.  Scale exponent = floor(log2(amax)) - 2 clamped to [-127, 127]
 * (all-zero block: -127); element code = nearest E2M1 value to w / 2^exp,
 * ties to the even code, magnitudes past 6 saturate to 6, sign bit = sign of w. */

/* Tiled layouts 1 and 2 hold the same bytes for the tensor-core kernels.
 * Rows form tiles of 16 "mma rows": layout 1 puts rows 16T..16T+15 in tile T;
 * layout 2 (a [2n][k] gate/up matrix, row i pairing with row n + i) puts rows
 * 8T..8T+7 as mma rows 0..7 and rows n+8T..n+8T+7 as mma rows 8..15.  Tile T's
 * nibbles occupy bytes [8kT, 8k(T+1)): for K blocks 2P and 2P+1 (32 elements
 * each) and lane L = 4g + t (g < 8, t < 4), 16 bytes at 8kT + (32P + L) * 16
 * hold canonical bytes [4t, 4t+4) of block 2P of mma row g, then of mma row
 * g + 8, then the same two for block 2P+1.  Tile T's scales occupy bytes
 * [kT/2, k(T+1)/2): for block group Q (blocks 4Q..4Q+3) and g, 8 bytes at
 * kT/2 + (8Q + g) * 8 hold, per block 4Q+j, the scale of mma row g (byte 2j)
 * and of mma row g + 8 (byte 2j + 1).  Tiled layouts need k % 128 == 0 and
 * rows % 16 == 0. */

/* UMMA layouts 3 and 4 hold the same bytes as tcgen05 block-scaled operands
 * (no swizzle, K-major core matrices of 8 rows x 16 bytes).  Rows form tiles
 * of 128 "mma rows": layout 3 puts rows 128T..128T+127 in tile T; layout 4 (a
 * [2n][k] gate/up matrix) puts rows 64T..64T+63 as mma rows 0..63 and rows
 * n+64T..n+64T+63 as mma rows 64..127.  Tile T's nibbles occupy bytes
 * [64kT, 64k(T+1)): the 16 canonical bytes of K block b of mma row m at
 * 64kT + 2048b + 128(m/8) + 16(m%8).  Tile T's scales occupy bytes [4kT,
 * 4k(T+1)): the scale of (m, b) at 4kT + 512(b/4) + 16(m%32) + 4(m/32) + b%4.
 * UMMA layouts need k % 128 == 0 and rows % 128 == 0. */

/* Bytes of nibbles for rows x k (k % 32 == 0, and the layout's rules);
 * *scale_bytes gets the scale bytes when non-NULL.  The same for every
 * layout.  Returns 0 on bad arguments. */
size_t mxfp4_packed_bytes(int64_t rows, int64_t k, int layout, size_t* scale_bytes);

/* Host packer: w host fp32 [rows][k] -> q host [rows][k/2], s host [rows][k/32]. */
int mxfp4_pack(const float* w, int64_t rows, int64_t k, uint8_t* q, uint8_t* s, int layout);

/* Device packer, asynchronous on stream: w device fp32 -> q, s device. */
int mxfp4_pack_device(void* stream, const float* w, int64_t rows, int64_t k, uint8_t* q,
                      uint8_t* s, int layout);

/* Host conversion between layouts (0 to 4) of one rows x k matrix: q_in, s_in
 * host in layout `from`; q_out, s_out host in layout `to` (same sizes, must not
 * overlap the input).  Errors: INVALID_ARG, UNSUPPORTED (a layout's rules). */
int mxfp4_repack(const uint8_t* q_in, const uint8_t* s_in, int64_t rows, int64_t k, int from,
                 int to, uint8_t* q_out, uint8_t* s_out);

/* Canonical packed bytes -> tiled or UMMA layout 1 to 4, asynchronous on stream, for
 * n_mat matrices stored back to back (rows x k each): q_in, s_in device
 * canonical; q_out, s_out device, the same sizes, must not overlap the input.
 * Errors: INVALID_ARG, UNSUPPORTED (layout rules, 16-byte alignment), CUDA. */
int mxfp4_retile_device(void* stream, const uint8_t* q_in, const uint8_t* s_in, int64_t n_mat,
                        int64_t rows, int64_t k, int layout, uint8_t* q_out, uint8_t* s_out);

/* Router + top-k that allocates nothing (no counterpart in the paper: it
 * exists for callers that cannot call cudaMalloc, e.g. code running inside a
 * stream capture it does not own, runtimes that hand over a fixed memory pool,
 * or callers that must not synchronise the device).  It needs no layer handle:
 * router_w device bf16 [E][d], router_bias device fp32 [E], x device bf16
 * [B][d]; outputs idx device int32 [B][k] and w device fp32 [B][k], exactly
 * as moe_router_topk.  Its scratch (logits, ticket, status word, routing
 * tables; 284,416 bytes) is one static device array that every GPU loading
 * this library holds until the process exits; each call looks up the current
 * device's address of it.  Limits: B <= 64, E <= 1024, k <= 32, d % 256 == 0,
 * d <= 7680 (as for a layer); larger sizes return MOE_ERR_UNSUPPORTED.  The
 * first call on each device (and the first with a new d) sizes the launch
 * (host-side queries, no allocation): make that call before any stream
 * capture.  A CUDA error already pending when the call starts is returned
 * (MOE_ERR_CUDA, its code kept for moe_last_cuda_error) and nothing is
 * launched.  Every call shares the one array, so calls that overlap on the GPU
 * (two streams, or two threads) race; calls in one stream are safe. */
int moe_router_topk_noalloc(void* stream, const void* router_w, const float* router_bias,
                            const void* x, int B, int d, int n_experts, int top_k,
                            float routed_scale, int32_t* idx, float* w);

/* Status word of the allocation-free router on the current device: 0, or
 * MOE_ERR_TIMEOUT when a bounded device-side wait of an earlier call expired
 * (its outputs are then not valid).  Each call clears the word when it
 * starts, so this reports the calls since the last one started; synchronises
 * the device, then clears the word. */
int moe_router_topk_noalloc_status(int* device_status);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/* The last CUDA error code a call saw (cudaError_t as int), 0 if none. */
int moe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
