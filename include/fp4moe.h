/*
 * fp4moe - routed mixture-of-experts layer over block-scaled FP4 weights,
 * for NVIDIA GB300 (sm_103a).  C ABI.
 *
 * The layer (one call of fp4moe_forward) computes, for T tokens x[T, H]:
 *   1. router logits l = x . Wr^T (bf16 inputs, fp32 accumulation), sigmoid
 *      scores s, corrected scores c = s + bias, grouped top-k on c, routing
 *      weights from s                      ("Kimi-K2.7-Code on Gaudi 2",
 *      section "What was built": grouped top-k router, sigmoid scoring with
 *      correction bias);
 *   2. an expert histogram, prefix sum and stable permutation of the routes;
 *   3. on-the-fly MXFP4 or NVFP4 quantisation of x ("Serve Kimi-K2.5-MXFP4 on
 *      MI355X with ATOM", section "Stage B: Dynamic Activation Quantization";
 *      "Serving NVFP4 models on AMD Instinct MI355 accelerators", section
 *      "Weight Dequantization and Activation QDQ");
 *   4. the gate/up grouped GEMM on block-scaled FP4 tensor cores, SwiGLU and
 *      requantisation of the intermediate (A4W4);
 *   5. the down grouped GEMM whose epilogue adds w * y into the output
 *      (section "Stage D: MXFP4 Fused MoE": two-stage fused MoE, atomic
 *      combine variant).
 * fp4moe_mxfp4_to_fp8_rowscale is the exact per-channel MXFP4 -> FP8
 * conversion of "Kimi-K2.7-Code on Gaudi 2", section "Exact MXFP4 to FP8
 * per-channel conversion".
 *
 * Conventions for every entry point:
 *   - Pointers are CUDA device pointers owned by the caller unless stated.
 *     The library allocates no device memory; scratch lives in a caller
 *     workspace (fp4moe_workspace_size).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Every call is asynchronous on it; none synchronises the host.
 *   - Argument and shape errors are returned synchronously and launch nothing.
 *     Data-dependent conditions (NaN scale bytes, conversion rows outside the
 *     exactness contract, a device wait that timed out) are recorded in a
 *     status word in the workspace; fp4moe_get_status reads it.
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Packed FP4: element 2j of a row in the low nibble of byte j, element
 *     2j+1 in the high nibble.  E2M1 code: sign bit 3, exponent bits 2..1
 *     (bias 1), mantissa bit 0.
 *   - MXFP4 scales: one E8M0 byte per 32 consecutive K values (2^(b-127)).
 *     NVFP4 scales: one E4M3 byte per 16 K values, plus one fp32 tensor scale.
 */
#ifndef FP4MOE_H
#define FP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP4MOE_OK = 0,
  FP4MOE_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum   */
  FP4MOE_ERR_UNSUPPORTED_SHAPE = 2, /* a size outside the supported set        */
  FP4MOE_ERR_WORKSPACE = 3,         /* workspace missing or too small          */
  FP4MOE_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed       */
  FP4MOE_ERR_TIMEOUT = 5,           /* a device-side wait ran out (status word) */
  FP4MOE_ERR_NAN_SCALE = 6,         /* an E8M0 scale byte 255 was seen          */
  FP4MOE_ERR_INEXACT = 7,           /* conversion row below the exponent floor */
  FP4MOE_ERR_DEVICE = 8             /* no sm_103 device is current             */
} fp4moe_status;

/* FP4MOE_FP8: the W8A8 layer of fp4moe_forward_w8a8 (E4M3 experts from the
 * exact conversion, per-token dynamic E4M3 activations). */
typedef enum { FP4MOE_MXFP4 = 0, FP4MOE_NVFP4 = 1, FP4MOE_FP8 = 2 } fp4moe_format;

/* Layer shape and routing parameters.
 *   T tokens, H hidden size, I expert intermediate size, E routed experts,
 *   top_k experts per token, n_group / topk_group grouped routing
 *   (n_group = 1: plain top-k), n_shared always-on shared experts (0 or 1),
 *   routed_scaling multiplies the routing weights, renormalize != 0 divides
 *   the chosen sigmoid scores by their sum first, fmt an fp4moe_format.
 * Supported: 1 <= T <= 65536; H % 256 == 0; I % 128 == 0; 1 <= E <= 512;
 *   1 <= top_k <= 16 and top_k <= E; E % n_group == 0; 2 <= E / n_group <= 64
 *   when n_group > 1 (a group's score sums its two largest scores);
 *   1 <= topk_group <= n_group <= 32; n_shared in {0, 1}. */
typedef struct {
  int32_t T, H, I, E, top_k, n_group, topk_group, n_shared;
  float routed_scaling;
  int32_t renormalize;
  int32_t fmt;
} fp4moe_dims;

/* Expert and router weights.
 *   w13       packed FP4 [E, 2I, H/2]: rows 0..I-1 gate, I..2I-1 up.
 *   w2        packed FP4 [E, H, I/2].
 *   w13_scale / w2_scale: block scales already repacked by fp4moe_pack_scales
 *             (E8M0 for MXFP4, E4M3 for NVFP4).
 *   g13, g2   NVFP4 only: fp32 tensor scales [E + n_shared] (shared expert
 *             last); NULL for MXFP4.
 *   sh13, sh13_scale, sh2, sh2_scale: the shared expert, same layouts with
 *             E = 1; NULL when n_shared == 0.
 *   w_router  bf16 [E, H].   bias  fp32 [E] correction bias.
 *   packed    0: the payloads w13, w2, sh13, sh2 are row-major as above;
 *             1: they hold the tiled layout of fp4moe_pack_weights (the
 *             GEMMs then read each weight tile as one contiguous block);
 *             2: as 1, except that w13 and sh13 hold the gate/up-paired
 *             layout of fp4moe_pack_gateup_weights and w13_scale and
 *             sh13_scale that of fp4moe_pack_gateup_scales (the gate/up
 *             GEMM then reads a K tile's gate and up blocks, and their
 *             scale groups, with one copy each);
 *             3: as 2, and w2 and sh2 (and w2_scale, sh2_scale) in the
 *             row-tile-paired layout: each 256-row slab of a down matrix
 *             packed as one gate/up pair with I = 128, that is
 *             fp4moe_pack_gateup_weights(src, dst, n_mat * H / 256, 128,
 *             I / 2) and fp4moe_pack_gateup_scales(src, dst,
 *             n_mat * H / 256, 128, kblocks, fmt), so that row tiles 2j
 *             and 2j + 1 of a K tile are adjacent (the down GEMM's units
 *             of two weight tiles then read both with one copy each).
 *             Needs H % 256 == 0 and, for fp4moe_forward_cols, h_begin
 *             and h_end multiples of 256 (else UNSUPPORTED_SHAPE).  Other
 *             values: INVALID_ARG. */
typedef struct {
  const uint8_t *w13, *w13_scale, *w2, *w2_scale;
  const float *g13, *g2;
  const uint8_t *sh13, *sh13_scale, *sh2, *sh2_scale;
  const uint16_t *w_router;
  const float *bias;
  int32_t packed;
} fp4moe_weights;

/* W8A8 expert weights: each expert matrix as fp4moe_mxfp4_to_fp8_rowscale
 * leaves it ("Kimi-K2.7-Code on Gaudi 2", section "Exact MXFP4 to FP8
 * per-channel conversion": E4M3 bytes and one fp32 power-of-two scale per row).
 *   w13 [E, 2I, H] E4M3 (gate rows, then up rows), w13_scale [E, 2I] fp32;
 *   w2 [E, H, I] E4M3, w2_scale [E, H] fp32;
 *   sh13 / sh13_scale / sh2 / sh2_scale: the shared expert (E = 1), NULL
 *   when n_shared == 0;  w_router bf16 [E, H];  bias fp32 [E]. */
typedef struct {
  const uint8_t *w13;
  const float *w13_scale;
  const uint8_t *w2;
  const float *w2_scale;
  const uint8_t *sh13;
  const float *sh13_scale;
  const uint8_t *sh2;
  const float *sh2_scale;
  const uint16_t *w_router;
  const float *bias;
} fp4moe_fp8_weights;

/* Byte offsets of the forward's intermediates inside the workspace, for
 * inspection after a call (all relative to the workspace base).  Row indices
 * refer to the padded permuted layout: routes of one expert occupy tiles of
 * n_tile rows, each tile at the start of its own 128-row slot. */
typedef struct {
  int64_t status;       /* int32[16] status word                            */
  int64_t logits;       /* fp32 [n_splits, T, E] partial router logits (the
                         * few-token MXFP4 path may use fewer or more
                         * splits; the region holds them)                  */
  int64_t topk_idx;     /* int32 [T, top_k], in descending corrected score  */
  int64_t topk_w;       /* fp32 [T, top_k]                                  */
  int64_t expert_count; /* int32 [E + n_shared] routes per expert           */
  int64_t expert_slot;  /* int32 [E + n_shared] first 128-row slot          */
  int64_t route_row;    /* int32 [T, top_k + n_shared] padded row of route  */
  int64_t row_tok;      /* int32 [rows_cap] token of each padded row        */
  int64_t row_w;        /* fp32  [rows_cap] routing weight of each row      */
  int64_t xq;           /* u8 [rows_cap, H/2] quantised activations (FP8:
                         * [rows_cap, H] E4M3)                               */
  int64_t xsf;          /* u8 tiled scales of xq (fp4moe_pack_scales layout);
                         * FP8: fp32 [rows_cap] per-row scales              */
  int64_t hq;           /* u8 [rows_cap, I/2] quantised intermediate (FP8:
                         * [rows_cap, I] E4M3)                               */
  int64_t hsf;          /* u8 tiled scales of hq; FP8: fp32 [rows_cap]      */
  int64_t h32;          /* fp32 [rows_cap, I] pre-quantisation h (NVFP4, FP8) */
  int64_t gscale;       /* fp32 [2 + E + n_shared]: g_x, spare, g_h[e]       */
  int64_t out_acc;      /* fp32 [T, H] combine accumulator                  */
  int64_t total_bytes;
  int32_t n_splits;     /* router split-K factor                            */
  int32_t n_tile;       /* tokens per GEMM tile                             */
  int32_t rows_cap;     /* rows of the padded permuted layout               */
  int32_t x_by_token;   /* 1: xq / xsf rows are token rows (few-token MXFP4
                         * path: x quantised once, the gate/up GEMM reads
                         * every token and keeps the routed ones); 0: route
                         * rows of the padded permuted layout               */
} fp4moe_ws_layout;

/* Optional instrumentation for fp4moe_forward (and the other layer entry
 * points that take one).  A zero-filled struct changes nothing.
 *   events[i] (cudaEvent_t as void*, nullable) is recorded on the stream
 *     before stage i: 0 router, 1 top-k, 2 permutation, 3 activation
 *     quantisation, 4 gate/up GEMM, 5 down GEMM, 6 finalise, 7 end.
 *   h_pre (nullable): fp32 [rows_cap, I]; when set the gate/up epilogue also
 *     writes each h value there before quantising it.
 *   logits (nullable): fp32 [T, E]; the router logits as the top-k step
 *     summed them (split-K partials added in split order).
 *   scores (nullable): fp32 [T, E]; the sigmoid scores s = 1 / (1 + e^-l)
 *     the top-k step selected from (corrected scores are fp32(s + bias)).
 *   wait_limit_ns: limit of the expert GEMMs' pipeline waits in
 *     nanoseconds; 0 keeps the default of 2 s.  The waits that drain copies
 *     already issued keep the default.
 *   withhold_first_stage: test knob, 0 in normal use.  When non-zero, CTA 0
 *     of the gate/up GEMM never fills its first pipeline stage, so that
 *     CTA's MMA issuer waits for it until wait_limit_ns runs out; the call
 *     then records FP4MOE_ERR_TIMEOUT in the status word, abandons that
 *     CTA's work (the output is not valid) and returns normally.  It
 *     exercises the timeout path without any fault.
 *   down_cta_pair: 0 in normal use.  When non-zero, down GEMM units that
 *     cover two 112-token slots (MXFP4 layers with >= 160 routes per expert,
 *     an output range of a multiple of 256 rows) run on clusters of two CTAs
 *     as M = 256 MMAs (tcgen05 .cta_group::2): one CTA issues for both SMs,
 *     each CTA holds half the weight rows and one slot of tokens.  Same
 *     results as the default single-CTA units; measured slower on GB300
 *     (the per-instruction cost of the pair's MMAs and scale copies), kept
 *     selectable for comparison. */
typedef struct {
  void *events[8];
  float *h_pre;
  float *logits;
  float *scores;
  int64_t wait_limit_ns;
  int32_t withhold_first_stage;
  int32_t down_cta_pair;
} fp4moe_debug;

/* Library version as major*10000 + minor*100 + patch. */
int32_t fp4moe_version(void);

/* Human-readable name of a status code (static string). */
const char *fp4moe_status_string(int32_t status);

/* Workspace bytes fp4moe_forward needs for these dims (0 on invalid dims). */
size_t fp4moe_workspace_size(const fp4moe_dims *dims);

/* Fills *out with the workspace layout of these dims. */
fp4moe_status fp4moe_workspace_layout(const fp4moe_dims *dims, fp4moe_ws_layout *out);

/* Bytes of the tiled scale layout for n_mat matrices of `rows` rows and
 * `kblocks` scale blocks per row (rows % 128 == 0, kblocks % 4 == 0). */
size_t fp4moe_packed_scales_bytes(int64_t n_mat, int32_t rows, int32_t kblocks, int32_t fmt);

/* Repacks row-major block scales src[n_mat, rows, kblocks] into the tiled
 * layout the GEMMs load: for each matrix, 128-row tile and group of four
 * blocks, 512 bytes where row r = 32*m1 + m0 and block k1 sit at byte
 * 16*m0 + 4*m1 + k1.  Groups are padded to whole 256-value K tiles with the
 * scale 1.0.  This is the one-time weight preparation step, the counterpart
 * of the pre-shuffled weight operand of "Serve Kimi-K2.5-MXFP4 on MI355X with
 * ATOM", section "Stage C: MXFP4 Linear GEMM".  dst holds
 * fp4moe_packed_scales_bytes bytes. */
fp4moe_status fp4moe_pack_scales(const uint8_t *src, uint8_t *dst, int64_t n_mat, int32_t rows,
                                 int32_t kblocks, int32_t fmt, void *stream);

/* The block scales of gate/up matrices src[n_mat, 2I, kblocks] (rows 0..I-1
 * gate, I..2I-1 up; I % 128 == 0) in the gate/up-paired order: the same
 * 512-byte groups as fp4moe_pack_scales, but per matrix ordered by pair p
 * (row tiles p and p + I/128), K tile kt, then gate before up, so that the
 * gate and up groups of one K tile are adjacent.  With A groups per K tile
 * (MXFP4 2, NVFP4 4) and KT K tiles, group a of K tile kt of row tile
 * h*(I/128) + p (h: 0 gate, 1 up) of matrix m sits at byte
 *   ((((m*(I/128) + p)*KT + kt)*2 + h)*A + a) * 512.
 * dst holds fp4moe_packed_scales_bytes(n_mat, 2I, kblocks, fmt) bytes.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE. */
fp4moe_status fp4moe_pack_gateup_scales(const uint8_t *src, uint8_t *dst, int64_t n_mat, int32_t I,
                                        int32_t kblocks, int32_t fmt, void *stream);

/* Bytes of the tiled payload layout for n_mat FP4 matrices of `rows` rows
 * and `kbytes` bytes per row (rows % 128 == 0, kbytes % 16 == 0): each row
 * padded to whole K tiles of 128 bytes (256 FP4 values).  0 for an
 * unsupported shape. */
size_t fp4moe_packed_weights_bytes(int64_t n_mat, int32_t rows, int32_t kbytes);

/* Repacks row-major FP4 payloads src[n_mat, rows, kbytes] into the tiled
 * layout the GEMMs can stream as whole tiles: for each matrix, 128-row tile
 * rt and K tile kt (row-major order, kt innermost), one contiguous block of
 * 128 rows x 128 bytes holding bytes kt*128 .. kt*128+127 of those rows,
 * zero codes past kbytes.  Byte (r, c) of matrix m lands at
 *   m*rows*KT*128 + ((r/128)*KT + c/128)*16384 + (r%128)*128 + c%128,
 * KT = ceil(kbytes/128).  With the scale repacking of fp4moe_pack_scales
 * this is the one-time weight preparation, the counterpart of the
 * pre-shuffled weight operand of "Serve Kimi-K2.5-MXFP4 on MI355X with
 * ATOM", section "Stage C: MXFP4 Linear GEMM".  src and dst are device
 * buffers (dst: fp4moe_packed_weights_bytes bytes, not overlapping src);
 * stream ordered.  Errors: INVALID_ARG (null pointer), UNSUPPORTED_SHAPE. */
fp4moe_status fp4moe_pack_weights(const uint8_t *src, uint8_t *dst, int64_t n_mat, int32_t rows, int32_t kbytes,
                                  void *stream);

/* The tiled payload layout of gate/up matrices src[n_mat, 2I, kbytes]
 * (rows 0..I-1 gate, I..2I-1 up; I % 128 == 0) in the gate/up-paired order:
 * the blocks of fp4moe_pack_weights, per matrix ordered by pair p, K tile kt,
 * then gate before up.  Byte (r, c) of matrix m, with P = I/128,
 * rt = r/128 = h*P + p, lands at
 *   m*2I*KT*128 + (((p*KT + c/128)*2 + h))*16384 + (r%128)*128 + c%128.
 * Same size as fp4moe_pack_weights(n_mat, 2I, kbytes).  Errors: INVALID_ARG,
 * UNSUPPORTED_SHAPE. */
fp4moe_status fp4moe_pack_gateup_weights(const uint8_t *src, uint8_t *dst, int64_t n_mat, int32_t I, int32_t kbytes,
                                         void *stream);

/* Router: logits, sigmoid + bias, grouped top-k and routing weights
 * ("Kimi-K2.7-Code on Gaudi 2", section "What was built").
 *   x [T, H] bf16, w_router [E, H] bf16, bias [E] fp32 ->
 *   topk_idx [T, top_k] int32 (descending corrected score, ties to the lower
 *   expert index), topk_w [T, top_k] fp32, logits_out [T, E] fp32 (nullable).
 * ws: a workspace of fp4moe_workspace_size(dims) bytes. */
fp4moe_status fp4moe_route(const fp4moe_dims *dims, const uint16_t *x, const uint16_t *w_router,
                           const float *bias, int32_t *topk_idx, float *topk_w, float *logits_out,
                           void *ws, size_t ws_bytes, void *stream);

/* Size of the fixed device scratch array used by fp4moe_route_noalloc. */
#define FP4MOE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* Router for callers that cannot allocate device memory (no counterpart on the
 * pages: it is fp4moe_route with its scratch moved into the library).
 * Engines that plan all device memory ahead and forbid later allocations, or
 * code that must not call cudaMalloc because it may synchronise the device,
 * cannot hand fp4moe_route a workspace.  This entry point keeps the scratch
 * in one file-scope device array of FP4MOE_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library holds until process exit, and allocates nothing
 * itself.
 *   Arguments and outputs as fp4moe_route, without the workspace.
 *   Scratch per call: a 256-byte status word, then ceil(T/32) * (E +
 *   n_shared) * 4 bytes of per-chunk expert counts rounded up to 256, then
 *   n_splits * T * E * 4 bytes of partial logits.  n_splits is
 *   fp4moe_route's split count (fp4moe_workspace_layout) when that fits, else
 *   the largest divisor of H / 256 below it that fits; the logits are then
 *   summed in another order than fp4moe_route's, so near-ties may route
 *   differently.  fp4moe_route_noalloc_scratch_bytes gives the bytes a call
 *   uses (0: the dims do not fit even with one split, or are invalid).
 *   Returns FP4MOE_ERR_WORKSPACE when not even one split fits.
 *   Each call looks up the array's device address with the device current;
 *   make the first call on each device before any stream capture.
 *   All calls share the array: calls that overlap on the GPU race, so
 *   serialise them (one stream, or host-side ordering).  Each call clears the
 *   status word and the counts; the array otherwise keeps the last call's
 *   data.  A device wait that times out is recorded in the array's status
 *   word; fp4moe_route_noalloc_status reads it. */
size_t fp4moe_route_noalloc_scratch_bytes(const fp4moe_dims *dims);
fp4moe_status fp4moe_route_noalloc(const fp4moe_dims *dims, const uint16_t *x, const uint16_t *w_router,
                                   const float *bias, int32_t *topk_idx, float *topk_w, float *logits_out,
                                   void *stream);

/* Synchronises `stream` and reads the status word of the last
 * fp4moe_route_noalloc call on the current device: *st the first recorded
 * condition (FP4MOE_OK if none), *count how many were recorded.  Either
 * output may be NULL.  Allocates nothing. */
fp4moe_status fp4moe_route_noalloc_status(void *stream, fp4moe_status *st, int64_t *count);

/* Activation quantisation ("Serve Kimi-K2.5-MXFP4 on MI355X with ATOM",
 * section "Stage B: Dynamic Activation Quantization"; "Serving NVFP4 models on
 * AMD Instinct MI355 accelerators", section "Weight Dequantization and
 * Activation QDQ").
 *   x [rows, cols] bf16 (x_is_fp32 = 0) or fp32 (x_is_fp32 = 1), row-major.
 *   codes [rows, cols/2] packed E2M1 (element 2j in the low nibble), each the
 *   round-to-nearest-even grid point (ties to the even code, saturating at
 *   +-6, sign bit kept: a negative value that rounds to zero gives code 0x8).
 *   scales row-major: MXFP4 [rows, cols/32] E8M0 bytes, e = floor(log2 amax)
 *   - 2; NVFP4 [rows, cols/16] E4M3 bytes.
 *   NVFP4 tensor scale: global_in (nullable, fp32 device scalar) is used when
 *   given, else g = amax(x) / 2688 is computed over the whole tensor; the g
 *   used is written to global_out (nullable).
 *   cols % 32 == 0.  ws must hold >= 256 bytes (amax scratch + status). */
fp4moe_status fp4moe_quantize_act(const void *x, int32_t x_is_fp32, int64_t rows, int32_t cols,
                                  int32_t fmt, const float *global_in, uint8_t *codes,
                                  uint8_t *scales, float *global_out, void *ws, size_t ws_bytes,
                                  void *stream);

/* The whole MoE layer: out[T, H] (bf16) for x[T, H] (bf16).  All weights as
 * in fp4moe_weights.  dbg is nullable.  ws: fp4moe_workspace_size(dims) bytes;
 * its intermediates stay readable after the call (fp4moe_workspace_layout). */
fp4moe_status fp4moe_forward(const fp4moe_dims *dims, const fp4moe_weights *w, const uint16_t *x,
                             uint16_t *out, const fp4moe_debug *dbg, void *ws, size_t ws_bytes,
                             void *stream);

/* The layer restricted to output columns [h_begin, h_end): the per-rank step
 * of an output-partitioned tensor-parallel MoE ("Inside the Kimi K3
 * optimization effort", section "MoE: remove duplicate work across GPUs":
 * each rank adds only its owned output coordinates, the existing all-reduce
 * assembles the layer output, and each rank needs only its rows of the down
 * projection).  Routing, activation quantisation and the gate/up GEMM run in
 * full; the down GEMM reads rows [h_begin, h_end) of w2 (and sh2) only and
 * writes those columns of out; every other column of out is zero, so the
 * ranks' outputs sum exactly to the layer output.  Arguments as for
 * fp4moe_forward (MXFP4 / NVFP4); 0 <= h_begin < h_end <= H, both multiples
 * of 128 (of 256 with packed == 3), else FP4MOE_ERR_UNSUPPORTED_SHAPE. */
fp4moe_status fp4moe_forward_cols(const fp4moe_dims *dims, const fp4moe_weights *w, const uint16_t *x,
                                  uint16_t *out, int32_t h_begin, int32_t h_end, const fp4moe_debug *dbg,
                                  void *ws, size_t ws_bytes, void *stream);

/* The W8A8 MoE layer on the exactly converted FP8 experts ("Kimi-K2.7-Code on
 * Gaudi 2", section "Exact MXFP4 to FP8 per-channel conversion": per-channel
 * FP8 weights, dynamic per-token FP8 activations).  Routing and permutation
 * as in fp4moe_forward; each token's x and each route's intermediate h are
 * quantised to E4M3 with sigma = amax / 448 over the row (code = RNE(v /
 * sigma), saturating; both correctly rounded fp32 steps; sigma = 0 gives
 * signed zeros); the expert GEMMs multiply E4M3 by E4M3 on the tensor cores
 * and apply the weight row scale and sigma in their epilogues.
 *   dims->fmt must be FP4MOE_FP8; w as fp4moe_fp8_weights; x, out bf16
 *   [T, H]; ws: fp4moe_workspace_size(dims) bytes (its layout as
 *   fp4moe_workspace_layout describes, with the FP8 meanings); dbg as for
 *   fp4moe_forward (nullable).  Pointers 16-byte aligned. */
fp4moe_status fp4moe_forward_w8a8(const fp4moe_dims *dims, const fp4moe_fp8_weights *w, const uint16_t *x,
                                  uint16_t *out, const fp4moe_debug *dbg, void *ws, size_t ws_bytes,
                                  void *stream);

/* The NVFP4 layer in emulation mode ("Serving NVFP4 models on AMD Instinct
 * MI355 accelerators", sections "Weight Dequantization and Activation QDQ"
 * and "Memory Management"): the dispatched experts' NVFP4 weights are
 * dequantised to BF16 at call time into the workspace, x and the
 * intermediate pass through an NVFP4 quantise-dequantise round trip into
 * BF16, and the expert GEMMs multiply BF16 by BF16 with fp32 accumulation.
 * Each BF16 value is bf16_rn(fp32(E2M1(q) * fp32(E4M3(s) * g))).  A reference
 * and speed comparison for the native NVFP4 fp4moe_forward.
 *   dims->fmt FP4MOE_NVFP4; w as for fp4moe_forward (NVFP4); ws:
 *   fp4moe_emulation_workspace_size(dims) bytes (the forward's layout first,
 *   then BF16 rows of x and h and BF16 copies of every expert matrix). */
size_t fp4moe_emulation_workspace_size(const fp4moe_dims *dims);
fp4moe_status fp4moe_forward_nvfp4_emulated(const fp4moe_dims *dims, const fp4moe_weights *w, const uint16_t *x,
                                            uint16_t *out, const fp4moe_debug *dbg, void *ws, size_t ws_bytes,
                                            void *stream);

/* Dense block-scaled FP4 linear layer ("Serve Kimi-K2.5-MXFP4 on MI355X with
 * ATOM", section "Stage C: MXFP4 Linear GEMM": bf16 activations quantised
 * on the fly, block-scaled FP4 product, bf16 output):
 *   out[T, N] = quantize(x)[T, K] . W[N, K]^T
 *   x bf16 [T, K] quantised as fp4moe_quantize_act does (MXFP4 per 32;
 *   NVFP4 per 16 with one tensor scale over x); w packed FP4 [N, K/2];
 *   w_scale its block scales repacked by fp4moe_pack_scales (n_mat = 1,
 *   rows = N); g_w NVFP4 only: device fp32 tensor scale of W (NULL for MXFP4).
 *   1 <= T <= 65536, K % 256 == 0, N % 256 == 0.  ws:
 *   fp4moe_linear_workspace_size bytes.  Pointers 16-byte aligned. */
size_t fp4moe_linear_workspace_size(int32_t fmt, int32_t T, int32_t K, int32_t N);
fp4moe_status fp4moe_linear(int32_t fmt, int32_t T, int32_t K, int32_t N, const uint16_t *x, const uint8_t *w,
                            const uint8_t *w_scale, const float *g_w, uint16_t *out, void *ws, size_t ws_bytes,
                            void *stream);

/* Exact MXFP4 -> FP8 (E4M3) per-channel conversion ("Kimi-K2.7-Code on
 * Gaudi 2", section "Exact MXFP4 to FP8 per-channel conversion").
 *   codes [rows, K/2] packed E2M1, scales [rows, K/32] E8M0 row-major ->
 *   fp8_out [rows, K] E4M3 bytes, row_scale [rows] fp32 = 2^k with
 *   k = floor(log2 max|v|) - 7, row_status [rows] (nullable): 0 exact and
 *   every element exponent in [-5, 7]; 1 some element below the -5 floor
 *   (written round-to-nearest-even, possibly inexact); 2 a scale byte 255
 *   (bytes 0, scale NaN).  All-zero rows: scale 1.0.  K % 32 == 0.
 *   Rows with status 1 or 2 are counted in the workspace status word
 *   (FP4MOE_ERR_INEXACT / FP4MOE_ERR_NAN_SCALE); ws >= 256 bytes. */
fp4moe_status fp4moe_mxfp4_to_fp8_rowscale(const uint8_t *codes, const uint8_t *scales_e8m0,
                                           int64_t rows, int32_t K, uint8_t *fp8_out,
                                           float *row_scale, uint8_t *row_status, void *ws,
                                           size_t ws_bytes, void *stream);

/* Weight validation: counts the NaN block-scale bytes among n bytes of
 * scales (MXFP4: E8M0 byte 255, "Serve Kimi-K2.5-MXFP4 on MI355X with ATOM",
 * section "The Kimi-K2.5-MXFP4 Model on gfx950"; NVFP4: E4M3 bytes 0x7F and
 * 0xFF).  The layer does not test its weight scales on every call, since
 * that would read them again; run this once on each scale tensor (row-major
 * or repacked by fp4moe_pack_scales: every byte is a scale or the padding
 * scale 1.0).  NaN bytes are recorded in the status word of ws (>= 256
 * bytes) as FP4MOE_ERR_NAN_SCALE with their count; fp4moe_get_status reads
 * it.  scales 16-byte aligned.  Errors: INVALID_ARG, WORKSPACE, DEVICE. */
fp4moe_status fp4moe_check_scales(const uint8_t *scales, int64_t n, int32_t fmt, void *ws, size_t ws_bytes,
                                  void *stream);

/* Clears the workspace status word (asynchronous). */
fp4moe_status fp4moe_clear_status(void *ws, void *stream);

/* Synchronises `stream` and reads the workspace status word: *st the first
 * recorded condition (FP4MOE_OK if none), *count how many were recorded.
 * Either output may be NULL. */
fp4moe_status fp4moe_get_status(void *ws, void *stream, fp4moe_status *st, int64_t *count);

#ifdef __cplusplus
}
#endif

#endif /* FP4MOE_H */
