/*
 * nvfp4moe.h -- C ABI of the NVFP4 mixture-of-experts decode path for GB300
 * (sm_103a).
 *
 * The operation: a routed mixture-of-experts FFN whose weights are NVFP4 --
 * FP4 E2M1 elements, one E4M3 block scale per 16 elements along K, and one
 * FP32 per-tensor scale ("The Benchmark That Confirmed the Ceiling: NVFP4
 * Cutlass on sm_120", section "The NVFP4 Pivot").  One layer is
 *   route top-k -> permute by expert -> grouped GEMM gate_up -> SwiGLU ->
 *   requantise to NVFP4 -> grouped GEMM down -> weighted combine,
 * with tiny and ragged per-expert M ("The 2x Gap: Diagnosing Suboptimal FP4
 * GEMM Kernels on Blackwell SM120", section "The Investigation So Far":
 * 256 experts, 8 active, ~16 tokens per expert).  Modes: W4A4 (FP4
 * activations too) and W4A16 (BF16 activations, FP4 weights dequantised in
 * the kernel) ("The 24% Ceiling", section "The Core Insight"); W4A8 (FP8
 * activations, "Native FP4 Is Slower Than Emulated FP4", section 1); and
 * MXFP4 weights and activations.
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers unless a comment says otherwise.  The
 *    caller owns and frees every buffer; the library never allocates device
 *    memory and keeps no per-call state (only cached device properties and
 *    kernel attributes).
 *  - Every call only enqueues work on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns without synchronising.
 *  - Kernels are launched as programmatic dependents of the preceding kernel
 *    on the stream: a kernel's prologue (barrier setup, TMEM allocation) may
 *    overlap that kernel's end, but it reads and writes memory only after
 *    that kernel has completed, so stream order holds as with plain launches.
 *    Inside moe_layer_forward the W4A4 and MXFP4 grouped GEMMs also read the
 *    routing and start their first weight copies during that overlap: both
 *    were final before the preceding kernel started, so the order is the
 *    same.
 *  - Arguments are validated on the host before anything is launched, so a
 *    failing call launches nothing.  The return value is an nvfp4_status.
 *  - Kernels that consume routing data check it and report problems through
 *    the optional `dev_status` word (int32, device memory; the kernel writes
 *    a nonzero nvfp4_status there and skips the bad work; it never traps).
 *  - All device pointers must be 16-byte aligned.
 *  - Layouts are row-major.  NVFP4 tensors [rows, cols] are stored as
 *      codes  uint8 [rows, cols/2]  (element 2i in the low nibble of byte i)
 *      scales uint8 [rows, cols/16] (E4M3 "FN" block scales, linear)
 *      S      fp32 scalar           (per-tensor decode scale)
 *    and decode as value = e2m1(code) * e4m3(scale) * S.
 *  - Requires compute capability 10.3 (GB300); other devices get
 *    NVFP4_E_ARCH.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t; /* the same type as cudaStream_t */

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_E_INVAL = 1,          /* null pointer, negative size, bad enum       */
  NVFP4_E_SHAPE = 2,          /* a size violates a documented constraint     */
  NVFP4_E_ALIGN = 3,          /* a pointer is not 16-byte aligned            */
  NVFP4_E_WORKSPACE = 4,      /* workspace missing or too small              */
  NVFP4_E_ARCH = 5,           /* device is not compute capability 10.3       */
  NVFP4_E_CUDA = 6,           /* a CUDA runtime/driver call failed           */
  NVFP4_E_DEVICE_TIMEOUT = 7, /* (device) a bounded wait ran out             */
  NVFP4_E_BAD_ROUTING = 8     /* (device) inconsistent expert offsets / ids  */
} nvfp4_status;

enum { NVFP4_DT_BF16 = 0, NVFP4_DT_F32 = 1 };
enum { NVFP4_SCALE_STATIC = 0, NVFP4_SCALE_DYNAMIC = 1 };
enum { MOE_W4A4 = 0, MOE_W4A16 = 1, MOE_MXW4A4 = 2, MOE_W4A8 = 3, MOE_W4A16F = 4 };
enum { MOE_ACT_NONE = 0, MOE_ACT_NVFP4 = 1, MOE_ACT_BF16 = 2 };

/* Human-readable name of a status code (static string, never NULL). */
const char* nvfp4_status_string(int status);

/* Checks that the current device is a GB300 (CC 10.3) and caches its
 * properties.  Returns NVFP4_OK or NVFP4_E_ARCH / NVFP4_E_CUDA. */
int nvfp4_device_check(void);

/* ------------------------------------------------------------------------
 * nvfp4_quantize -- NVFP4 quantisation of a row-major matrix.
 * Defined by "The Benchmark That Confirmed the Ceiling", section "The NVFP4
 * Pivot" (group-16 E4M3 scales over FP4 E2M1) and the per-tensor `alpha` of
 * the scaled FP4 GEMM interface ("The 2x Gap", section "Discovering the
 * sgl_kernel Alternative").  Per 16-element block along a row:
 *   b = (amax_block / 6) / S               (two fp32 IEEE divisions)
 *   scale = E4M3(b)                        (round-to-nearest-even, saturate 448)
 *   d = e4m3(scale) * S                    (fp32)
 *   code_i = E2M1(x_i / d)                 (RNE, saturate 6, sign kept)
 * S == 0 or d == 0 gives scale 0 and codes 0.
 *   x          [rows, cols] of x_dtype (NVFP4_DT_BF16 or NVFP4_DT_F32), row
 *              stride ld_x elements (ld_x >= cols)
 *   S          device fp32 scalar.  scale_mode NVFP4_SCALE_STATIC: read.
 *              NVFP4_SCALE_DYNAMIC: written with amax(|x|) / 2688.
 *   codes      out [rows, cols/2]; scales out [rows, cols/16]
 *   workspace  >= nvfp4_quantize_workspace_bytes() bytes (dynamic mode only;
 *              may be NULL in static mode)
 * Constraints: cols % 16 == 0, ld_x % 8 == 0 (bf16) / % 4 == 0 (f32).
 * ------------------------------------------------------------------------ */
size_t nvfp4_quantize_workspace_bytes(int64_t rows, int64_t cols);
int nvfp4_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x, float* S,
                   int scale_mode, uint8_t* codes, uint8_t* scales, void* workspace, size_t workspace_bytes,
                   nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * nvfp4_pack_weight_scales -- one-time reshuffle of expert weight block
 * scales from the linear layout [E, N, K/16] into the layout the grouped
 * GEMM reads (no counterpart on the pages; it is weight preparation, done
 * once per set of weights, outside the per-step path).
 * Packed layout: for expert e, 128-row tile nt = n / 128, 64-column block
 * kb = k / 64, a 512-byte atom at byte offset ((e*N/128 + nt)*K/64 + kb)*512;
 * inside it, row r = n % 128 and scale j = (k % 64) / 16 sit at byte
 * (r % 32) * 16 + (r / 32) * 4 + j.
 *   scales_linear  [E, N, K/16];  scales_packed  out, E*N*K/16 bytes.
 * Constraints: N % 128 == 0, K % 256 == 0.
 * ------------------------------------------------------------------------ */
int nvfp4_pack_weight_scales(const uint8_t* scales_linear, int E, int N, int K, uint8_t* scales_packed,
                             nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP4 -- the group-32 format with UE8M0 (power-of-two) block scales that
 * "The Benchmark That Confirmed the Ceiling", sections "The Optimization Hierarchy" and
 * "The NVFP4 Pivot", names as the stock checkpoint's.  The pages define only
 * the block size and the scale type; the conversion follows the OCP MX rule:
 *   per 32-element block: E = floor(log2(amax)) - 2, clamped to [-127, 127]
 *   (an all-zero block takes -127); scale code E + 127 (UE8M0, value
 *   2^(code-127)); element code = E2M1(RNE, satfinite, sign kept) of
 *   x * 2^-E.  No per-tensor scale.
 * Layouts: codes as NVFP4 (two per byte, element 2i in the low nibble);
 * activation scales [rows, mxfp4_scale_pitch(cols)] bytes, the row pitch
 * being cols/32 rounded up to a multiple of 16 and at least 128 (padding
 * written as zero) so that the grouped GEMM fetches them efficiently with TMA.
 * Mode MOE_MXW4A4 of the grouped GEMM, SwiGLU/requant and layer calls runs
 * both operands in MXFP4 on tcgen05.mma kind::mxf4nvf4 .scale_vec::2X.
 * ------------------------------------------------------------------------ */
int64_t mxfp4_scale_pitch(int64_t cols);

/* mxfp4_quantize -- x [rows, cols] (bf16 or fp32, row stride ld_x elements)
 * to codes [rows, cols/2] and scales [rows, mxfp4_scale_pitch(cols)].
 * Constraints: cols % 32 == 0; ld_x >= cols, ld_x % 8 == 0 (bf16) or % 4 == 0
 * (fp32); x and codes 16-byte aligned. */
int mxfp4_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* codes,
                   uint8_t* scales, nvfp4_stream_t stream);

/* mxfp4_pack_weight_scales -- one-time reshuffle of MXFP4 expert weight
 * scales from the linear layout [E, N, K/32] into the layout the grouped
 * GEMM reads (weight preparation, no counterpart on the pages).  For expert
 * e, 128-row tile nt = n / 128 and 64-column block kb = k / 64, a 256-byte
 * block at ((e*N/128 + nt)*K/64 + kb)*256; inside it, row r = n % 128 and
 * scale j = (k % 64) / 32 sit at byte (r % 32) * 8 + (r / 32) * 2 + j.
 *   scales_linear  [E, N, K/32];  scales_packed  out, E*N*K/32 bytes.
 * Constraints: N % 128 == 0, K % 256 == 0. */
int mxfp4_pack_weight_scales(const uint8_t* scales_linear, int E, int N, int K, uint8_t* scales_packed,
                             nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_quantize -- FP8 activations for the W4A8 mode.  "Native FP4 Is Slower
 * Than Emulated FP4", section 1: NVFP4 as "FP4 weights with FP8
 * activations".  The page gives the element type only; the scale is read as
 * one fp32 per-tensor decode scale, as for NVFP4's tensor level:
 *   S = amax(|x|) / 448                   (dynamic; or a caller-given S)
 *   code = sign(x / S) | E4M3(|x / S|)    (x / S one fp32 IEEE division;
 *                                          RNE, saturating at 448; the sign
 *                                          bit is kept when the magnitude
 *                                          rounds to zero)
 *   value = e4m3(code) * S; S == 0 gives all codes 0.
 *   x          [rows, cols] of x_dtype (NVFP4_DT_BF16 or NVFP4_DT_F32), row
 *              stride ld_x elements
 *   S          device fp32 scalar; NVFP4_SCALE_STATIC: read,
 *              NVFP4_SCALE_DYNAMIC: written
 *   codes      out [rows, cols], one E4M3 byte per element
 *   workspace  >= nvfp4_quantize_workspace_bytes() bytes (dynamic mode only)
 * Constraints: cols % 16 == 0; ld_x % 8 == 0 (bf16) or % 4 == 0 (f32).
 * ------------------------------------------------------------------------ */
int fp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x, float* S, int scale_mode,
                 uint8_t* codes, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_router_logits -- the router scores that the routing step ranks ("The
 * 2x Gap", section "The Investigation So Far": each token goes to 8 of 256
 * experts by these scores):
 *   logits[t, e] = sum_h x[t, h] * w_router[e, h]
 * bf16 inputs, fp32 accumulation on the tensor cores, fp32 output.  K is
 * split over the SMs and the partial sums are added in a fixed order, so
 * the result is reproducible bit for bit.  Its output feeds
 * moe_align_permute / moe_route_quantize_nvfp4 / _mxfp4 directly.
 *   x bf16 [T, H]; w_router bf16 [E, H]; logits fp32 [T, E]
 *   workspace >= moe_router_logits_workspace_bytes(T, H, E) (for the current
 *   device: the split depends on its SM count)
 *   dev_status: optional; a bounded device wait that runs out sets
 *   NVFP4_E_DEVICE_TIMEOUT.
 * Constraints: H % 64 == 0, T >= 0, E >= 1; pointers 16-byte aligned.
 * ------------------------------------------------------------------------ */
size_t moe_router_logits_workspace_bytes(int T, int H, int E);
int moe_router_logits(const void* x, const void* w_router, int T, int H, int E, float* logits,
                      int32_t* dev_status, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_router_route -- the router and the routing in one call: router logits
 * (as moe_router_logits), then top-k, softmax and the expert permutation (as
 * moe_align_permute) ("The 2x Gap", section "The Investigation So Far": each
 * token goes to 8 of 256 experts by these scores).  For a decode batch
 * (T <= 32) it is two kernels: the router GEMM, then one kernel that sums the
 * GEMM's K-range partials in a fixed order, selects the top k of each token
 * and builds the permutation; larger T runs the router GEMM, its reduce and
 * the routing kernel.  Either way the results are bitwise those of
 * moe_router_logits followed by moe_align_permute.
 *   x bf16 [T, H]; w_router bf16 [E, H]
 *   logits  optional out fp32 [T, E] (NULL: not returned)
 *   topk_ids, topk_w, expert_offsets, perm, inv: as moe_align_permute
 *   workspace >= moe_router_route_workspace_bytes(T, H, E, k) (for the
 *   current device)
 *   dev_status: optional; NVFP4_E_DEVICE_TIMEOUT from the router GEMM's
 *   bounded waits, NVFP4_E_BAD_ROUTING from the routing.
 * Constraints: H % 64 == 0, 1 <= k <= min(E, 32), E <= 1024.
 * ------------------------------------------------------------------------ */
size_t moe_router_route_workspace_bytes(int T, int H, int E, int k);
int moe_router_route(const void* x, const void* w_router, int T, int H, int E, int k, float* logits,
                     int32_t* topk_ids, float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv,
                     int32_t* dev_status, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_align_permute -- router top-k plus the expert permutation.
 * Routing: "The 2x Gap", section "The Investigation So Far" (top-8 of 256
 * experts); "Native FP4 Is Slower ...", section 1 (22 of 512).  Per token t:
 *   topk_ids[t, :] = the k experts with the largest logits, in descending
 *                    logit order, ties to the lower expert id;
 *   topk_w[t, j]   = exp(l_j - l_max) / sum over the k selected (fp32).
 * Permutation ("expert-scatter-gather", "The 2x Gap", same section): the
 * T*k (token, slot) pairs sorted stably by (expert, token):
 *   expert_offsets [E+1]: exclusive prefix sum of per-expert counts;
 *   perm[r]             : source token of permuted row r;
 *   inv[t*k + j]        : permuted row of pair (t, j).
 * Optional gather (act_kind != MOE_ACT_NONE): permuted activation rows
 *   act_out[r] = act_in[perm[r]]; NVFP4 rows copy codes [.., act_cols/2] and
 *   scales [.., act_cols/16]; BF16 rows copy [.., act_cols] bf16.
 *   logits  fp32 [T, E];  topk_ids int32 [T, k];  topk_w fp32 [T, k]
 *   workspace >= moe_align_permute_workspace_bytes(T, E, k)
 * Constraints: 1 <= k <= min(E, 32), E <= 1024, T >= 0; act_cols % 32 == 0.
 * ------------------------------------------------------------------------ */
size_t moe_align_permute_workspace_bytes(int T, int E, int k);
int moe_align_permute(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                      int32_t* expert_offsets, int32_t* perm, int32_t* inv, int act_kind, const void* act_in,
                      const uint8_t* act_in_scales, int64_t act_cols, void* act_out, uint8_t* act_out_scales,
                      int32_t* dev_status, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_route_quantize_nvfp4 -- the W4A4 front half of the layer in one call:
 * routing and permutation exactly as moe_align_permute, and the activations
 * x quantised to NVFP4 with the dynamic per-tensor scale exactly as
 * nvfp4_quantize, written straight into permuted order.  Results are
 * identical to nvfp4_quantize(x, DYNAMIC) followed by moe_align_permute with
 * an NVFP4 gather; the fused form reads x once (routing and amax in one
 * pass) and skips the unpermuted intermediate.
 *   x bf16 [T, H]; logits fp32 [T, E]
 *   outputs: topk_ids, topk_w, expert_offsets, perm, inv as in
 *   moe_align_permute; S_x (device fp32 scalar, amax(|x|)/2688); a_codes
 *   [T*k, H/2], a_scales [T*k, H/16] in permuted row order
 *   workspace >= moe_align_permute_workspace_bytes(T, E, k)
 * Constraints: as moe_align_permute, and H % 256 == 0.
 * ------------------------------------------------------------------------ */
int moe_route_quantize_nvfp4(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                             float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, float* S_x,
                             uint8_t* a_codes, uint8_t* a_scales, int32_t* dev_status, void* workspace,
                             size_t workspace_bytes, nvfp4_stream_t stream);

/* moe_route_quantize_mxfp4 -- the same front half for MOE_MXW4A4: routing
 * and permutation as moe_align_permute, and x quantised to MXFP4 (as
 * mxfp4_quantize) straight into permuted order: a_codes [T*k, H/2], a_scales
 * [T*k, mxfp4_scale_pitch(H)].  Identical to mxfp4_quantize followed by a
 * row gather.  Constraints: as moe_route_quantize_nvfp4. */
int moe_route_quantize_mxfp4(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                             float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, uint8_t* a_codes,
                             uint8_t* a_scales, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                             nvfp4_stream_t stream);

/* moe_route_quantize_fp8 -- the same front half for MOE_W4A8: routing and
 * permutation as moe_align_permute, and x quantised to FP8 with the dynamic
 * per-tensor scale exactly as fp8_quantize, written straight into permuted
 * order: a_codes [T*k, H] (one byte per element), S_x (device fp32 scalar,
 * amax(|x|) / 448).  Constraints: as moe_route_quantize_nvfp4. */
int moe_route_quantize_fp8(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                           float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, float* S_x,
                           uint8_t* a_codes, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                           nvfp4_stream_t stream);

/* moe_route_quantize_fp8_f16 -- moe_route_quantize_fp8 with every FP8 code
 * written as its value in f16 (E4M3 values are f16 values: exact) for the
 * MOE_W4A16F GEMM: a_f16 [T*k, H] holds e4m3(code), a_rs [T*k] holds S_x for
 * every row, so that GEMM forms exactly the MOE_W4A8 products.  The layer's
 * W4A8 path runs this form.  S_x, routing outputs and constraints as
 * moe_route_quantize_fp8. */
int moe_route_quantize_fp8_f16(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                               float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, float* S_x,
                               void* a_f16, float* a_rs, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                               nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_grouped_gemm_nvfp4 -- ragged grouped GEMM over experts.
 * "The 2x Gap", sections "The Investigation So Far" and "Discovering the
 * sgl_kernel Alternative" (scaled FP4 GEMM: block scales on both operands
 * and one alpha); "The Benchmark That Confirmed the Ceiling", section "The
 * NVFP4 Pivot" (native FP4xFP4 versus W4A16 dequantise-to-BF16).  For every
 * permuted row r of expert e (expert_offsets[e] <= r < expert_offsets[e+1]):
 *   W4A4 : out[r, n] = a_S * w_S[e] * sum_k dec(a[r,k]) * dec(w[e,n,k])
 *   W4A16: out[r, n] =        w_S[e] * sum_k a[r,k]      * dec(w[e,n,k])
 *   MXW4A4: out[r, n] =              sum_k dec(a[r,k]) * dec(w[e,n,k])
 *   W4A8 : out[r, n] = a_S * w_S[e] * sum_k e4m3(a[r,k]) * dec(w[e,n,k])
 *   W4A16F: out[r, n] = a_S[r] * w_S[e] * sum_k a[r,k] * dec(w[e,n,k])
 * with dec(.) = e2m1(code) * e4m3(block scale) (MXFP4: * 2^(scale-127) per
 * 32 elements), fp32 accumulation.
 *   W4A4 : a = codes [R, K/2], a_scales = [R, K/16], a_S = device fp32 scalar
 *   W4A16: a = bf16 [R, K], a_scales = NULL, a_S = NULL
 *   MXW4A4: a = codes [R, K/2], a_scales [R, mxfp4_scale_pitch(K)], a_S and
 *          w_S unused (may be NULL)
 *   W4A8 : a = FP8 E4M3 codes [R, K] (fp8_quantize), a_scales = NULL, a_S =
 *          device fp32 scalar; runs on F16 operands (e2m1 * e4m3 weights and
 *          E4M3 activations are both exact in f16), fp32 accumulation
 *   W4A16F: the W4A16 product on bf16 rows carried as F16 (moe_gather_f16,
 *          moe_swiglu_f16): a = f16 [R, K] holding a_bf16[r] * 2^e_r, a_S =
 *          fp32 [R] holding 2^-e_r (a power of two, so the rescale is exact),
 *          a_scales = NULL; runs on F16 operands.  The weight dequantisation
 *          then needs no f16 -> bf16 widening, which made the W4A16 stage
 *          1.3x longer on GB300.
 *   w_codes        [E, N, K/2]
 *   w_scales_packed  from nvfp4_pack_weight_scales (mxfp4_pack_weight_scales)
 *   w_S            fp32 [E]
 *   expert_offsets int32 [E+1], expert_offsets[E] must equal R (checked on
 *                  the device; a violation sets dev_status to
 *                  NVFP4_E_BAD_ROUTING and skips the bad experts)
 *   out            fp32 [R, N]
 * Constraints: N % 128 == 0, K % 256 == 0, R >= 0.  Rows of out that belong
 * to no expert are not written.
 * ------------------------------------------------------------------------ */
int moe_grouped_gemm_nvfp4(int mode, const void* a, const uint8_t* a_scales, const float* a_S,
                           const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                           const int32_t* expert_offsets, int E, int N, int K, int R, float* out,
                           int32_t* dev_status, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_gather_f16 -- bf16 activation rows carried as F16 for MOE_W4A16F.
 * The pages define no such step: it is an exact carrier of the W4A16
 * operand for F16 tensor-core operands.  For r < R with src = perm[r] (or r
 * when perm is NULL):
 *   e_r       = 14 - floor(log2(max_k |x[src, k]|)), capped at 126 (0 for a
 *               row of zeros), so the row's largest magnitude maps into
 *               [2^14, 2^15) and nothing overflows f16;
 *   a_f16[r]  = f16(x[src] * 2^e_r) -- exact for every element within a
 *               factor 2^28 of the row's max (an f16 normal then), rounded to
 *               the f16 subnormal grid below that (absolute error <= 2^-39 of
 *               the row's max);
 *   a_rs[r]   = 2^-e_r (fp32).
 *   x bf16 [T, H]; perm int32 [R] (values in [0, T)) or NULL with R <= T;
 *   a_f16 f16 [R, H]; a_rs fp32 [R]
 * Constraints: H % 8 == 0; x and a_f16 16-byte aligned.
 * ------------------------------------------------------------------------ */
int moe_gather_f16(const void* x, int T, int H, const int32_t* perm, int R, void* a_f16, float* a_rs,
                   nvfp4_stream_t stream);

/* moe_swiglu_f16 -- the W4A16 SwiGLU (as moe_swiglu_requant with MOE_W4A16:
 * h = bf16(silu(g) * u)) written as F16 rows for MOE_W4A16F, with the
 * per-row powers of two of moe_gather_f16: h_f16[r] = f16(h[r] * 2^e_r),
 * h_rs[r] = 2^-e_r.  G fp32 [R, 2I]; h_f16 f16 [R, I]; h_rs fp32 [R].
 * Constraints: I % 16 == 0; G and h_f16 16-byte aligned. */
int moe_swiglu_f16(const float* G, int R, int I, void* h_f16, float* h_rs, nvfp4_stream_t stream);

/* moe_swiglu_fp8_f16 -- the W4A8 SwiGLU (as moe_swiglu_requant with MOE_W4A8:
 * FP8 codes of h with the static decode scale *S_h) with every code written
 * as its f16 value for the MOE_W4A16F GEMM: h_f16 [R, I], h_rs[r] = *S_h.
 * Constraints: I % 16 == 0; G and h_f16 16-byte aligned. */
int moe_swiglu_fp8_f16(const float* G, int R, int I, const float* S_h, void* h_f16, float* h_rs,
                       nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_swiglu_requant -- SwiGLU on the gate_up output and requantisation.
 * Defined by the layer this library implements -- gate_up, then SwiGLU,
 * then requantisation to NVFP4, then down -- which is the routed-expert FFN
 * of the models on the pages ("Native FP4 Is Slower Than Emulated FP4",
 * section 1: an NVFP4 MoE with 512 routed experts; the pages print no
 * activation formula, so SwiGLU is the layer definition's own step).  The
 * requantisation is nvfp4_quantize's rule ("The Benchmark That Confirmed the
 * Ceiling", section "The NVFP4 Pivot").
 * h[r, i] = silu(G[r, i]) * G[r, I + i], silu(x) = x / (1 + exp(-x)), fp32.
 *   W4A4 : h is quantised to NVFP4 with the static decode scale *S_h
 *          (same rule as nvfp4_quantize): h_codes [R, I/2], h_scales
 *          [R, I/16]; h_bf16 unused (NULL).
 *   W4A16: h is rounded to bf16 (RNE) into h_bf16 [R, I]; the NVFP4 outputs
 *          and S_h are unused (NULL).
 *   MXW4A4: h is quantised to MXFP4 (as mxfp4_quantize): h_codes [R, I/2],
 *          h_scales [R, mxfp4_scale_pitch(I)]; S_h and h_bf16 unused.  The
 *          block scales come from h itself, so no calibration is needed.
 *   W4A8 : h is quantised to FP8 with the static decode scale *S_h (as
 *          fp8_quantize): h_codes [R, I]; h_scales and h_bf16 unused.
 *   G fp32 [R, 2I] (gate columns 0..I-1, up columns I..2I-1).
 * Constraints: I % 16 == 0.
 * ------------------------------------------------------------------------ */
int moe_swiglu_requant(const float* G, int R, int I, int mode, const float* S_h, uint8_t* h_codes,
                       uint8_t* h_scales, void* h_bf16, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_combine -- weighted combine of the expert outputs: the scatter half
 * of the expert-scatter-gather pattern ("The 2x Gap", section "Discovering
 * the sgl_kernel Alternative"), in which the layer definition combines the
 * expert outputs with a weighted scatter.  Done here as a gather
 * (deterministic, no atomics):
 *   out[t, n] = sum_{j < k} topk_w[t, j] * Y[inv[t*k + j], n]   (fp32, j order)
 *   Y fp32 [T*k, H]; out [T, H] of out_dtype (NVFP4_DT_F32 or NVFP4_DT_BF16).
 *   inv: the caller's permutation (from moe_align_permute).  Each entry is
 *   checked on the device: an entry outside [0, T*k) contributes nothing,
 *   and sets NVFP4_E_BAD_ROUTING in dev_status (optional, may be NULL);
 *   no out-of-range row is ever read.
 * Constraints: H % 4 == 0, 1 <= k <= 32 (as routing).
 * ------------------------------------------------------------------------ */
int moe_combine(const float* Y, const int32_t* inv, const float* topk_w, int T, int k, int H, int out_dtype,
                void* out, int32_t* dev_status, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_layer_forward -- the whole layer in one call: every step above,
 * enqueued in order on `stream` with no host synchronisation, so the call
 * can be captured in a CUDA graph.
 *   mode        MOE_W4A4, MOE_W4A16, MOE_MXW4A4 or MOE_W4A8 (MOE_W4A16 runs
 *               moe_gather_f16, MOE_W4A16F GEMMs and moe_swiglu_f16: the
 *               W4A16 products, with the bf16 operands carried as F16 rows;
 *               MOE_W4A8 runs moe_route_quantize_fp8_f16, MOE_W4A16F GEMMs
 *               and moe_swiglu_fp8_f16: the W4A8 products)
 *   x           bf16 [T, H]; logits fp32 [T, E]
 *   w13_*       gate_up weights: codes [E, 2I, H/2], packed scales, S [E]
 *   w2_*        down weights:    codes [E, H, I/2],  packed scales, S [E]
 *               (MXW4A4: MXFP4 packed scales; w13_S, w2_S unused, may be NULL)
 *   S_h         device fp32 scalar, static decode scale of h (W4A4: NVFP4's
 *               per-tensor scale; W4A8: the FP8 scale; unused otherwise)
 *   out         fp32 [T, H]
 *   workspace   >= moe_layer_workspace_bytes(mode, T, H, I, E, k); holds
 *               every intermediate (routing, activations, G, h, Y)
 * Constraints: H % 256 == 0, I % 256 == 0 (2I and H % 128 follow).
 * ------------------------------------------------------------------------ */
size_t moe_layer_workspace_bytes(int mode, int T, int H, int I, int E, int k);
int moe_layer_forward(int mode, const void* x, const float* logits, int T, int H, int I, int E, int k,
                      const uint8_t* w13_codes, const uint8_t* w13_scales_packed, const float* w13_S,
                      const uint8_t* w2_codes, const uint8_t* w2_scales_packed, const float* w2_S,
                      const float* S_h, float* out, int32_t* dev_status, void* workspace,
                      size_t workspace_bytes, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_layer_forward_host -- moe_layer_forward from and to page-locked host
 * memory, for a caller whose step inputs arrive on the host and whose result
 * is read there (one decode step end to end).  An interface convenience of
 * this library: the computation is moe_layer_forward's.
 *   x_host       bf16 [T, H], page-locked (cudaHostAlloc / registered)
 *   logits_host  fp32 [T, E], page-locked
 *   out_host     fp32 [T, H], page-locked; written by the device
 *   other arguments as for moe_layer_forward
 *   workspace    >= moe_layer_host_workspace_bytes(mode, T, H, I, E, k):
 *                moe_layer_workspace_bytes plus device copies of x and logits
 * The copies are kernels, not DMA transfers: a staging kernel reads x and
 * logits over the host link into the workspace, and the combine kernel
 * writes each output row straight into out_host, so the whole step is one
 * chain of programmatically dependent kernels (no copy-engine nodes when
 * captured in a graph).  The result is bitwise that of moe_layer_forward.
 * out_host is complete once the stream's work up to this call has finished.
 * Errors: NVFP4_E_INVAL if a buffer is not page-locked host memory; the
 * other codes as for moe_layer_forward.
 * ------------------------------------------------------------------------ */
size_t moe_layer_host_workspace_bytes(int mode, int T, int H, int I, int E, int k);
int moe_layer_forward_host(int mode, const void* x_host, const float* logits_host, int T, int H, int I, int E, int k,
                           const uint8_t* w13_codes, const uint8_t* w13_scales_packed, const float* w13_S,
                           const uint8_t* w2_codes, const uint8_t* w2_scales_packed, const float* w2_S,
                           const float* S_h, float* out_host, int32_t* dev_status, void* workspace,
                           size_t workspace_bytes, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_align_permute_noalloc -- moe_align_permute for callers that cannot
 * give the library scratch memory.  (The reference pages have no counterpart:
 * this is an interface convenience of this library, not a step of the method.)
 *
 * Some callers own every byte of device memory themselves -- a serving engine
 * or plugin host with one pre-reserved arena and no workspace hook -- or run
 * latency-critical code that must never call cudaMalloc, which can
 * synchronise the whole device.  They can pass inputs and outputs but no
 * workspace.  This entry point computes exactly what moe_align_permute
 * computes (same arguments and results, minus `workspace`) and keeps its
 * scratch in a fixed array of NVFP4MOE_NOALLOC_SCRATCH_BYTES bytes inside the
 * library's own device memory: it allocates nothing and calls no allocating
 * routine.
 *   - Limit: a call needs 256 + 4 * B * E + 4 * B bytes of scratch (each
 *     term after the first rounded up to 256), B = ceil(T / 32); a larger
 *     problem (e.g. T > 4064 tokens at E = 1024 experts, T > 32480 at
 *     E = 128) is refused with NVFP4_E_WORKSPACE before anything is
 *     launched.  (Where the array holds four times that, routing runs in
 *     blocks of eight tokens as moe_align_permute does from 33 tokens;
 *     otherwise in blocks of 32: the results are the same.)
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current), and so does the first call
 *     after a device reset (cudaDeviceReset destroys the context, and the
 *     next one may hold the array at another address); make those calls
 *     before any stream capture.
 *   - The array is shared by every call on a device and stays allocated while
 *     the library is loaded.  Calls that overlap on the GPU (different streams
 *     with no ordering between them) race on it; order them on one stream.
 *     Nothing in it has to start at zero: each call writes every scratch word
 *     before reading it.
 * ------------------------------------------------------------------------ */
#define NVFP4MOE_NOALLOC_SCRATCH_BYTES (512 * 1024)
int moe_align_permute_noalloc(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                              int32_t* expert_offsets, int32_t* perm, int32_t* inv, int act_kind, const void* act_in,
                              const uint8_t* act_in_scales, int64_t act_cols, void* act_out,
                              uint8_t* act_out_scales, int32_t* dev_status, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
