// kernels.h -- launchers of the NVFP4 MoE kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace nvfp4moe {

int num_sms();  // SM count of the current device (cached)

// Launch `kernel` with programmatic stream serialization: it may begin while
// the preceding kernel on the stream drains, and runs its global-memory-free
// prologue (barrier setup, TMEM allocation, descriptor prefetch) in that
// window; pdl_wait() inside the kernel orders everything else after the
// predecessor.  Returns the launch status.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Opt a kernel into `bytes` of dynamic shared memory on the current device
// (once per kernel and device).
cudaError_t ensure_dynamic_smem(const void* func, int bytes);

// Fault injection for the failure-detection tests: the environment variable
// NVFP4MOE_TEST_DROP_STAGE=n, read once per process, makes the FIRST grouped
// GEMM (W4A4, MXFP4, W4A16) or router GEMM launch of the process never arm
// its pipeline stage n; that launch's bounded waits run out, it reports
// NVFP4_E_DEVICE_TIMEOUT in dev_status, drains, frees TMEM and returns.  Every
// later launch gets -1 (no injection).
int fault_injection_drop_stage();

cudaError_t launch_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld, float* S,
                            int dynamic, uint32_t* amax_ws, uint8_t* codes, uint8_t* scales, cudaStream_t st);
cudaError_t launch_pack_scales(const uint8_t* in, int E, int N, int K, uint8_t* out, cudaStream_t st);
cudaError_t launch_swiglu_requant(const float* G, int R, int I, int mode, const float* S_h, uint8_t* h_codes,
                                  uint8_t* h_scales, void* h_bf16, cudaStream_t st);
// F16 carrier of BF16 rows: a_f16[r] = x[perm[r] or r] * 2^e_r, rs[r] = 2^-e_r
// (H % 8 == 0, 16-byte aligned rows); the SwiGLU of W4A16 (h rounded to bf16)
// carried the same way (I % 4 == 0).
cudaError_t launch_gather_f16(const void* x_bf16, int64_t H, const int32_t* perm, int R, void* a_f16, float* rs,
                              cudaStream_t st);
cudaError_t launch_swiglu_f16(const float* G, int R, int I, void* h_f16, float* rs, cudaStream_t st);
// out[0, n) = 0 before a GEMM's K parts add into it; the GEMM launched next
// (a programmatic dependent) may start its prologue during the fill.
cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t st);
cudaError_t launch_combine(const float* Y, const int32_t* inv, const float* w, int T, int k, int H,
                           int out_dtype, void* out, int32_t* dev_status, cudaStream_t st);
// Copy bytes16 (a multiple of 16) from src16 to dst16 and bytes4 (a multiple
// of 4) from src4 to dst4 with SM loads: the sources may be page-locked host
// memory (device views of it), read over the host link.
cudaError_t launch_stage_in(const void* src16, void* dst16, int64_t bytes16, const void* src4, void* dst4,
                            int64_t bytes4, cudaStream_t st);

// Routing: top-k + stable counting sort + optional gather.  ws must hold
// route_workspace_bytes(T, E) -- or, when ws_bytes says it holds less, at
// least route_workspace_min_bytes(T, E) (routing then runs in blocks of 32
// tokens, the layout with the smallest scratch).
size_t route_workspace_bytes(int T, int E);
size_t route_workspace_min_bytes(int T, int E);
// Routing alone; with x_bf16 != NULL it also leaves amax(|x|) ([T, H] bf16)
// as fp32 bits in the second word of ws (for nvfp4 quantisation).
cudaError_t launch_route_only(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                              int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* dev_status, void* ws,
                              cudaStream_t st, const void* x_bf16, int64_t H, size_t ws_bytes = (size_t)-1);
cudaError_t launch_gather(const int32_t* perm, int R, int act_kind, const void* act_in, const uint8_t* act_in_scales,
                          int64_t act_cols, void* act_out, uint8_t* act_out_scales, cudaStream_t st);
// Quantise x [T, H] bf16 with S = amax/2688 (amax bits from the routing
// pass; S written to *S) and write each token's NVFP4 row to its k permuted
// rows inv[t*k + j].
cudaError_t launch_quantize_scatter(const void* x_bf16, int T, int H, int k, const int32_t* inv,
                                    const uint32_t* amax_bits, float* S, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st);
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                         int32_t* offsets, int32_t* perm, int32_t* inv, int act_kind, const void* act_in,
                         const uint8_t* act_in_scales, int64_t act_cols, void* act_out, uint8_t* act_out_scales,
                         int32_t* dev_status, void* ws, cudaStream_t st, size_t ws_bytes = (size_t)-1);

// Grouped GEMMs.  Return cudaSuccess or the launch/setup error; host-side
// argument checks happen before these are called.  early = true only where
// the offsets, the weights and a_S were written by grids that completed
// before the kernel preceding the GEMM passed its griddepcontrol.wait (a
// layer's chain of this library's kernels): the GEMM then reads the routing
// and issues its first weight copies before its own wait.
cudaError_t launch_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_S,
                             const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                             const int32_t* offsets, int E, int N, int K, int R, float* out, int32_t* dev_status,
                             cudaStream_t st, bool early = false);
// The CTA-pair (.cta_group::2) grouped GEMM for many tokens per expert:
// eligible when N % 256 == 0 and the experts see >= 1024 rows on average.
bool gemm_w4a4_pair_eligible(int E, int N, int R);
cudaError_t launch_gemm_w4a4_pair(bool mx, const uint8_t* a_codes, const uint8_t* a_scales, const float* a_S,
                                  const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                                  const int32_t* offsets, int E, int N, int K, int R, float* out, int32_t* dev_status,
                                  cudaStream_t st);
cudaError_t launch_gemm_w4a16(const void* a_bf16, const uint8_t* w_codes, const uint8_t* w_scales_packed,
                              const float* w_S, const int32_t* offsets, int E, int N, int K, int R, float* out,
                              int32_t* dev_status, cudaStream_t st);
// W4A8: FP8 E4M3 token codes [R, K] with the per-tensor decode scale *a_S.
// W4A16 on F16-carried rows: a_f16 [R, K] holds x_r * 2^e_r, a_rs [R] = 2^-e_r.
cudaError_t launch_gemm_w4a16_f16(const void* a_f16, const float* a_rs, const uint8_t* w_codes,
                                  const uint8_t* w_scales_packed, const float* w_S, const int32_t* offsets, int E,
                                  int N, int K, int R, float* out, int32_t* dev_status, cudaStream_t st);
cudaError_t launch_gemm_w4a8(const uint8_t* a_fp8, const float* a_S, const uint8_t* w_codes,
                             const uint8_t* w_scales_packed, const float* w_S, const int32_t* offsets, int E, int N,
                             int K, int R, float* out, int32_t* dev_status, cudaStream_t st);
// FP8 (E4M3) activations with one per-tensor decode scale (the W4A8 mode):
// dynamic S = amax / 448 written to *S, or static *S read.
cudaError_t launch_fp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld, float* S,
                                int dynamic, uint32_t* amax_ws, uint8_t* codes, cudaStream_t st);
// x [T, H] bf16 -> FP8 codes of each token in its k permuted rows (amax bits
// from the routing pass; S written to *S).
// With f16_out != NULL the codes are written as their f16 values (the F16
// carrier of MOE_W4A16F) and rs[r] = S for every written row r.
cudaError_t launch_fp8_quantize_scatter(const void* x_bf16, int T, int H, int k, const int32_t* inv,
                                        const uint32_t* amax_bits, float* S, uint8_t* codes, cudaStream_t st,
                                        void* f16_out = nullptr, float* rs = nullptr);
// The W4A8 SwiGLU's FP8 codes written as their f16 values, h_rs[r] = *S_h.
cudaError_t launch_swiglu_fp8_f16(const float* G, int R, int I, const float* S_h, void* h_f16, float* h_rs,
                                  cudaStream_t st);

// Router logits [T, E] = x [T, H] . W [E, H]^T (bf16 in, fp32 out) on the
// tensor cores, K split over the SMs; workspace holds the fp32 partials
// (router_workspace_bytes; 0 when the problem is not split).
size_t router_workspace_bytes(int T, int H, int E);
cudaError_t launch_router_logits(const void* x_bf16, const void* w_bf16, int T, int H, int E, float* logits,
                                 void* workspace, int32_t* dev_status, cudaStream_t st);
// Router logits + top-k + permutation: for T <= 32 two launches (the router
// GEMM, then one fused kernel: fixed-order partial sums, top-k, stable
// permutation); otherwise the router GEMM, its reduce and the routing kernel.
// logits may be NULL (not returned).
size_t router_route_workspace_bytes(int T, int H, int E);
cudaError_t launch_router_route(const void* x_bf16, const void* w_bf16, int T, int H, int E, int k, float* logits,
                                int32_t* ids, float* w, int32_t* offsets, int32_t* perm, int32_t* inv,
                                int32_t* dev_status, void* workspace, cudaStream_t st);

// ---------------------------------------------------------------------------
// MXFP4 (32-element blocks, UE8M0 scales)
// ---------------------------------------------------------------------------

// Row pitch in bytes of an MXFP4 scale tensor with `cols` columns: cols/32
// rounded up to a multiple of 16 (TMA rows start on 16-byte boundaries), and
// at least 128: the grouped GEMM fetches 16 bytes of every row per two K
// stages, and with rows narrower than a 128-byte line those fetches slowed
// the whole kernel by a fifth (K = 2048) to a third (K = 1024) on GB300.
// The padding bytes are written as zero.
__host__ __device__ constexpr int64_t mx_scale_pitch(int64_t cols) {
  return ((cols / 32 + 15) / 16) * 16 < 128 ? 128 : ((cols / 32 + 15) / 16) * 16;
}

cudaError_t launch_mx_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                               uint8_t* scales, cudaStream_t st);
// Quantise x [T, H] bf16 to MXFP4 and write each token's row to its k
// permuted rows inv[t*k + j].
cudaError_t launch_mx_quantize_scatter(const void* x_bf16, int T, int H, int k, const int32_t* inv, uint8_t* codes,
                                       uint8_t* scales, cudaStream_t st);
// linear [E, N, K/32] -> per (expert, 128-row tile, K/64 step) 256-byte
// blocks: row r's two scales at (r % 32) * 8 + (r / 32) * 2.
cudaError_t launch_mx_pack_scales(const uint8_t* in, int E, int N, int K, uint8_t* out, cudaStream_t st);
cudaError_t launch_swiglu_requant_mx(const float* G, int R, int I, uint8_t* h_codes, uint8_t* h_scales,
                                     cudaStream_t st);
cudaError_t launch_gemm_mxw4a4(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* w_codes,
                               const uint8_t* w_scales_packed, const int32_t* offsets, int E, int N, int K, int R,
                               float* out, int32_t* dev_status, cudaStream_t st, bool early = false);

}  // namespace nvfp4moe
