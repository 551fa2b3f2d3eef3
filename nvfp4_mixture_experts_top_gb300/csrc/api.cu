// api.cu -- the C ABI declared in include/nvfp4moe.h: host-side argument
// validation, the device check, and enqueueing of the kernels.  No entry
// point allocates device memory or synchronises.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "../../include/nvfp4moe.h"
#include "kernels.h"

namespace nvfp4moe {

namespace {
constexpr int kMaxDevices = 64;
int g_checked[kMaxDevices];  // 0 unknown, 1 ok, 2 wrong arch
int g_sms[kMaxDevices];

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
}  // namespace

// The environment is read once per process (a libc scan of the environment
// on every launch would sit on the enqueue path of latency-bound decode
// steps); the injection then applies to the first qualifying launch only, so
// that a test can check in the same process and context that the next launch
// is correct again.
int fault_injection_drop_stage() {
  static std::atomic<int> pending{[] {
    const char* v = getenv("NVFP4MOE_TEST_DROP_STAGE");
    return (v == nullptr || *v == 0) ? -1 : atoi(v);
  }()};
  if (pending.load(std::memory_order_relaxed) < 0) return -1;
  return pending.exchange(-1, std::memory_order_relaxed);
}

int num_sms() {
  const int d = current_device();
  if (d < 0) return 1;
  if (g_sms[d] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

// cudaFuncAttributeMaxDynamicSharedMemorySize for `func` on the current
// device, set once per (kernel, device): a process may drive several GPUs.
cudaError_t ensure_dynamic_smem(const void* func, int bytes) {
  constexpr int kFuncs = 16;
  static const void* funcs[kFuncs];
  static bool done[kFuncs][kMaxDevices];
  const int d = current_device();
  if (d < 0) return cudaErrorInvalidDevice;
  int i = 0;
  while (i < kFuncs && funcs[i] != nullptr && funcs[i] != func) ++i;
  if (i == kFuncs) return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (funcs[i] == nullptr) funcs[i] = func;
  if (done[i][d]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[i][d] = true;
  return e;
}

static int device_check_impl() {
  const int d = current_device();
  if (d < 0) return NVFP4_E_CUDA;
  if (g_checked[d] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess)
      return NVFP4_E_CUDA;
    g_checked[d] = (major == 10 && minor == 3) ? 1 : 2;
    num_sms();
  }
  return g_checked[d] == 1 ? NVFP4_OK : NVFP4_E_ARCH;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_E_CUDA; }

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace nvfp4moe

using namespace nvfp4moe;

#define CHECK_ARCH()                  \
  do {                                \
    const int _s = device_check_impl(); \
    if (_s != NVFP4_OK) return _s;    \
  } while (0)

extern "C" {

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_E_INVAL: return "NVFP4_E_INVAL: null pointer, negative size or bad enum";
    case NVFP4_E_SHAPE: return "NVFP4_E_SHAPE: a size violates a documented constraint";
    case NVFP4_E_ALIGN: return "NVFP4_E_ALIGN: a pointer is not 16-byte aligned";
    case NVFP4_E_WORKSPACE: return "NVFP4_E_WORKSPACE: workspace missing or too small";
    case NVFP4_E_ARCH: return "NVFP4_E_ARCH: device is not compute capability 10.3";
    case NVFP4_E_CUDA: return "NVFP4_E_CUDA: a CUDA call failed";
    case NVFP4_E_DEVICE_TIMEOUT: return "NVFP4_E_DEVICE_TIMEOUT: a bounded device wait ran out";
    case NVFP4_E_BAD_ROUTING: return "NVFP4_E_BAD_ROUTING: inconsistent expert offsets or ids";
    default: return "unknown nvfp4_status";
  }
}

int nvfp4_device_check(void) { return device_check_impl(); }

size_t nvfp4_quantize_workspace_bytes(int64_t rows, int64_t cols) {
  (void)rows;
  (void)cols;
  return 256;
}

int nvfp4_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x, float* S, int scale_mode,
                   uint8_t* codes, uint8_t* scales, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (rows < 0 || cols < 0 || S == nullptr) return NVFP4_E_INVAL;
  if (x_dtype != NVFP4_DT_BF16 && x_dtype != NVFP4_DT_F32) return NVFP4_E_INVAL;
  if (scale_mode != NVFP4_SCALE_STATIC && scale_mode != NVFP4_SCALE_DYNAMIC) return NVFP4_E_INVAL;
  if (cols % 16 != 0 || ld_x < cols) return NVFP4_E_SHAPE;
  if ((x_dtype == NVFP4_DT_BF16 && ld_x % 8 != 0) || (x_dtype == NVFP4_DT_F32 && ld_x % 4 != 0))
    return NVFP4_E_SHAPE;
  if (rows > 0 && cols > 0) {
    if (x == nullptr || codes == nullptr || scales == nullptr) return NVFP4_E_INVAL;
    if (!aligned16(x) || !aligned16(codes)) return NVFP4_E_ALIGN;
  }
  if (!aligned16(S)) return NVFP4_E_ALIGN;
  if (scale_mode == NVFP4_SCALE_DYNAMIC) {
    if (workspace == nullptr || workspace_bytes < nvfp4_quantize_workspace_bytes(rows, cols))
      return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  }
  CHECK_ARCH();
  return cuda_status(launch_quantize(x, x_dtype, rows, cols, ld_x, S, scale_mode == NVFP4_SCALE_DYNAMIC,
                                     static_cast<uint32_t*>(workspace), codes, scales,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4_pack_weight_scales(const uint8_t* scales_linear, int E, int N, int K, uint8_t* scales_packed,
                             nvfp4_stream_t stream) {
  if (E < 0 || N < 0 || K < 0) return NVFP4_E_INVAL;
  if (N % 128 != 0 || K % 256 != 0) return NVFP4_E_SHAPE;
  if ((int64_t)E * N * K == 0) return NVFP4_OK;
  if (scales_linear == nullptr || scales_packed == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(scales_linear) || !aligned16(scales_packed)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(launch_pack_scales(scales_linear, E, N, K, scales_packed, reinterpret_cast<cudaStream_t>(stream)));
}

int64_t mxfp4_scale_pitch(int64_t cols) { return cols < 0 ? 0 : mx_scale_pitch(cols); }

int mxfp4_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* codes,
                   uint8_t* scales, nvfp4_stream_t stream) {
  if (rows < 0 || cols < 0) return NVFP4_E_INVAL;
  if (x_dtype != NVFP4_DT_BF16 && x_dtype != NVFP4_DT_F32) return NVFP4_E_INVAL;
  if (cols % 32 != 0 || ld_x < cols) return NVFP4_E_SHAPE;
  if ((x_dtype == NVFP4_DT_BF16 && ld_x % 8 != 0) || (x_dtype == NVFP4_DT_F32 && ld_x % 4 != 0))
    return NVFP4_E_SHAPE;
  if (rows == 0 || cols == 0) return NVFP4_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(x) || !aligned16(codes)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(launch_mx_quantize(x, x_dtype, rows, cols, ld_x, codes, scales,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int mxfp4_pack_weight_scales(const uint8_t* scales_linear, int E, int N, int K, uint8_t* scales_packed,
                             nvfp4_stream_t stream) {
  if (E < 0 || N < 0 || K < 0) return NVFP4_E_INVAL;
  if (N % 128 != 0 || K % 256 != 0) return NVFP4_E_SHAPE;
  if ((int64_t)E * N * K == 0) return NVFP4_OK;
  if (scales_linear == nullptr || scales_packed == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(scales_linear) || !aligned16(scales_packed)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(
      launch_mx_pack_scales(scales_linear, E, N, K, scales_packed, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_router_logits_workspace_bytes(int T, int H, int E) {
  if (T < 0 || H < 0 || E < 0) return 0;
  // at least 256 bytes, so that a non-null, aligned workspace always exists
  const size_t b = router_workspace_bytes(T, H, E);
  return b > 256 ? b : 256;
}

int moe_router_logits(const void* x, const void* w_router, int T, int H, int E, float* logits, int32_t* dev_status,
                      void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0) return NVFP4_E_INVAL;
  if (H % 64 != 0) return NVFP4_E_SHAPE;
  if (T == 0) return NVFP4_OK;
  if (x == nullptr || w_router == nullptr || logits == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(logits)) return NVFP4_E_ALIGN;
  if (workspace == nullptr || workspace_bytes < moe_router_logits_workspace_bytes(T, H, E)) return NVFP4_E_WORKSPACE;
  if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(launch_router_logits(x, w_router, T, H, E, logits, workspace, dev_status,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_router_route_workspace_bytes(int T, int H, int E, int k) {
  (void)k;
  if (T < 0 || H < 0 || E < 0) return 0;
  return router_route_workspace_bytes(T, H, E);
}

int moe_router_route(const void* x, const void* w_router, int T, int H, int E, int k, float* logits,
                     int32_t* topk_ids, float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv,
                     int32_t* dev_status, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (H % 64 != 0 || k > E || k > 32 || E > 1024) return NVFP4_E_SHAPE;
  if (expert_offsets == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(expert_offsets)) return NVFP4_E_ALIGN;
  if (T > 0) {
    if (x == nullptr || w_router == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr ||
        inv == nullptr)
      return NVFP4_E_INVAL;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(perm) ||
        !aligned16(inv) || (logits != nullptr && !aligned16(logits)))
      return NVFP4_E_ALIGN;
    if (workspace == nullptr || workspace_bytes < moe_router_route_workspace_bytes(T, H, E, k))
      return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  }
  CHECK_ARCH();
  return cuda_status(launch_router_route(x, w_router, T, H, E, k, logits, topk_ids, topk_w, expert_offsets, perm,
                                         inv, dev_status, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_align_permute_workspace_bytes(int T, int E, int k) {
  (void)k;
  if (T < 0 || E < 0) return 0;
  return route_workspace_bytes(T, E);
}

int moe_align_permute(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                      int32_t* expert_offsets, int32_t* perm, int32_t* inv, int act_kind, const void* act_in,
                      const uint8_t* act_in_scales, int64_t act_cols, void* act_out, uint8_t* act_out_scales,
                      int32_t* dev_status, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (T < 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (k > E || k > 32 || E > 1024) return NVFP4_E_SHAPE;
  if (expert_offsets == nullptr) return NVFP4_E_INVAL;
  if (act_kind != MOE_ACT_NONE && act_kind != MOE_ACT_NVFP4 && act_kind != MOE_ACT_BF16) return NVFP4_E_INVAL;
  if (T > 0) {
    if (logits == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr || inv == nullptr)
      return NVFP4_E_INVAL;
    if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(perm) || !aligned16(inv))
      return NVFP4_E_ALIGN;
    if (workspace == nullptr || workspace_bytes < route_workspace_bytes(T, E)) return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
    if (act_kind != MOE_ACT_NONE) {
      if (act_cols <= 0) return NVFP4_E_SHAPE;
      if (act_kind == MOE_ACT_NVFP4 && act_cols % 256 != 0) return NVFP4_E_SHAPE;
      if (act_kind == MOE_ACT_BF16 && act_cols % 8 != 0) return NVFP4_E_SHAPE;
      if (act_in == nullptr || act_out == nullptr) return NVFP4_E_INVAL;
      if (act_kind == MOE_ACT_NVFP4 && (act_in_scales == nullptr || act_out_scales == nullptr)) return NVFP4_E_INVAL;
      if (!aligned16(act_in) || !aligned16(act_out)) return NVFP4_E_ALIGN;
      if (act_kind == MOE_ACT_NVFP4 && (!aligned16(act_in_scales) || !aligned16(act_out_scales)))
        return NVFP4_E_ALIGN;
    }
  }
  if (!aligned16(expert_offsets)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(launch_route(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv, act_kind, act_in,
                                  act_in_scales, act_cols, act_out, act_out_scales, dev_status, workspace,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

int moe_route_quantize_nvfp4(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                             float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, float* S_x,
                             uint8_t* a_codes, uint8_t* a_scales, int32_t* dev_status, void* workspace,
                             size_t workspace_bytes, nvfp4_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (k > E || k > 32 || E > 1024 || H % 256 != 0) return NVFP4_E_SHAPE;
  if (expert_offsets == nullptr || S_x == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(expert_offsets) || !aligned16(S_x)) return NVFP4_E_ALIGN;
  if (T > 0) {
    if (x == nullptr || logits == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr ||
        inv == nullptr || a_codes == nullptr || a_scales == nullptr)
      return NVFP4_E_INVAL;
    if (!aligned16(x) || !aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(perm) ||
        !aligned16(inv) || !aligned16(a_codes) || !aligned16(a_scales))
      return NVFP4_E_ALIGN;
    if (workspace == nullptr || workspace_bytes < route_workspace_bytes(T, E)) return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  }
  CHECK_ARCH();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (cudaMemsetAsync(S_x, 0, sizeof(float), st) != cudaSuccess) return NVFP4_E_CUDA;
    return cuda_status(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st));
  }
  // routing (+ the activation amax in the same pass), then the quantiser
  // writes each token's NVFP4 row straight to its k permuted rows
  if (launch_route_only(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv, dev_status, workspace, st, x,
                        H) != cudaSuccess)
    return NVFP4_E_CUDA;
  return cuda_status(launch_quantize_scatter(x, T, H, k, inv, static_cast<const uint32_t*>(workspace) + 1, S_x,
                                             a_codes, a_scales, st));
}

int moe_route_quantize_mxfp4(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                             float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, uint8_t* a_codes,
                             uint8_t* a_scales, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                             nvfp4_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (k > E || k > 32 || E > 1024 || H % 256 != 0) return NVFP4_E_SHAPE;
  if (expert_offsets == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(expert_offsets)) return NVFP4_E_ALIGN;
  if (T > 0) {
    if (x == nullptr || logits == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr ||
        inv == nullptr || a_codes == nullptr || a_scales == nullptr)
      return NVFP4_E_INVAL;
    if (!aligned16(x) || !aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(perm) ||
        !aligned16(inv) || !aligned16(a_codes) || !aligned16(a_scales))
      return NVFP4_E_ALIGN;
    if (workspace == nullptr || workspace_bytes < route_workspace_bytes(T, E)) return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  }
  CHECK_ARCH();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) return cuda_status(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st));
  if (launch_route_only(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv, dev_status, workspace, st,
                        nullptr, 0) != cudaSuccess)
    return NVFP4_E_CUDA;
  return cuda_status(launch_mx_quantize_scatter(x, T, H, k, inv, a_codes, a_scales, st));
}

int fp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x, float* S, int scale_mode,
                 uint8_t* codes, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  if (rows < 0 || cols < 0 || S == nullptr) return NVFP4_E_INVAL;
  if (x_dtype != NVFP4_DT_BF16 && x_dtype != NVFP4_DT_F32) return NVFP4_E_INVAL;
  if (scale_mode != NVFP4_SCALE_STATIC && scale_mode != NVFP4_SCALE_DYNAMIC) return NVFP4_E_INVAL;
  if (cols % 16 != 0 || ld_x < cols) return NVFP4_E_SHAPE;
  if ((x_dtype == NVFP4_DT_BF16 && ld_x % 8 != 0) || (x_dtype == NVFP4_DT_F32 && ld_x % 4 != 0))
    return NVFP4_E_SHAPE;
  if (rows > 0 && cols > 0) {
    if (x == nullptr || codes == nullptr) return NVFP4_E_INVAL;
    if (!aligned16(x) || !aligned16(codes)) return NVFP4_E_ALIGN;
  }
  if (!aligned16(S)) return NVFP4_E_ALIGN;
  if (scale_mode == NVFP4_SCALE_DYNAMIC) {
    if (workspace == nullptr || workspace_bytes < nvfp4_quantize_workspace_bytes(rows, cols))
      return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  }
  CHECK_ARCH();
  return cuda_status(launch_fp8_quantize(x, x_dtype, rows, cols, ld_x, S, scale_mode == NVFP4_SCALE_DYNAMIC,
                                         static_cast<uint32_t*>(workspace), codes,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int moe_route_quantize_fp8(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                           float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, float* S_x,
                           uint8_t* a_codes, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                           nvfp4_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (k > E || k > 32 || E > 1024 || H % 256 != 0) return NVFP4_E_SHAPE;
  if (expert_offsets == nullptr || S_x == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(expert_offsets) || !aligned16(S_x)) return NVFP4_E_ALIGN;
  if (T > 0) {
    if (x == nullptr || logits == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr ||
        inv == nullptr || a_codes == nullptr)
      return NVFP4_E_INVAL;
    if (!aligned16(x) || !aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(perm) ||
        !aligned16(inv) || !aligned16(a_codes))
      return NVFP4_E_ALIGN;
    if (workspace == nullptr || workspace_bytes < route_workspace_bytes(T, E)) return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  }
  CHECK_ARCH();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (cudaMemsetAsync(S_x, 0, sizeof(float), st) != cudaSuccess) return NVFP4_E_CUDA;
    return cuda_status(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st));
  }
  // routing (+ the activation amax in the same pass), then each token's FP8
  // row goes straight to its k permuted rows
  if (launch_route_only(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv, dev_status, workspace, st, x,
                        H) != cudaSuccess)
    return NVFP4_E_CUDA;
  return cuda_status(launch_fp8_quantize_scatter(x, T, H, k, inv, static_cast<const uint32_t*>(workspace) + 1, S_x,
                                                 a_codes, st));
}

// early: see launch_gemm_w4a4 (true only from moe_layer_forward's chain)
static int grouped_gemm(int mode, const void* a, const uint8_t* a_scales, const float* a_S, const uint8_t* w_codes,
                        const uint8_t* w_scales_packed, const float* w_S, const int32_t* expert_offsets, int E,
                        int N, int K, int R, float* out, int32_t* dev_status, nvfp4_stream_t stream, bool early) {
  if (mode != MOE_W4A4 && mode != MOE_W4A16 && mode != MOE_MXW4A4 && mode != MOE_W4A8 && mode != MOE_W4A16F)
    return NVFP4_E_INVAL;
  if (E <= 0 || N < 0 || K < 0 || R < 0) return NVFP4_E_INVAL;
  if (N % 128 != 0 || K % 256 != 0) return NVFP4_E_SHAPE;
  if (R == 0 || N == 0 || K == 0) return NVFP4_OK;
  if (a == nullptr || w_codes == nullptr || w_scales_packed == nullptr || expert_offsets == nullptr ||
      out == nullptr)
    return NVFP4_E_INVAL;
  if (mode != MOE_MXW4A4 && w_S == nullptr) return NVFP4_E_INVAL;
  if (mode == MOE_W4A4 && (a_scales == nullptr || a_S == nullptr)) return NVFP4_E_INVAL;
  if ((mode == MOE_W4A8 || mode == MOE_W4A16F) && a_S == nullptr) return NVFP4_E_INVAL;
  if (mode == MOE_MXW4A4 && a_scales == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(a) || !aligned16(w_codes) || !aligned16(w_scales_packed) || !aligned16(out))
    return NVFP4_E_ALIGN;
  if ((mode == MOE_W4A4 || mode == MOE_MXW4A4) && !aligned16(a_scales)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (mode == MOE_W4A8)
    return cuda_status(launch_gemm_w4a8(static_cast<const uint8_t*>(a), a_S, w_codes, w_scales_packed, w_S,
                                        expert_offsets, E, N, K, R, out, dev_status, st));
  if (mode == MOE_W4A16F)
    return cuda_status(launch_gemm_w4a16_f16(a, a_S, w_codes, w_scales_packed, w_S, expert_offsets, E, N, K, R, out,
                                             dev_status, st));
  // many tokens per expert (prefill, large-M GEMMs): CTA pairs on one MMA
  if ((mode == MOE_W4A4 || mode == MOE_MXW4A4) && gemm_w4a4_pair_eligible(E, N, R))
    return cuda_status(launch_gemm_w4a4_pair(mode == MOE_MXW4A4, static_cast<const uint8_t*>(a), a_scales, a_S,
                                             w_codes, w_scales_packed, w_S, expert_offsets, E, N, K, R, out,
                                             dev_status, st));
  if (mode == MOE_MXW4A4)
    return cuda_status(launch_gemm_mxw4a4(static_cast<const uint8_t*>(a), a_scales, w_codes, w_scales_packed,
                                          expert_offsets, E, N, K, R, out, dev_status, st, early));
  if (mode == MOE_W4A4)
    return cuda_status(launch_gemm_w4a4(static_cast<const uint8_t*>(a), a_scales, a_S, w_codes, w_scales_packed, w_S,
                                        expert_offsets, E, N, K, R, out, dev_status, st, early));
  return cuda_status(
      launch_gemm_w4a16(a, w_codes, w_scales_packed, w_S, expert_offsets, E, N, K, R, out, dev_status, st));
}

int moe_grouped_gemm_nvfp4(int mode, const void* a, const uint8_t* a_scales, const float* a_S,
                           const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                           const int32_t* expert_offsets, int E, int N, int K, int R, float* out,
                           int32_t* dev_status, nvfp4_stream_t stream) {
  return grouped_gemm(mode, a, a_scales, a_S, w_codes, w_scales_packed, w_S, expert_offsets, E, N, K, R, out,
                      dev_status, stream, false);
}

int moe_route_quantize_fp8_f16(const void* x, const float* logits, int T, int H, int E, int k, int32_t* topk_ids,
                               float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv, float* S_x,
                               void* a_f16, float* a_rs, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                               nvfp4_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (k > E || k > 32 || E > 1024 || H % 256 != 0) return NVFP4_E_SHAPE;
  if (expert_offsets == nullptr || S_x == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(expert_offsets) || !aligned16(S_x)) return NVFP4_E_ALIGN;
  if (T > 0) {
    if (x == nullptr || logits == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr ||
        inv == nullptr || a_f16 == nullptr || a_rs == nullptr)
      return NVFP4_E_INVAL;
    if (!aligned16(x) || !aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(perm) ||
        !aligned16(inv) || !aligned16(a_f16))
      return NVFP4_E_ALIGN;
    if (workspace == nullptr || workspace_bytes < route_workspace_bytes(T, E)) return NVFP4_E_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_E_ALIGN;
  }
  CHECK_ARCH();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (cudaMemsetAsync(S_x, 0, sizeof(float), st) != cudaSuccess) return NVFP4_E_CUDA;
    return cuda_status(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st));
  }
  if (launch_route_only(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv, dev_status, workspace, st, x,
                        H) != cudaSuccess)
    return NVFP4_E_CUDA;
  return cuda_status(launch_fp8_quantize_scatter(x, T, H, k, inv, static_cast<const uint32_t*>(workspace) + 1, S_x,
                                                 nullptr, st, a_f16, a_rs));
}

int moe_swiglu_fp8_f16(const float* G, int R, int I, const float* S_h, void* h_f16, float* h_rs,
                       nvfp4_stream_t stream) {
  if (R < 0 || I < 0) return NVFP4_E_INVAL;
  if (I % 16 != 0) return NVFP4_E_SHAPE;
  if ((int64_t)R * I == 0) return NVFP4_OK;
  if (G == nullptr || S_h == nullptr || h_f16 == nullptr || h_rs == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(G) || !aligned16(h_f16)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(launch_swiglu_fp8_f16(G, R, I, S_h, h_f16, h_rs, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_gather_f16(const void* x, int T, int H, const int32_t* perm, int R, void* a_f16, float* a_rs,
                   nvfp4_stream_t stream) {
  if (T < 0 || H < 0 || R < 0) return NVFP4_E_INVAL;
  if (H % 8 != 0) return NVFP4_E_SHAPE;
  if ((int64_t)R * H == 0) return NVFP4_OK;
  if (x == nullptr || a_f16 == nullptr || a_rs == nullptr) return NVFP4_E_INVAL;
  if (perm == nullptr && R > T) return NVFP4_E_INVAL;
  if (!aligned16(x) || !aligned16(a_f16)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(launch_gather_f16(x, H, perm, R, a_f16, a_rs, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_swiglu_f16(const float* G, int R, int I, void* h_f16, float* h_rs, nvfp4_stream_t stream) {
  if (R < 0 || I < 0) return NVFP4_E_INVAL;
  if (I % 16 != 0) return NVFP4_E_SHAPE;
  if ((int64_t)R * I == 0) return NVFP4_OK;
  if (G == nullptr || h_f16 == nullptr || h_rs == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(G) || !aligned16(h_f16)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(launch_swiglu_f16(G, R, I, h_f16, h_rs, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_swiglu_requant(const float* G, int R, int I, int mode, const float* S_h, uint8_t* h_codes,
                       uint8_t* h_scales, void* h_bf16, nvfp4_stream_t stream) {
  if (mode != MOE_W4A4 && mode != MOE_W4A16 && mode != MOE_MXW4A4 && mode != MOE_W4A8) return NVFP4_E_INVAL;
  if (R < 0 || I < 0) return NVFP4_E_INVAL;
  if (I % (mode == MOE_MXW4A4 ? 32 : 16) != 0) return NVFP4_E_SHAPE;
  if ((int64_t)R * I == 0) return NVFP4_OK;
  if (G == nullptr) return NVFP4_E_INVAL;
  if (mode == MOE_MXW4A4) {
    if (h_codes == nullptr || h_scales == nullptr) return NVFP4_E_INVAL;
    if (!aligned16(G) || !aligned16(h_codes)) return NVFP4_E_ALIGN;
    CHECK_ARCH();
    return cuda_status(launch_swiglu_requant_mx(G, R, I, h_codes, h_scales, reinterpret_cast<cudaStream_t>(stream)));
  }
  if (mode == MOE_W4A4 && (S_h == nullptr || h_codes == nullptr || h_scales == nullptr)) return NVFP4_E_INVAL;
  if (mode == MOE_W4A8 && (S_h == nullptr || h_codes == nullptr)) return NVFP4_E_INVAL;
  if (mode == MOE_W4A16 && h_bf16 == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(G)) return NVFP4_E_ALIGN;
  if ((mode == MOE_W4A4 || mode == MOE_W4A8) && !aligned16(h_codes)) return NVFP4_E_ALIGN;
  if (mode == MOE_W4A16 && !aligned16(h_bf16)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(
      launch_swiglu_requant(G, R, I, mode, S_h, h_codes, h_scales, h_bf16, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_combine(const float* Y, const int32_t* inv, const float* topk_w, int T, int k, int H, int out_dtype,
                void* out, int32_t* dev_status, nvfp4_stream_t stream) {
  if (T < 0 || k <= 0 || H < 0) return NVFP4_E_INVAL;
  if (out_dtype != NVFP4_DT_F32 && out_dtype != NVFP4_DT_BF16) return NVFP4_E_INVAL;
  if (H % 4 != 0 || k > 32) return NVFP4_E_SHAPE;
  if ((int64_t)T * H == 0) return NVFP4_OK;
  if (Y == nullptr || inv == nullptr || topk_w == nullptr || out == nullptr) return NVFP4_E_INVAL;
  if (!aligned16(Y) || !aligned16(out)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  return cuda_status(
      launch_combine(Y, inv, topk_w, T, k, H, out_dtype, out, dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

// Carve the layer workspace into its regions (each 256-byte aligned).
struct LayerWs {
  int32_t *ids, *offsets, *perm, *inv;
  float *w, *S_x, *G, *Y;
  uint32_t* amax;
  void* route;
  uint8_t *xq_codes, *xq_scales, *a_codes, *a_scales, *h_codes, *h_scales;
  void *a_bf16, *h_bf16;  // W4A16: the F16-carried rows (same size)
  float *a_rs, *h_rs;     // W4A16: their per-row multipliers
  size_t total;
};

static LayerWs carve(void* base, int mode, int T, int H, int I, int E, int k) {
  LayerWs w;
  memset(&w, 0, sizeof(w));
  const size_t R = (size_t)T * k;
  size_t off = 0;
  uint8_t* b = static_cast<uint8_t*>(base);
  auto take = [&](size_t bytes) -> uint8_t* {
    uint8_t* p = b ? b + off : nullptr;
    off += align256(bytes);
    return p;
  };
  w.ids = reinterpret_cast<int32_t*>(take(R * 4));
  w.w = reinterpret_cast<float*>(take(R * 4));
  w.offsets = reinterpret_cast<int32_t*>(take((size_t)(E + 1) * 4));
  w.perm = reinterpret_cast<int32_t*>(take(R * 4));
  w.inv = reinterpret_cast<int32_t*>(take(R * 4));
  w.route = take(route_workspace_bytes(T, E));
  w.G = reinterpret_cast<float*>(take(R * 2 * I * 4));
  w.Y = reinterpret_cast<float*>(take(R * H * 4));
  if (mode == MOE_MXW4A4) {
    w.a_codes = take(R * H / 2);
    w.a_scales = take(R * (size_t)mx_scale_pitch(H));
    w.h_codes = take(R * I / 2);
    w.h_scales = take(R * (size_t)mx_scale_pitch(I));
  } else if (mode == MOE_W4A8) {
    // the FP8 activations travel as their f16 values (MOE_W4A16F GEMMs)
    w.S_x = reinterpret_cast<float*>(take(16));
    w.a_bf16 = take(R * H * 2);
    w.h_bf16 = take(R * I * 2);
    w.a_rs = reinterpret_cast<float*>(take(R * 4));
    w.h_rs = reinterpret_cast<float*>(take(R * 4));
  } else if (mode == MOE_W4A4) {
    w.S_x = reinterpret_cast<float*>(take(16));
    w.a_codes = take(R * H / 2);
    w.a_scales = take(R * H / 16);
    w.h_codes = take(R * I / 2);
    w.h_scales = take(R * I / 16);
  } else {
    w.a_bf16 = take(R * H * 2);
    w.h_bf16 = take(R * I * 2);
    w.a_rs = reinterpret_cast<float*>(take(R * 4));
    w.h_rs = reinterpret_cast<float*>(take(R * 4));
  }
  w.total = off;
  return w;
}

size_t moe_layer_workspace_bytes(int mode, int T, int H, int I, int E, int k) {
  if (T < 0 || H < 0 || I < 0 || E < 0 || k < 0) return 0;
  return carve(nullptr, mode, T, H, I, E, k).total;
}

int moe_layer_forward(int mode, const void* x, const float* logits, int T, int H, int I, int E, int k,
                      const uint8_t* w13_codes, const uint8_t* w13_scales_packed, const float* w13_S,
                      const uint8_t* w2_codes, const uint8_t* w2_scales_packed, const float* w2_S, const float* S_h,
                      float* out, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                      nvfp4_stream_t stream) {
  if (mode != MOE_W4A4 && mode != MOE_W4A16 && mode != MOE_MXW4A4 && mode != MOE_W4A8) return NVFP4_E_INVAL;
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (H % 256 != 0 || I % 256 != 0 || k > E || k > 32 || E > 1024) return NVFP4_E_SHAPE;
  if (T == 0) return NVFP4_OK;
  if (x == nullptr || logits == nullptr || w13_codes == nullptr || w13_scales_packed == nullptr ||
      w2_codes == nullptr || w2_scales_packed == nullptr || out == nullptr)
    return NVFP4_E_INVAL;
  if (mode != MOE_MXW4A4 && (w13_S == nullptr || w2_S == nullptr)) return NVFP4_E_INVAL;
  if ((mode == MOE_W4A4 || mode == MOE_W4A8) && S_h == nullptr) return NVFP4_E_INVAL;
  if (workspace == nullptr || workspace_bytes < moe_layer_workspace_bytes(mode, T, H, I, E, k))
    return NVFP4_E_WORKSPACE;
  if (!aligned16(workspace) || !aligned16(x) || !aligned16(out)) return NVFP4_E_ALIGN;
  CHECK_ARCH();
  const LayerWs w = carve(workspace, mode, T, H, I, E, k);
  const int R = T * k;
  int s;
  if (mode == MOE_MXW4A4) {
    s = moe_route_quantize_mxfp4(x, logits, T, H, E, k, w.ids, w.w, w.offsets, w.perm, w.inv, w.a_codes, w.a_scales,
                                 dev_status, w.route, route_workspace_bytes(T, E), stream);
    if (s != NVFP4_OK) return s;
    s = grouped_gemm(MOE_MXW4A4, w.a_codes, w.a_scales, nullptr, w13_codes, w13_scales_packed, nullptr, w.offsets, E,
                     2 * I, H, R, w.G, dev_status, stream, true);
    if (s != NVFP4_OK) return s;
    s = moe_swiglu_requant(w.G, R, I, MOE_MXW4A4, nullptr, w.h_codes, w.h_scales, nullptr, stream);
    if (s != NVFP4_OK) return s;
    s = grouped_gemm(MOE_MXW4A4, w.h_codes, w.h_scales, nullptr, w2_codes, w2_scales_packed, nullptr, w.offsets, E, H,
                     I, R, w.Y, dev_status, stream, true);
    if (s != NVFP4_OK) return s;
  } else if (mode == MOE_W4A8) {
    // FP8 quantisation as moe_route_quantize_fp8 / moe_swiglu_requant, with
    // the codes carried as their f16 values into the F16-operand GEMM (the
    // same products as the MOE_W4A8 GEMM, whose codes it converts itself)
    s = moe_route_quantize_fp8_f16(x, logits, T, H, E, k, w.ids, w.w, w.offsets, w.perm, w.inv, w.S_x, w.a_bf16,
                                   w.a_rs, dev_status, w.route, route_workspace_bytes(T, E), stream);
    if (s != NVFP4_OK) return s;
    s = moe_grouped_gemm_nvfp4(MOE_W4A16F, w.a_bf16, nullptr, w.a_rs, w13_codes, w13_scales_packed, w13_S,
                               w.offsets, E, 2 * I, H, R, w.G, dev_status, stream);
    if (s != NVFP4_OK) return s;
    s = moe_swiglu_fp8_f16(w.G, R, I, S_h, w.h_bf16, w.h_rs, stream);
    if (s != NVFP4_OK) return s;
    s = moe_grouped_gemm_nvfp4(MOE_W4A16F, w.h_bf16, nullptr, w.h_rs, w2_codes, w2_scales_packed, w2_S, w.offsets,
                               E, H, I, R, w.Y, dev_status, stream);
    if (s != NVFP4_OK) return s;
  } else if (mode == MOE_W4A4) {
    s = moe_route_quantize_nvfp4(x, logits, T, H, E, k, w.ids, w.w, w.offsets, w.perm, w.inv, w.S_x, w.a_codes,
                                 w.a_scales, dev_status, w.route, route_workspace_bytes(T, E), stream);
    if (s != NVFP4_OK) return s;
    s = grouped_gemm(MOE_W4A4, w.a_codes, w.a_scales, w.S_x, w13_codes, w13_scales_packed, w13_S, w.offsets, E,
                     2 * I, H, R, w.G, dev_status, stream, true);
    if (s != NVFP4_OK) return s;
    s = moe_swiglu_requant(w.G, R, I, MOE_W4A4, S_h, w.h_codes, w.h_scales, nullptr, stream);
    if (s != NVFP4_OK) return s;
    s = grouped_gemm(MOE_W4A4, w.h_codes, w.h_scales, S_h, w2_codes, w2_scales_packed, w2_S, w.offsets, E, H, I, R,
                     w.Y, dev_status, stream, true);
    if (s != NVFP4_OK) return s;
  } else {
    // W4A16: the bf16 activations (x, and h rounded to bf16) travel as F16
    // rows with per-row powers of two, which the F16 form of the dequantising
    // GEMM takes (the same products; see moe_gather_f16)
    s = moe_align_permute(logits, T, E, k, w.ids, w.w, w.offsets, w.perm, w.inv, MOE_ACT_NONE, nullptr, nullptr, 0,
                          nullptr, nullptr, dev_status, w.route, route_workspace_bytes(T, E), stream);
    if (s != NVFP4_OK) return s;
    s = moe_gather_f16(x, T, H, w.perm, R, w.a_bf16, w.a_rs, stream);
    if (s != NVFP4_OK) return s;
    s = moe_grouped_gemm_nvfp4(MOE_W4A16F, w.a_bf16, nullptr, w.a_rs, w13_codes, w13_scales_packed, w13_S,
                               w.offsets, E, 2 * I, H, R, w.G, dev_status, stream);
    if (s != NVFP4_OK) return s;
    s = moe_swiglu_f16(w.G, R, I, w.h_bf16, w.h_rs, stream);
    if (s != NVFP4_OK) return s;
    s = moe_grouped_gemm_nvfp4(MOE_W4A16F, w.h_bf16, nullptr, w.h_rs, w2_codes, w2_scales_packed, w2_S, w.offsets,
                               E, H, I, R, w.Y, dev_status, stream);
    if (s != NVFP4_OK) return s;
  }
  return moe_combine(w.Y, w.inv, w.w, T, k, H, NVFP4_DT_F32, out, dev_status, stream);
}

// Device view of page-locked host memory; false for any other pointer.
static bool host_view(const void* p, void** dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return false;
  *dev = a.devicePointer;
  return true;
}

size_t moe_layer_host_workspace_bytes(int mode, int T, int H, int I, int E, int k) {
  if (T < 0 || H < 0 || I < 0 || E < 0 || k < 0) return 0;
  return moe_layer_workspace_bytes(mode, T, H, I, E, k) + align256((size_t)T * H * 2) + align256((size_t)T * E * 4);
}

int moe_layer_forward_host(int mode, const void* x_host, const float* logits_host, int T, int H, int I, int E, int k,
                           const uint8_t* w13_codes, const uint8_t* w13_scales_packed, const float* w13_S,
                           const uint8_t* w2_codes, const uint8_t* w2_scales_packed, const float* w2_S,
                           const float* S_h, float* out_host, int32_t* dev_status, void* workspace,
                           size_t workspace_bytes, nvfp4_stream_t stream) {
  if (mode != MOE_W4A4 && mode != MOE_W4A16 && mode != MOE_MXW4A4 && mode != MOE_W4A8) return NVFP4_E_INVAL;
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (H % 256 != 0 || I % 256 != 0 || k > E || k > 32 || E > 1024) return NVFP4_E_SHAPE;
  if (T == 0) return NVFP4_OK;
  if (x_host == nullptr || logits_host == nullptr || out_host == nullptr) return NVFP4_E_INVAL;
  if (workspace == nullptr || workspace_bytes < moe_layer_host_workspace_bytes(mode, T, H, I, E, k))
    return NVFP4_E_WORKSPACE;
  if (!aligned16(workspace) || !aligned16(x_host) || !aligned16(out_host) ||
      (reinterpret_cast<uintptr_t>(logits_host) & 3u) != 0)
    return NVFP4_E_ALIGN;
  CHECK_ARCH();
  void *xd, *ld, *od;
  if (!host_view(x_host, &xd) || !host_view(logits_host, &ld) || !host_view(out_host, &od)) return NVFP4_E_INVAL;
  // the inputs' device copies sit after the layer's own workspace
  const size_t layer_bytes = moe_layer_workspace_bytes(mode, T, H, I, E, k);
  uint8_t* x_dev = static_cast<uint8_t*>(workspace) + layer_bytes;
  float* lg_dev = reinterpret_cast<float*>(x_dev + align256((size_t)T * H * 2));
  if (launch_stage_in(xd, x_dev, (int64_t)T * H * 2, ld, lg_dev, (int64_t)T * E * 4,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NVFP4_E_CUDA;
  // the combine kernel writes the output straight into the host buffer
  return moe_layer_forward(mode, x_dev, lg_dev, T, H, I, E, k, w13_codes, w13_scales_packed, w13_S, w2_codes,
                           w2_scales_packed, w2_S, S_h, static_cast<float*>(od), dev_status, workspace, layer_bytes,
                           stream);
}

}  // extern "C"
