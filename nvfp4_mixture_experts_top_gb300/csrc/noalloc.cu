// noalloc.cu -- moe_align_permute_noalloc: the routing/permutation entry point
// for callers that cannot hand the library any scratch memory.
//
// Who needs it: code whose device memory is owned by someone else -- a
// serving engine or plugin host that reserves one arena up front and offers
// no workspace hook -- and latency-critical paths that must never call
// cudaMalloc, which can synchronise the whole device.  Such a caller can
// still pass its inputs and outputs, but not the scratch moe_align_permute
// wants.  This variant keeps that scratch in a fixed array in the library's
// own device memory instead.
//
// The array lives for as long as the library is loaded, once on every GPU that
// loads it, and is shared by every call on that GPU: two calls that overlap on
// the GPU (different streams, no ordering between them) race on it and give
// undefined results.  Every scratch word is written before it is read within
// one call (the per-chunk expert masks and activation maxima are rebuilt from
// the inputs each time), so the caller never has to clear anything between
// calls.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "../../include/nvfp4moe.h"
#include "kernels.h"

namespace nvfp4moe {
namespace {

// Fixed scratch: a 256-byte header, then per 32-token chunk and expert one
// 32-bit token mask, then per chunk one activation maximum.
__device__ __align__(256) static uint8_t g_route_scratch[NVFP4MOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_route_scratch, per device, for the CUDA context it was
// looked up in.  In host code the array's name is only a host-side stand-in;
// a kernel must be given the address the runtime reports.  A device reset
// destroys the context and the module with it, and the next context may load
// the array elsewhere, so the cached address is tagged with the context's
// unique id and looked up again when the current context differs.  A mutex
// guards the cache: two host threads may make their first call together.
constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;  // 0: nothing cached
  void* ptr;
};
ScratchSlot g_slot[kMaxDevices];
std::mutex g_slot_mu;

// Unique id of the calling thread's current context (0 if there is none or
// the driver entry points are unavailable).  Driver entry points are fetched
// through the runtime, so the library does not link libcuda.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  }
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_E_CUDA;
  std::lock_guard<std::mutex> lock(g_slot_mu);
  ScratchSlot& slot = g_slot[dev];
  const unsigned long long id = current_context_id();
  if (id != 0 && slot.ctx_id == id) {
    *out = slot.ptr;
    return NVFP4_OK;
  }
  // first call in this context (this also makes the device's primary
  // context current if the runtime had not yet done so)
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_route_scratch) != cudaSuccess || ptr == nullptr) return NVFP4_E_CUDA;
  slot.ptr = ptr;
  slot.ctx_id = current_context_id();  // 0 if unknown: then looked up on every call
  *out = ptr;
  return NVFP4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace nvfp4moe

extern "C" int moe_align_permute_noalloc(const float* logits, int T, int E, int k, int32_t* topk_ids,
                                         float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv,
                                         int act_kind, const void* act_in, const uint8_t* act_in_scales,
                                         int64_t act_cols, void* act_out, uint8_t* act_out_scales,
                                         int32_t* dev_status, nvfp4_stream_t stream) {
  using namespace nvfp4moe;
  // the same argument rules as moe_align_permute, minus the workspace
  if (T < 0 || E <= 0 || k <= 0) return NVFP4_E_INVAL;
  if (k > E || k > 32 || E > 1024) return NVFP4_E_SHAPE;
  if (expert_offsets == nullptr) return NVFP4_E_INVAL;
  if (act_kind != MOE_ACT_NONE && act_kind != MOE_ACT_NVFP4 && act_kind != MOE_ACT_BF16) return NVFP4_E_INVAL;
  // the fixed scratch must hold this problem, otherwise refuse before any work
  if (route_workspace_min_bytes(T, E) > (size_t)NVFP4MOE_NOALLOC_SCRATCH_BYTES) return NVFP4_E_WORKSPACE;
  if (T > 0) {
    if (logits == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr || inv == nullptr)
      return NVFP4_E_INVAL;
    if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(perm) || !aligned16(inv))
      return NVFP4_E_ALIGN;
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
  const int arch = nvfp4_device_check();
  if (arch != NVFP4_OK) return arch;
  void* scratch = nullptr;
  const int s = scratch_for_current_device(&scratch);
  if (s != NVFP4_OK) return s;
  const cudaError_t e = launch_route(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv, act_kind,
                                     act_in, act_in_scales, act_cols, act_out, act_out_scales, dev_status, scratch,
                                     reinterpret_cast<cudaStream_t>(stream), (size_t)NVFP4MOE_NOALLOC_SCRATCH_BYTES);
  return e == cudaSuccess ? NVFP4_OK : NVFP4_E_CUDA;
}
