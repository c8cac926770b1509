// pw_moe_forward_noalloc: the fused MoE layer forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand us a workspace: code that runs where every
// device allocation is forbidden or already fixed up front (an inference
// runtime that reserves its whole memory pool at start-up and rejects later
// cudaMalloc calls, or a plugin host that only passes tensors in and out).
// For them the forward's scratch (routing results, permutation, fp32 copies of
// the tokens, the intermediate h and y rows) lives in one file-scope device
// array of fixed size, reserved on every GPU that loads this library for as
// long as the process lives.  Nothing here calls cudaMalloc, cudaFree or any
// allocating library routine.

#include <cuda.h>
#include <nvtx3/nvToolsExt.h>
#include <cudaTypedefs.h>
#include <cstdio>
#include <mutex>

#include "pw_internal.h"

namespace pw {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB per device

// NVTX range around the call (a no-op when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Scratch for pw_moe_forward_noalloc.  Host code must not use this name as a
// pointer: it is a host-side stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;   // the context the address belongs to (0: none yet)
  void* ptr;
};
ScratchSlot g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Unique id of the calling thread's current context (0 when none is current or
// the driver cannot say).  A device reset ends the context and with it the
// array's address; the next context has another id.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device, looked up once per
// device and context (the lookup may load this library's kernels onto the device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  const unsigned long long id = current_context_id();
  ScratchSlot& sl = g_scratch[dev];
  if (id == 0 || sl.ctx_id != id || !sl.ptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    sl.ptr = p;
    sl.ctx_id = current_context_id();   // the lookup made the device's context current
  }
  *out = sl.ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace pw

extern "C" int pw_moe_forward_noalloc(pw_table* t, int layer, const void* x, const float* logits,
                                      int T, int top_k, int renorm, const void* residual, void* out,
                                      pw_stream_t compute) {
  pw::NvtxRange nvtx_range("pw_moe_forward_noalloc");
  int E = 0, H = 0, I = 0;   // the table's shapes size the scratch layout
  if (!t || pw::table_shape(t, &E, &H, &I) != PW_OK)
    return pw::set_error(PW_EINVAL, "pw_moe_forward_noalloc: null or invalid table");
  if (T < 0 || top_k < 1 || top_k > E)
    return pw::set_error(PW_EINVAL, "pw_moe_forward_noalloc: bad T or top_k");
  const size_t need = pw_workspace_bytes(T, E, top_k, H, I);
  if (need > pw::kStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "pw_moe_forward_noalloc: this batch needs %zu bytes of scratch, more than the %zu "
             "reserved; use pw_moe_forward with your own workspace",
             need, pw::kStaticScratchBytes);
    return pw::set_error(PW_ENOMEM, msg);
  }
  void* ws = nullptr;
  const cudaError_t e = pw::scratch_address(&ws);
  if (e != cudaSuccess) {
    char msg[200];
    snprintf(msg, sizeof msg, "pw_moe_forward_noalloc: scratch lookup failed: %s",
             cudaGetErrorString(e));
    return pw::set_error(PW_ECUDA, msg);
  }
  // The array keeps the previous call's contents; the forward resets what its
  // CTAs share before any of them reads it, so nothing needs clearing here.
  return pw_moe_forward(t, layer, x, logits, T, top_k, renorm, residual, out, nullptr, nullptr,
                        nullptr, nullptr, ws, pw::kStaticScratchBytes, compute);
}

extern "C" int pw_noalloc_status(pw_stream_t s, int* status) {
  if (!status) return pw::set_error(PW_EINVAL, "pw_noalloc_status: null status");
  void* ws = nullptr;
  const cudaError_t e = pw::scratch_address(&ws);
  if (e != cudaSuccess) {
    char msg[200];
    snprintf(msg, sizeof msg, "pw_noalloc_status: scratch lookup failed: %s", cudaGetErrorString(e));
    return pw::set_error(PW_ECUDA, msg);
  }
  return pw_workspace_status(ws, s, status);
}
