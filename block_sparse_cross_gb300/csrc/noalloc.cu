// Forward pass for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocating
// routine) at the point where they run attention: code executed from another
// framework's per-call hook, where that framework owns every device byte and
// forbids allocation inside the hook, and services that freeze device
// allocation after start-up so that memory use stays fixed. They cannot
// provide the two workspaces splitkv_fwd needs. splitkv_fwd_noalloc builds
// the plan and keeps the forward partials in one file-scope device array
// instead, reserved once per device when the library's module is loaded.
//
// The array is shared by every call on a device and keeps the last call's
// contents. Nothing in it needs to start at zero: the planner rewrites its
// header (including the status word) and every array it later reads, and
// the forward writes every partial slot the merge reads. Two calls whose
// work overlaps on the GPU (different streams, or different host threads
// without ordering) race on the array and corrupt each other's results.
#include <cuda_runtime.h>

#include <mutex>

#include "layout.h"

namespace {

// Bytes of the per-device scratch array (plan workspace + forward partials).
constexpr size_t kStaticScratchBytes = SPLITKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device, looked up once
// per device (the host-side symbol is only a stand-in and must never be
// handed to a kernel).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return SPLITKV_EDEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SPLITKV_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPLITKV_OK;
}

}  // namespace

extern "C" int splitkv_fwd_noalloc(const splitkv_problem* prob, const void* Q, const void* Kc,
                                   const void* Vc, const void* Kd, const void* Vd, void* O,
                                   float* LSE, splitkv_stream stream) {
  size_t plan_bytes = 0, work_bytes = 0;
  int st = splitkv_workspace_size(prob, &plan_bytes, &work_bytes);
  if (st != SPLITKV_OK) return st;
  const size_t plan_span = skv::align_up(plan_bytes, 256);
  // larger problems do not fit the fixed array: use splitkv_plan + splitkv_fwd
  if (plan_span + work_bytes > kStaticScratchBytes) return SPLITKV_EWORKSPACE;
  void* base = nullptr;
  if ((st = scratch_for_current_device(&base)) != SPLITKV_OK) return st;
  char* plan_ws = static_cast<char*>(base);
  char* work = plan_ws + plan_span;
  if ((st = splitkv_plan(prob, plan_ws, plan_bytes, stream)) != SPLITKV_OK) return st;
  return splitkv_fwd(prob, plan_ws, Q, Kc, Vc, Kd, Vd, O, LSE, work, work_bytes, stream);
}
