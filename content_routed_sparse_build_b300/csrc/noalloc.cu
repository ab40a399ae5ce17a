// noalloc.cu -- decode attention whose scratch is a fixed block of device
// memory defined inside the library instead of a caller-supplied workspace.
//
// Who needs it: a caller that has no way to hand over device memory at the
// point of the call.  Two cases this serves: C code embedded in a host
// runtime that owns every device allocation (a plugin of an inference
// server, a custom operator of another framework), where a cudaMalloc of its
// own would bypass that runtime's memory accounting (and freeing it again
// waits for the whole device); and a latency-bound decode loop that must not
// reach the allocator on any step.  Such a caller cannot keep a workspace
// tensor of its own, so the library reserves one block per device, once,
// when its device code is loaded, and every call of this entry point reuses
// it.  Nothing here calls cudaMalloc, cudaFree or any library routine that
// allocates.
//
// The work itself is ssa_attend_decode unchanged: this file only finds the
// block, prepares it once per device and passes it as the workspace.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace {

// The scratch block.  Its first 256 bytes are laid out like any workspace
// header (the first word is the sticky device error record); the rest is the
// decode plan and partials.  Static device memory is reserved per device when
// the module is loaded and lives until the context is destroyed.
static __device__ __align__(256) unsigned char g_decode_scratch[SSA_NOALLOC_SCRATCH_BYTES];

struct DeviceScratch {
  CUcontext ctx = nullptr;  // context the address below belongs to
  void* addr = nullptr;     // device address of g_decode_scratch in that context
};

std::mutex g_setup_mutex;
DeviceScratch g_scratch[ssa::kMaxDevices];

// The driver's cuCtxGetCurrent, through the runtime's entry-point query (the
// library links no driver library of its own).
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }
  return fn;
}

// Looks up the block in the current device's current context (every call)
// and clears its header once per context (the error record must start at
// zero; the plan kernel resets everything else it reads): after
// cudaDeviceReset the device has a new context, whose block may sit
// elsewhere, and the clear runs again.  The clear is ordered on `st` before
// this call's kernels.
int setup_current_device(cudaStream_t st, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSA_ERR_CUDA;
  if (dev < 0 || dev >= ssa::kMaxDevices) return SSA_ERR_UNSUPPORTED;
  // the lookup also makes the device's (primary) context current if no call
  // has yet; it is a host-side table lookup and allocates nothing
  void* p = nullptr;
  if (cudaGetSymbolAddress((void**)&p, g_decode_scratch) != cudaSuccess || p == nullptr) return SSA_ERR_CUDA;
  auto get_ctx = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceScratch& s = g_scratch[dev];
  if (s.ctx != ctx || s.addr != p) {
    if (cudaMemsetAsync(p, 0, ssa::kWsHeader, st) != cudaSuccess) return SSA_ERR_CUDA;
    s.addr = p;
    s.ctx = ctx;
  }
  *out = s.addr;
  return SSA_OK;
}

}  // namespace

extern "C" {

int ssa_attend_decode_noalloc(const ssa_params* p, const void* Q, int64_t pos, const void* K,
                              const void* V, const int32_t* sel, void* O, float* lse, void** scratch,
                              void* stream) {
  // ssa_workspace_size returns 0 only for parameters that ssa_attend_decode
  // rejects (a valid decode problem needs at least the header): let it
  // return its own status for them, before it touches anything.
  const size_t need = ssa_workspace_size(p, 1, SSA_OP_DECODE);
  if (need == 0) return ssa_attend_decode(p, Q, pos, K, V, sel, O, lse, nullptr, 0, stream);
  if (need > (size_t)SSA_NOALLOC_SCRATCH_BYTES) return SSA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  const int rc = setup_current_device(st, &ws);
  if (rc != SSA_OK) return rc;
  if (scratch) *scratch = ws;
  return ssa_attend_decode(p, Q, pos, K, V, sel, O, lse, ws, (size_t)SSA_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
