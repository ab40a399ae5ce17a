// prefill.cu -- prefill attention fast path (span-major tiles + merge).
#include "internal.h"

namespace ssa {

bool prefill_fast_supported(const Problem&) { return false; }
size_t prefill_ws_bytes(const Problem&, int64_t) { return 0; }
cudaError_t launch_attend_prefill(const Problem&, const void*, int64_t, int64_t, const void*,
                                  const void*, const int32_t*, void*, float*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ssa
