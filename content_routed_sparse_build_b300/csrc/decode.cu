// decode.cu -- decode attention fast path (split spans + merge).
#include "internal.h"

namespace ssa {

bool decode_fast_supported(const Problem&) { return false; }
size_t decode_ws_bytes(const Problem&) { return 0; }
cudaError_t launch_attend_decode(const Problem&, const void*, int64_t, const void*, const void*,
                                 const int32_t*, void*, float*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ssa
