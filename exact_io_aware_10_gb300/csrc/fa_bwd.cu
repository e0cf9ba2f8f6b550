// Backward attention (placeholder until the recomputation kernels land).
#include "fa_internal.h"

namespace fa {
fa_status bwd_launch(const void*, const void*, const void*, const void*, const void*, const float*, void*, void*, void*,
                     int, int, int, int, int, float, const int32_t*, void*, cudaStream_t) {
  return FA_ERR_UNSUPPORTED;
}
}  // namespace fa
