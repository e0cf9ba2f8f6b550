// Paged decode (placeholder until the split-KV kernels land).
#include "fa_internal.h"

namespace fa {
fa_status decode_launch(const void*, const void*, const void*, const int32_t*, const int32_t*, void*, float*, int, int,
                        int, int, int, int, int, int, float, void*, cudaStream_t) {
  return FA_ERR_UNSUPPORTED;
}
}  // namespace fa
