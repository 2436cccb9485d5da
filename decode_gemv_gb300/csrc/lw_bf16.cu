// BF16 exponent-coded weights: kernels and launchers (placeholder until the
// BF16 path lands).
#include "lw_internal.h"
#include "lw_launch.h"

namespace lw {

lw_status launch_bf16_product(const lw_dev_bundle*, const uint16_t*, int, float*, float*, int32_t*,
                              cudaStream_t) {
  return fail(LW_ERR_UNSUPPORTED, "BF16 products are not built yet");
}

lw_status launch_bf16_decode(const lw_dev_bundle*, void*, int32_t*, cudaStream_t) {
  return fail(LW_ERR_UNSUPPORTED, "BF16 decode is not built yet");
}

}  // namespace lw
