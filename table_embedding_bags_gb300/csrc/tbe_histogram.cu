// tbe_histogram.cu -- small-table histogram x table forward (placeholder).
#include "tbe_internal.cuh"

namespace tbe {
int launch_forward_histogram(const Plan&, const FwdArgs&, int32_t*, cudaStream_t) {
  return TBE_ERR_UNSUPPORTED;
}
}  // namespace tbe
