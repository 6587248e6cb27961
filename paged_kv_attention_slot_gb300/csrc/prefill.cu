// Causal prefill / prefix-cached extend on tcgen05 tensor cores (work in progress).
#include "pkv_internal.h"

namespace pkv {

int prefill_supported(const char** why) {
  if (why) *why = "the prefill kernel is not built yet";
  return 0;
}

cudaError_t launch_prefill(const RunParams&, const void*, const void*, const void*, int64_t, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pkv
