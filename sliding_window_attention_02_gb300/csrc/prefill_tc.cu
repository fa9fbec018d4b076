// tcgen05 prefill placeholder (replaced by the tensor-core kernel).
#include "rswa_internal.h"

namespace rswa {

bool prefill_tc_supported(const CacheView&) { return false; }

cudaError_t launch_prefill_tc(const CacheView&, const SeqTable&, const void*,
                              const void*, const void*, void*, int64_t,
                              cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace rswa
