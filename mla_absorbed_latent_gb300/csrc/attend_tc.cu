// tcgen05 split-KV decode (placeholder until the tensor-core kernel lands).
#include "mla_common.cuh"

namespace mla {

int attend_tc_workers(int num_sms) { return num_sms / 2; }

cudaError_t launch_attend_tc(const void*, int, int, int, const void*, const int32_t*, int, int, float, const int*,
                             int, float*, float*, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
