// ua_prefill.cu -- placeholder until the tcgen05 prefill kernel lands; the
// planner sends no tile here while the prefill path is disabled.
#include "ua_kernels.h"

namespace ua {

cudaError_t launch_prefill(int, const PrefillParams &, const CUtensorMap &, const CUtensorMap &,
                           const CUtensorMap &, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace ua
