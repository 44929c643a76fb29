// Causal / chunked prefill on tcgen05 tensor cores (in progress).
#include "internal.h"

namespace sinkattn {

cudaError_t launch_prefill(const PrefillArgs &, const CUtensorMap &, const CUtensorMap &,
                           const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                           cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace sinkattn
