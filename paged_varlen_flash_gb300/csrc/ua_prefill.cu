// ua_prefill.cu -- tensor-core prefill path (not built yet for any head size).
#include "ua_prefill.h"

namespace ua {

bool prefill_supported(int) { return false; }

void plan_prefill(const FwdParams&, int, PrefillPlan* plan) { *plan = PrefillPlan(); }

cudaError_t launch_prefill(const PrefillPlan&, const CUtensorMap&, const CUtensorMap&,
                           const FwdParams&, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace ua
