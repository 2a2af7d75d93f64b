// prefill.cu -- chunked-prefill attention (tcgen05 / TMEM / TMA).
#include <cuda_runtime.h>

#include "pd_internal.h"

namespace pd {
pd_status launch_prefill(const PrefillArgs&) { return PD_ERR_UNSUPPORTED; }
}  // namespace pd
