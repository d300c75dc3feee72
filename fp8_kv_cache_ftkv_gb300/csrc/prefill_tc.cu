// prefill_tc.cu -- prefill attention on the tcgen05 tensor cores (placeholder until the kernel lands).
#include "ftkv_internal.h"

namespace ftkv {
cudaError_t launch_prefill_tc(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace ftkv
