// cbq_umma.cu -- verify-round kernel (TMA + tcgen05 block-scaled FP8 MMA).
// Placeholder until the tcgen05 kernel lands: reports "invalid argument" so
// that CBQ_PATH_MMA fails loudly instead of computing anything else.
#include <cuda_runtime.h>

#include "cbq_internal.h"

namespace cbq {

int launch_umma(const UmmaParams&, bool, cudaStream_t) { return CBQ_EINVAL; }
unsigned take_status_umma(cudaStream_t) { return 0u; }

}  // namespace cbq
