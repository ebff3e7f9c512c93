// phase1_mma.cu -- phase-1 partial attention on tcgen05 tensor cores for
// work items with at least 16 rows.  Until the tensor-core kernel is in
// place, no head size is reported as supported and the library runs those
// items on the CUDA-core kernel.
#include <cuda_runtime.h>

#include "deft_internal.h"

namespace deft {

bool mma_supported(int32_t) { return false; }

int launch_phase1_mma(const AttnArgs &, const DevPartition &, void *)
{
    return (int)cudaErrorNotSupported;
}

}  // namespace deft
