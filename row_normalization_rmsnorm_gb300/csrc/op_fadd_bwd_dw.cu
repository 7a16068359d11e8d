// Launch of the FusedAddRMSNorm backward row kernels, weight trainable (dW): one translation unit per
// flag combination, so the instantiations compile in parallel.
#include "kernels.cuh"

namespace gb300norm {

template int launch_typed<FADD_BWD, true, false>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t, int*);

}  // namespace gb300norm
