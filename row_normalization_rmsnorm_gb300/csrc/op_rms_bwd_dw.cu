// Launch of the RMSNorm backward row kernels, weight trainable (dW): one translation unit per
// flag combination, so the instantiations compile in parallel.
#include "kernels.cuh"

namespace gb300norm {

template int launch_typed<RMS_BWD, true, false>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t, int*);

}  // namespace gb300norm
