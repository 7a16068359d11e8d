// Launch of the LayerNorm backward row kernels, weight and bias frozen: one translation unit per
// flag combination, so the instantiations compile in parallel.
#include "kernels.cuh"

namespace gb300norm {

template int launch_typed<LN_BWD, false, false>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t, int*);

}  // namespace gb300norm
