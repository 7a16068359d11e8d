// Launch of the LayerNorm backward row kernels, dB only: one translation unit per
// flag combination, so the instantiations compile in parallel.
#include "kernels.cuh"

namespace gb300norm {

template int launch_typed<LN_BWD, false, true>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t, int*);

}  // namespace gb300norm
