// Instantiations of the FADD_FWD row kernels.
#include "kernels.cuh"

namespace gb300norm {

int launch_op_fadd_fwd(const RowParams& p, int dtype, int wdtype, const DevInfo& di, bool aligned, cudaStream_t st,
                   int* grid) {
  return launch_typed<FADD_FWD, false, false>(p, dtype, wdtype, di, aligned, st, grid);
}

}  // namespace gb300norm
