// Instantiations of the FADD_BWD row kernels, trainable (dW) and frozen.
#include "kernels.cuh"

namespace gb300norm {

int launch_op_fadd_bwd(const RowParams& p, int dtype, int wdtype, bool dw, const DevInfo& di, bool aligned,
                   cudaStream_t st, int* grid) {
  if (dw) return launch_typed<FADD_BWD, true, false>(p, dtype, wdtype, di, aligned, st, grid);
  return launch_typed<FADD_BWD, false, false>(p, dtype, wdtype, di, aligned, st, grid);
}

}  // namespace gb300norm
