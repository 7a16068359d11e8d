// Dispatch of the FADD_BWD row kernels, trainable (dW) and frozen; the
// instantiations live in op_fadd_bwd_dw.cu and op_fadd_bwd_frozen.cu.
#include "kernels.cuh"

namespace gb300norm {

extern template int launch_typed<FADD_BWD, true, false>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t,
                                                        int*);
extern template int launch_typed<FADD_BWD, false, false>(const RowParams&, int, int, const DevInfo&, bool,
                                                         cudaStream_t, int*);

int launch_op_fadd_bwd(const RowParams& p, int dtype, int wdtype, bool dw, const DevInfo& di, bool aligned,
                       cudaStream_t st, int* grid) {
  if (dw) return launch_typed<FADD_BWD, true, false>(p, dtype, wdtype, di, aligned, st, grid);
  return launch_typed<FADD_BWD, false, false>(p, dtype, wdtype, di, aligned, st, grid);
}

}  // namespace gb300norm
