// Instantiations of the LN_BWD row kernels: dW and dB are independent flags.
#include "kernels.cuh"

namespace gb300norm {

int launch_op_ln_bwd(const RowParams& p, int dtype, int wdtype, bool dw, bool db, const DevInfo& di, bool aligned,
                     cudaStream_t st, int* grid) {
  if (dw && db) return launch_typed<LN_BWD, true, true>(p, dtype, wdtype, di, aligned, st, grid);
  if (dw) return launch_typed<LN_BWD, true, false>(p, dtype, wdtype, di, aligned, st, grid);
  if (db) return launch_typed<LN_BWD, false, true>(p, dtype, wdtype, di, aligned, st, grid);
  return launch_typed<LN_BWD, false, false>(p, dtype, wdtype, di, aligned, st, grid);
}

}  // namespace gb300norm
