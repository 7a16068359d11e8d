// Dispatch of the LN_BWD row kernels: dW and dB are independent flags.  The
// four instantiations live in op_ln_bwd_{dw_db,dw,db,frozen}.cu.
#include "kernels.cuh"

namespace gb300norm {

extern template int launch_typed<LN_BWD, true, true>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t,
                                                     int*);
extern template int launch_typed<LN_BWD, true, false>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t,
                                                      int*);
extern template int launch_typed<LN_BWD, false, true>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t,
                                                      int*);
extern template int launch_typed<LN_BWD, false, false>(const RowParams&, int, int, const DevInfo&, bool, cudaStream_t,
                                                       int*);

int launch_op_ln_bwd(const RowParams& p, int dtype, int wdtype, bool dw, bool db, const DevInfo& di, bool aligned,
                     cudaStream_t st, int* grid) {
  if (dw && db) return launch_typed<LN_BWD, true, true>(p, dtype, wdtype, di, aligned, st, grid);
  if (dw) return launch_typed<LN_BWD, true, false>(p, dtype, wdtype, di, aligned, st, grid);
  if (db) return launch_typed<LN_BWD, false, true>(p, dtype, wdtype, di, aligned, st, grid);
  return launch_typed<LN_BWD, false, false>(p, dtype, wdtype, di, aligned, st, grid);
}

}  // namespace gb300norm
