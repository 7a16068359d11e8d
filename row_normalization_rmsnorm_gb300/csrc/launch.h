// launch.h -- internal interface between the C ABI (api.cu) and the
// per-operation translation units that instantiate the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/gb300norm.h"
#include "common.cuh"

namespace gb300norm {

// Internal: "this kernel family cannot take the shape, try the next one".
constexpr int NORM_ERR_UNSUPPORTED_INTERNAL = -1;

// Remember `e` as this thread's last CUDA error; returns NORM_ERR_CUDA.
int cuda_fail(cudaError_t e);

// Counts one successful kernel launch of this library (norm_debug_launches).
void count_launch();

// Launch status of the kernel just enqueued: NORM_OK or NORM_ERR_CUDA.
inline int launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NORM_OK : cuda_fail(e);
}

// Launch `kernel` on `st` with programmatic stream serialisation (see
// grid_dependency_wait in common.cuh), as thread-block clusters of
// `cluster` CTAs along x when cluster > 1.  NORM_OK or NORM_ERR_CUDA.
template <class... KArgs, class... Args>
int launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return cuda_fail(e);
  count_launch();
  return NORM_OK;
}

template <class... KArgs, class... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, 1, st, std::forward<Args>(args)...);
}

// What the launchers need to know about the current device.
struct DevInfo {
  int dev = 0;
  int sms = 0;               // streaming multiprocessors
  int smem_optin = 0;        // max dynamic shared memory per CTA (opt-in)
  int smem_per_sm = 0;       // shared memory per SM
  int smem_reserved = 0;     // shared memory the system reserves per CTA
  int64_t max_partial_rows = 0;  // dW/dB partial rows the workspace holds
  int force_path = 0;        // 0 = automatic, 2 = always the loop kernels
  // test hooks (0 = automatic): staged chunks per thread, CTAs per SM,
  // stages, the cap on row bytes in flight per SM (units of 16 KB), and
  // CTAs per thread-block cluster sharing a row
  int tune_npt = 0;
  int tune_max_ctas = 0;
  int tune_max_stages = 0;
  int tune_inflight_16k = 0;
  int tune_cluster = 0;
};

// Partial rows of the dW / dB workspace for M rows of N columns on a device
// with `sms` SMs: one per row-kernel CTA, and up to k CTAs per SM with
// k = 16384 / N kept within [2, 8].  Narrow rows get more resident CTAs (the
// row kernels of a trainable backward need them to keep enough warps in
// flight) while the partial rows stay near 64 KB x SMs in total, so the
// column reduction reads about the same bytes whatever N.
inline int64_t partial_rows_per_sm(int64_t N) {
  const int64_t k = N > 0 ? 16384 / N : 8;
  return k < 2 ? 2 : (k > 8 ? 8 : k);
}
inline int64_t partial_rows(int64_t M, int64_t N, int sms) {
  const int64_t cap = partial_rows_per_sm(N) * (int64_t)sms;
  return M < cap ? M : cap;
}

// Row kernels.  `aligned`: every streamed row (inputs and outputs) starts on
// a 16-byte boundary.  *grid receives the number of CTAs launched (= the
// number of partial rows written when dW / dB are computed).
int launch_op_rms_fwd(const RowParams&, int dtype, int wdtype, const DevInfo&, bool aligned, cudaStream_t, int* grid);
int launch_op_rms_bwd(const RowParams&, int dtype, int wdtype, bool dw, const DevInfo&, bool aligned, cudaStream_t,
                      int* grid);
int launch_op_ln_fwd(const RowParams&, int dtype, int wdtype, const DevInfo&, bool aligned, cudaStream_t, int* grid);
int launch_op_ln_bwd(const RowParams&, int dtype, int wdtype, bool dw, bool db, const DevInfo&, bool aligned,
                     cudaStream_t, int* grid);
int launch_op_fadd_fwd(const RowParams&, int dtype, int wdtype, const DevInfo&, bool aligned, cudaStream_t, int* grid);
int launch_op_fadd_bwd(const RowParams&, int dtype, int wdtype, bool dw, const DevInfo&, bool aligned, cudaStream_t,
                       int* grid);

// Stage 2 of the dW / dB reduction: out[j] = sum over g < G of ws[g*N + j],
// in increasing g, converted once to out_dtype.  ws_db / db may be null.
int launch_colreduce(const float* ws_dw, void* dw, const float* ws_db, void* db, int G, int N, int out_dtype,
                     cudaStream_t st);

// Sum over ranks: out[j] = sum over r < world of parts[r*N + j], in
// increasing r, converted once to out_dtype.
int launch_rank_sum(const float* parts, void* out, int world, int N, int out_dtype, cudaStream_t st);

}  // namespace gb300norm
