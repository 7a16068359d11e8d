// noalloc.cu -- norm_rms_bwd_noalloc: the trainable RMSNorm backward for
// callers that cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is unavailable or
// forbidden -- a CUDA-graph node body, an allocator-free inference runtime,
// a plugin host that owns every byte of device memory, or a caller inside a
// stream capture that must not call the allocator.  norm_rms_bwd needs a
// caller-provided workspace for the per-CTA dW partial sums; this entry point
// keeps those partial sums in a fixed array compiled into the library
// instead, so the caller passes only the inputs and the outputs.
//
// The array (kScratchBytes, 16 MiB) lives in device memory of every GPU on
// which this library's device code is loaded, for as long as the process
// runs.  All calls on a device share it: two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on it and give
// wrong dW.  No part of it needs clearing between calls: the row kernel
// writes every partial value it later reads.
#include <mutex>

#include "launch.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;

// The scratch itself.  In host code this name is only a host-side handle
// for the symbol, never a device address: the device address is obtained
// with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct ScratchAddr {
  std::mutex mu;
  void* ptr[64] = {};
};
ScratchAddr g_scratch;

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gb300norm::cuda_fail(e);
  if (dev < 0 || dev >= 64) return gb300norm::cuda_fail(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> g(g_scratch.mu);
  if (!g_scratch.ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return gb300norm::cuda_fail(e);
    g_scratch.ptr[dev] = p;
  }
  *out = g_scratch.ptr[dev];
  return NORM_OK;
}

}  // namespace

extern "C" {

size_t norm_noalloc_scratch_bytes(void) { return kScratchBytes; }

int norm_rms_bwd_noalloc(const void* dy, int64_t dy_stride, const void* x, int64_t x_stride, const void* w,
                         const float* rstd, void* dx, int64_t dx_stride, void* dw, int dw_dtype, int64_t M,
                         int64_t N, float offset, float eps, int dtype, int w_dtype, gb300norm_stream_t stream) {
  if (!dw) {
    // frozen weight: no partial sums, nothing to hold
    return norm_rms_bwd(dy, dy_stride, x, x_stride, w, rstd, dx, dx_stride, nullptr, dw_dtype, nullptr, 0, M, N,
                        offset, eps, dtype, w_dtype, stream);
  }
  size_t need = 0;
  int rc = norm_bwd_workspace_bytes(M, N, 1, 0, &need);
  if (rc != NORM_OK) return rc;
  if (need > kScratchBytes) return NORM_ERR_TOO_LARGE;
  void* scratch = nullptr;
  if (need > 0) {
    rc = scratch_address(&scratch);
    if (rc != NORM_OK) return rc;
  }
  return norm_rms_bwd(dy, dy_stride, x, x_stride, w, rstd, dx, dx_stride, dw, dw_dtype, scratch,
                      need > 0 ? kScratchBytes : 0, M, N, offset, eps, dtype, w_dtype, stream);
}

}  // extern "C"
