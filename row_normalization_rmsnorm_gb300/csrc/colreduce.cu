// colreduce.cu -- stage 2 of the dW / dB column reduction.
//
// The row kernels leave one FP32 partial row per CTA ([G][N]).  Each CTA of
// this kernel owns 32 adjacent columns: its 8 warps sum interleaved subsets of
// the partial rows (warp k takes rows k, k+8, ..., in eight independent
// chains), coalesced 128-byte row segments, and warp 0 adds the 8 subtotals
// in order.  The order of every
// addition is fixed by (G, N), so dW / dB are bit-identical from run to run.
// With G = 0 (no rows) the outputs are set to zero.
#include "launch.h"

namespace gb300norm {

template <class TO>
__global__ void __launch_bounds__(256) colreduce_kernel(const float* __restrict__ ws0, TO* __restrict__ out0,
                                                        const float* __restrict__ ws1, TO* __restrict__ out1,
                                                        int G, int N) {
  const float* ws = blockIdx.y ? ws1 : ws0;
  TO* out = blockIdx.y ? out1 : out0;
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int col = blockIdx.x * 32 + lane;
  __shared__ float part[8][33];
  // The partial rows are written by the row kernel launched just before on
  // the same stream; this kernel may start while that grid drains, so it
  // waits here until the grid has completed and its writes are visible.
  grid_dependency_wait();
  grid_launch_dependents();
  // eight independent chains per thread (rows grp + 8u, u < 8, of each
  // block of 64 rows), joined in a fixed order
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (col < N) {
    int g = grp;
    for (; g + 56 < G; g += 64) {
      float t[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) t[u] = ws[(int64_t)(g + 8 * u) * N + col];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = fadd(a[u], t[u]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (g + 8 * u < G) a[u] = fadd(a[u], ws[(int64_t)(g + 8 * u) * N + col]);
    }
  }
  const float acc = fadd(fadd(fadd(a[0], a[1]), fadd(a[2], a[3])), fadd(fadd(a[4], a[5]), fadd(a[6], a[7])));
  part[grp][lane] = acc;
  __syncthreads();
  if (grp == 0 && col < N) {
    float s = part[0][lane];
#pragma unroll
    for (int k = 1; k < 8; ++k) s = fadd(s, part[k][lane]);
    out[col] = from_f<TO>(s);
  }
}

template <class TO>
static int launch_cr(const float* a, void* da, const float* b, void* db, int G, int N, cudaStream_t st) {
  return launch_pdl(colreduce_kernel<TO>, dim3((unsigned)((N + 31) / 32), db ? 2u : 1u), dim3(256), 0, st, a,
                    static_cast<TO*>(da), b, static_cast<TO*>(db), G, N);
}

int launch_colreduce(const float* ws_dw, void* dw, const float* ws_db, void* db, int G, int N, int out_dtype,
                     cudaStream_t st) {
  // The kernel takes one (partial, output) pair per blockIdx.y; when only dB
  // is wanted it goes in the first slot.
  if (!dw) { ws_dw = ws_db; dw = db; ws_db = nullptr; db = nullptr; }
  if (!dw) return NORM_OK;
  switch (out_dtype) {
    case NORM_F32: return launch_cr<float>(ws_dw, dw, ws_db, db, G, N, st);
    case NORM_F16: return launch_cr<__half>(ws_dw, dw, ws_db, db, G, N, st);
    case NORM_BF16: return launch_cr<__nv_bfloat16>(ws_dw, dw, ws_db, db, G, N, st);
    default: return NORM_ERR_DTYPE;
  }
}

}  // namespace gb300norm
