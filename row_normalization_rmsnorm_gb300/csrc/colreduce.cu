// colreduce.cu -- stage 2 of the dW / dB column reduction.
//
// The row kernels leave one FP32 partial row per CTA ([G][N]).  Each CTA of
// this kernel owns 32 adjacent columns: its 8 warps sum interleaved subsets of
// the partial rows (warp k takes rows k, k+8, ..., in eight independent
// chains), coalesced 128-byte row segments, and warp 0 adds the 8 subtotals
// in order; the cluster form below serves many partial rows.  The order of
// every addition is fixed by (G, N), so dW / dB are bit-identical from run to
// run.
// With G = 0 (no rows) the outputs are set to zero.
#include <cooperative_groups.h>

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

// The form for many partial rows (G >= kCrClusterRows, N % 4 == 0: every
// partial row then starts on a 16-byte boundary, as the workspace is 16-byte
// aligned and the dB partials start partial_rows(M, N, SMs) * N floats after
// the dW ones, see run_bwd in api.cu).  A
// thread-block cluster of kCrCluster CTAs owns 128 adjacent columns (lane l:
// columns 4l..4l+3, 16-byte loads) and splits the G partial rows among its
// kCrCluster x 8 warps: warp w of CTA r takes rows (8r + w) + 8 kCrCluster i,
// i = 0, 1, ..., in four independent chains (i mod 4) joined as
// (c0 + c1) + (c2 + c3).  Each CTA adds its warps' sums in warp order; CTA 0
// of the cluster adds the CTAs' sums in rank order, read through distributed
// shared memory, and writes the 128 outputs.  The order of every addition is
// fixed by (G, N).  With hundreds of partial rows the scalar form's eight
// chains per warp become a long series of dependent load rounds; the cluster
// spreads them over 8x the warps.  With fewer rows its fixed cost (cluster
// launch and barriers) does not pay.
constexpr int kCrCluster = 8;
constexpr int kCrClusterRows = 512;

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  const float2 lo = fadd2(make_float2(a.x, a.y), make_float2(b.x, b.y));
  const float2 hi = fadd2(make_float2(a.z, a.w), make_float2(b.z, b.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

template <class TO>
__global__ void __cluster_dims__(kCrCluster, 1, 1) __launch_bounds__(256)
    colreduce_cluster_kernel(const float* __restrict__ ws0, TO* __restrict__ out0, const float* __restrict__ ws1,
                             TO* __restrict__ out1, int G, int N) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tile = blockIdx.x / kCrCluster;
  const float* ws = blockIdx.y ? ws1 : ws0;
  TO* out = blockIdx.y ? out1 : out0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int col = tile * 128 + lane * 4;
  __shared__ float4 part[8][32];
  __shared__ float4 csum[32];
  // The partial rows come from the row kernel launched just before on this
  // stream; wait until that grid has completed and its writes are visible.
  grid_dependency_wait();
  grid_launch_dependents();
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 a[4] = {z, z, z, z};
  if (col < N) {
    constexpr int W = 8 * kCrCluster;   // warps of the cluster
    const float4* base = reinterpret_cast<const float4*>(ws + col);
    const int64_t rs = N / 4;           // row stride in float4
    int g = rank * 8 + warp;
    for (; g + 3 * W < G; g += 4 * W) {
      float4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) t[u] = base[(int64_t)(g + u * W) * rs];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = add4(a[u], t[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (g + u * W < G) a[u] = add4(a[u], base[(int64_t)(g + u * W) * rs]);
    }
  }
  part[warp][lane] = add4(add4(a[0], a[1]), add4(a[2], a[3]));
  __syncthreads();
  if (warp == 0) {
    float4 s = part[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) s = add4(s, part[w][lane]);
    csum[lane] = s;
  }
  cluster.sync();   // every CTA's csum written and visible to the cluster
  if (rank == 0 && warp == 0 && col < N) {
    float4 s = csum[lane];
#pragma unroll
    for (int r = 1; r < kCrCluster; ++r) s = add4(s, cluster.map_shared_rank(csum, r)[lane]);
    out[col] = from_f<TO>(s.x);
    out[col + 1] = from_f<TO>(s.y);
    out[col + 2] = from_f<TO>(s.z);
    out[col + 3] = from_f<TO>(s.w);
  }
  cluster.sync();   // the other CTAs keep their shared memory until CTA 0 has read it
}

template <class TO>
static int launch_cr(const float* a, void* da, const float* b, void* db, int G, int N, cudaStream_t st) {
  if (G >= kCrClusterRows && N % 4 == 0)
    return launch_pdl(colreduce_cluster_kernel<TO>, dim3((unsigned)((N + 127) / 128 * kCrCluster), db ? 2u : 1u),
                      dim3(256), 0, st, a, static_cast<TO*>(da), b, static_cast<TO*>(db), G, N);
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

// The sum over ranks of an M-sharded backward's dW / dB: each rank's FP32
// column sums (one row of `parts`, [world][N]) are added in rank order,
// out[j] = ((parts[0][j] + parts[1][j]) + parts[2][j]) + ..., and converted
// once.  Consecutive threads take consecutive columns, so every rank's row
// is read coalesced.
template <class TO>
__global__ void __launch_bounds__(256) rank_sum_kernel(const float* __restrict__ parts, TO* __restrict__ out,
                                                      int world, int N) {
  // the gathered rows come from work issued before this kernel on the stream
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < N; j += step) {
    float s = parts[j];
    for (int r = 1; r < world; ++r) s = fadd(s, parts[(int64_t)r * N + j]);
    out[j] = from_f<TO>(s);
  }
}

int launch_rank_sum(const float* parts, void* out, int world, int N, int out_dtype, cudaStream_t st) {
  const int64_t blocks = ((int64_t)N + 255) / 256;
  const dim3 grid((unsigned)(blocks < 4096 ? blocks : 4096));
  switch (out_dtype) {
    case NORM_F32: return launch_pdl(rank_sum_kernel<float>, grid, dim3(256), 0, st, parts, static_cast<float*>(out),
                                     world, N);
    case NORM_F16: return launch_pdl(rank_sum_kernel<__half>, grid, dim3(256), 0, st, parts,
                                     static_cast<__half*>(out), world, N);
    case NORM_BF16: return launch_pdl(rank_sum_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, parts,
                                      static_cast<__nv_bfloat16*>(out), world, N);
    default: return NORM_ERR_DTYPE;
  }
}

}  // namespace gb300norm
