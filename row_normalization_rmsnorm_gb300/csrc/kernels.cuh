// kernels.cuh -- the row kernels of every operation, and their launch logic.
//
// Two kernel families share the per-element arithmetic:
//
//  * staged_kernel: persistent CTAs (a multiple of the SM count) stream rows
//    through a ring of S shared-memory stages.  One thread issues a bulk copy
//    per input row through the TMA engine (cp.async.bulk + mbarrier
//    transaction counts) S-1 rows ahead; all threads reduce the row from
//    shared memory, and write outputs with 16-byte streaming stores straight
//    from registers.  W' = float(w) + offset and the dW / dB accumulators
//    live in registers for the thread's fixed columns.  Needs every row start
//    16-byte aligned and N a multiple of 16 bytes of elements.
//
//  * loop_kernel: any N, stride and alignment.  A CTA walks a row with scalar
//    coalesced loads, re-reading it (from L2) for each pass, and accumulates
//    dW / dB in its own FP32 partial row in the workspace.
//
// Both write, for dW / dB, one FP32 partial row per CTA; colreduce_kernel
// then sums the partial rows in a fixed order (deterministic), replacing the
// global sum over per-program partial buffers described on "perf(norm): skip
// dW/dB calculation when parameters are frozen", Motivation.  The DW / DB
// template flags remove every weight-gradient instruction, register and
// store when the parameter is frozen (same page, Key Changes).
#pragma once

#include <mutex>
#include <map>
#include <tuple>

#include "common.cuh"
#include "launch.h"

namespace gb300norm {

template <int OP> struct OpInfo;
template <> struct OpInfo<RMS_FWD>  { static constexpr int NIN = 1; static constexpr bool BWD = false; };
template <> struct OpInfo<RMS_BWD>  { static constexpr int NIN = 2; static constexpr bool BWD = true; };
template <> struct OpInfo<LN_FWD>   { static constexpr int NIN = 1; static constexpr bool BWD = false; };
template <> struct OpInfo<LN_BWD>   { static constexpr int NIN = 2; static constexpr bool BWD = true; };
template <> struct OpInfo<FADD_FWD> { static constexpr int NIN = 2; static constexpr bool BWD = false; };
template <> struct OpInfo<FADD_BWD> { static constexpr int NIN = 3; static constexpr bool BWD = true; };

__device__ __forceinline__ float div_n(float s, int N) { return __fdiv_rn(s, (float)N); }

// ===========================================================================
// Staged (TMA bulk copy) kernel
// ===========================================================================
constexpr int kStagedHeader = 1024;   // bytes: S mbarriers (<= 32) + reduction banks
constexpr int kMaxStages = 16;

template <int OP, class T, class TW, int NPT, bool DW, bool DB>
__global__ void __launch_bounds__(512) staged_kernel(const RowParams p, const int S) {
  constexpr int VEC = 16 / (int)sizeof(T);
  constexpr bool LN = (OP == LN_FWD || OP == LN_BWD);
  constexpr bool BWD = OpInfo<OP>::BWD;
  constexpr int NB = (OP == LN_FWD) ? NPT : 1;   // bias registers
  constexpr int NDW = DW ? NPT : 1;
  constexpr int NDB = DB ? NPT : 1;
  constexpr int NR = (OP == LN_BWD) ? 2 : 1;     // values reduced per backward row
  const int N = p.N;
  const int nchunks = N / VEC;
  const int tid = threadIdx.x, nt = blockDim.x;
  const uint32_t row_bytes = (uint32_t)N * (uint32_t)sizeof(T);
  const int nin = (OP == FADD_BWD && p.in2 == nullptr) ? 2 : OpInfo<OP>::NIN;
  const uint32_t stage_bytes = (uint32_t)nin * row_bytes;

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + 256);
  unsigned char* stages = smem + kStagedHeader;
  // abort_flag[k & 1] is raised while row k is awaited and read after row
  // k's barrier, so a thread already waiting for row k+1 cannot change what
  // the others read for row k.
  __shared__ int abort_flag[2];

  // Per-thread constant columns: W' = float(w) + offset (and the LayerNorm
  // bias) in FP32, formed once per CTA.
  float wv[NPT][VEC];
  float bv[NB][VEC];
  const bool has_b = (OP == LN_FWD) && p.b != nullptr;
  const TW* wp = static_cast<const TW*>(p.w);
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    const int c = tid + j * nt;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      wv[j][v] = (c < nchunks) ? fadd(to_f(wp[c * VEC + v]), p.offset) : 0.f;
      if constexpr (OP == LN_FWD)
        bv[j][v] = (has_b && c < nchunks) ? to_f(static_cast<const TW*>(p.b)[c * VEC + v]) : 0.f;
    }
  }
  float dwa[NDW][VEC];
  float dba[NDB][VEC];
#pragma unroll
  for (int j = 0; j < NDW; ++j)
#pragma unroll
    for (int v = 0; v < VEC; ++v) dwa[j][v] = 0.f;
#pragma unroll
  for (int j = 0; j < NDB; ++j)
#pragma unroll
    for (int v = 0; v < VEC; ++v) dba[j][v] = 0.f;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    abort_flag[0] = 0;
    abort_flag[1] = 0;
  }
  __syncthreads();

  const int64_t G = gridDim.x;
  const int64_t row0 = blockIdx.x;
  const int64_t nrows = (p.M - row0 + G - 1) / G;   // >= 1: the grid never exceeds M
  const uint64_t pol = l2_policy_evict_first();
  const char* g0 = static_cast<const char*>(p.in0);
  const char* g1 = static_cast<const char*>(p.in1);
  const char* g2 = static_cast<const char*>(p.in2);
  int64_t issued = 0;   // rows of this CTA whose copies have been issued (thread 0)

  auto issue = [&](int64_t k) {
    const int s = (int)(k % S);
    const int64_t row = row0 + k * G;
    unsigned char* dst = stages + (size_t)s * stage_bytes;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&bars[s], stage_bytes);
    bulk_g2s(dst, g0 + row * p.s_in0 * (int64_t)sizeof(T), row_bytes, &bars[s], pol);
    if (nin > 1) bulk_g2s(dst + row_bytes, g1 + row * p.s_in1 * (int64_t)sizeof(T), row_bytes, &bars[s], pol);
    if (nin > 2) bulk_g2s(dst + 2 * row_bytes, g2 + row * p.s_in2 * (int64_t)sizeof(T), row_bytes, &bars[s], pol);
  };
  if (tid == 0) {
    for (; issued < nrows && issued < S - 1; ++issued) issue(issued);
  }

  int bank = 0;
  int64_t k = 0;
  bool aborted = false;
  for (; k < nrows; ++k) {
    const int64_t row = row0 + k * G;
    const int s = (int)(k % S);
    const int fl = (int)(k & 1);
    if (!mbar_wait_bounded(&bars[s], (uint32_t)((k / S) & 1))) {
      atomicOr(p.status, STATUS_WAIT_TIMEOUT);
      abort_flag[fl] = 1;
    }
    const T* r0 = reinterpret_cast<const T*>(stages + (size_t)s * stage_bytes);
    const T* r1 = r0 + N;
    const T* r2 = r1 + N;

    // After the first barrier of row k every thread has finished row k-1, so
    // its stage can take the copy of row k+S-1.
    bool refilled = false;
    auto after_first_barrier = [&]() {
      if (refilled) return;
      refilled = true;
      if (tid == 0 && !abort_flag[fl] && issued < nrows) { issue(issued); ++issued; }
    };

    // ---- row statistics -------------------------------------------------
    float mean = 0.f, rstd = 0.f;
    const bool need_stats = !BWD || p.rstd_in == nullptr;
    if (!need_stats) {
      rstd = p.rstd_in[row];
      if constexpr (LN) mean = p.mean_in[row];
    } else if constexpr (LN) {
      float a[1] = {0.f};
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (c < nchunks) {
          Vec16<T> xv; xv.u = reinterpret_cast<const uint4*>(r0)[c];
#pragma unroll
          for (int v = 0; v < VEC; ++v) a[0] = fadd(a[0], to_f(xv.e[v]));
        }
      }
      block_sum<1>(a, red, bank);
      after_first_barrier();
      mean = div_n(a[0], N);
      float q[1] = {0.f};
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (c < nchunks) {
          Vec16<T> xv; xv.u = reinterpret_cast<const uint4*>(r0)[c];
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const float d = fsub(to_f(xv.e[v]), mean);
            q[0] = ffma(d, d, q[0]);
          }
        }
      }
      block_sum<1>(q, red, bank);
      rstd = inv_rms(div_n(q[0], N), p.eps);
    } else {
      float a[1] = {0.f};
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (c < nchunks) {
          Vec16<T> xv; xv.u = reinterpret_cast<const uint4*>(r0)[c];
          if constexpr (OP == FADD_FWD) {
            Vec16<T> rv; rv.u = reinterpret_cast<const uint4*>(r1)[c];
            Vec16<T> hv;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              const float h = fadd(to_f(xv.e[v]), to_f(rv.e[v]));
              a[0] = ffma(h, h, a[0]);
              hv.e[v] = from_f<T>(h);      // the residual stream passed on, rounded once
            }
            st_global_cs16(static_cast<T*>(p.out1) + row * p.s_out1 + (int64_t)c * VEC, hv.u);
          } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              const float h = to_f(xv.e[v]);
              a[0] = ffma(h, h, a[0]);
            }
          }
        }
      }
      block_sum<1>(a, red, bank);
      after_first_barrier();
      rstd = inv_rms(div_n(a[0], N), p.eps);
    }

    if constexpr (!BWD) {
      // ---- forward outputs ----------------------------------------------
      if (abort_flag[fl]) { aborted = true; break; }
      if (tid == 0) {
        if (p.rstd_out) p.rstd_out[row] = rstd;
        if (LN && p.mean_out) p.mean_out[row] = mean;
      }
      T* yrow = static_cast<T*>(p.out0) + row * p.s_out0;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (c < nchunks) {
          Vec16<T> xv; xv.u = reinterpret_cast<const uint4*>(r0)[c];
          Vec16<T> rv;
          if constexpr (OP == FADD_FWD) rv.u = reinterpret_cast<const uint4*>(r1)[c];
          Vec16<T> yv;
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            float xf = to_f(xv.e[v]);
            if constexpr (OP == FADD_FWD) xf = fadd(xf, to_f(rv.e[v]));
            float yf;
            if constexpr (OP == LN_FWD) yf = fadd(fmul(fmul(fsub(xf, mean), rstd), wv[j][v]), bv[j][v]);
            else                        yf = fmul(fmul(xf, rstd), wv[j][v]);
            yv.e[v] = from_f<T>(yf);
          }
          st_global_cs16(yrow + (int64_t)c * VEC, yv.u);
        }
      }
    } else {
      // ---- backward: row sums of g (LayerNorm) and g*xhat -----------------
      float a[NR];
#pragma unroll
      for (int i = 0; i < NR; ++i) a[i] = 0.f;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (c < nchunks) {
          Vec16<T> xv; xv.u = reinterpret_cast<const uint4*>(r0)[c];
          Vec16<T> dv; dv.u = reinterpret_cast<const uint4*>(r1)[c];
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const float xf = to_f(xv.e[v]);
            const float g = fmul(to_f(dv.e[v]), wv[j][v]);
            if constexpr (LN) {
              const float xh = fmul(fsub(xf, mean), rstd);
              a[0] = fadd(a[0], g);
              a[NR - 1] = ffma(g, xh, a[NR - 1]);
            } else {
              const float xh = fmul(xf, rstd);
              a[0] = ffma(g, xh, a[0]);
            }
          }
        }
      }
      block_sum<NR>(a, red, bank);
      after_first_barrier();
      if (abort_flag[fl]) { aborted = true; break; }
      const float mg = LN ? div_n(a[0], N) : 0.f;
      const float mgx = div_n(a[NR - 1], N);
      T* dxrow = static_cast<T*>(p.out0) + row * p.s_out0;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (c < nchunks) {
          Vec16<T> xv; xv.u = reinterpret_cast<const uint4*>(r0)[c];
          Vec16<T> dv; dv.u = reinterpret_cast<const uint4*>(r1)[c];
          Vec16<T> hv;
          const bool has_dh = (OP == FADD_BWD) && nin > 2;
          if (has_dh) hv.u = reinterpret_cast<const uint4*>(r2)[c];
          Vec16<T> ov;
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const float xf = to_f(xv.e[v]);
            const float dyf = to_f(dv.e[v]);
            const float g = fmul(dyf, wv[j][v]);
            float xh, dx;
            if constexpr (LN) {
              xh = fmul(fsub(xf, mean), rstd);
              dx = fmul(rstd, fsub(fsub(g, mg), fmul(xh, mgx)));
            } else {
              xh = fmul(xf, rstd);
              dx = fmul(rstd, fsub(g, fmul(xh, mgx)));
            }
            if (has_dh) dx = fadd(dx, to_f(hv.e[v]));
            ov.e[v] = from_f<T>(dx);
            if constexpr (DW) dwa[j][v] = ffma(dyf, xh, dwa[j][v]);
            if constexpr (DB) dba[j][v] = fadd(dba[j][v], dyf);
          }
          st_global_cs16(dxrow + (int64_t)c * VEC, ov.u);
        }
      }
    }
  }

  if (aborted) {
    // Bounded drain of the copies still in flight into this CTA's shared
    // memory, then leave without writing partial sums.
    if (tid == 0) {
      for (int64_t kk = k; kk < issued; ++kk) (void)mbar_wait_bounded(&bars[kk % S], (uint32_t)((kk / S) & 1));
    }
    return;
  }

  if constexpr (DW || DB) {
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int c = tid + j * nt;
      if (c < nchunks) {
        const int64_t off = (int64_t)blockIdx.x * N + (int64_t)c * VEC;
#pragma unroll
        for (int v = 0; v < VEC; v += 4) {
          if constexpr (DW)
            *reinterpret_cast<float4*>(p.ws_dw + off + v) = make_float4(dwa[j][v], dwa[j][v + 1], dwa[j][v + 2], dwa[j][v + 3]);
          if constexpr (DB)
            *reinterpret_cast<float4*>(p.ws_db + off + v) = make_float4(dba[j][v], dba[j][v + 1], dba[j][v + 2], dba[j][v + 3]);
        }
      }
    }
  }
}

// ===========================================================================
// Loop kernel (any alignment, any N)
// ===========================================================================
template <int OP, class T, class TW, bool DW, bool DB>
__global__ void __launch_bounds__(512) loop_kernel(const RowParams p) {
  constexpr bool LN = (OP == LN_FWD || OP == LN_BWD);
  constexpr bool BWD = OpInfo<OP>::BWD;
  constexpr int NR = (OP == LN_BWD) ? 2 : 1;
  const int N = p.N;
  const int tid = threadIdx.x, nt = blockDim.x;
  __shared__ float red[2 * 32 * 2];
  int bank = 0;
  const TW* wp = static_cast<const TW*>(p.w);
  const TW* bp = static_cast<const TW*>(p.b);
  float* wsw = nullptr;
  float* wsb = nullptr;
  if constexpr (DW) wsw = p.ws_dw + (int64_t)blockIdx.x * N;
  if constexpr (DB) wsb = p.ws_db + (int64_t)blockIdx.x * N;
  bool first = true;

  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const T* x = static_cast<const T*>(p.in0) + row * p.s_in0;
    const T* i1 = nullptr;
    const T* i2 = nullptr;
    if constexpr (OpInfo<OP>::NIN > 1) i1 = static_cast<const T*>(p.in1) + row * p.s_in1;
    if constexpr (OP == FADD_BWD) {
      if (p.in2) i2 = static_cast<const T*>(p.in2) + row * p.s_in2;
    }
    T* o0 = static_cast<T*>(p.out0) + row * p.s_out0;

    float mean = 0.f, rstd = 0.f;
    const bool need_stats = !BWD || p.rstd_in == nullptr;
    if (!need_stats) {
      rstd = p.rstd_in[row];
      if constexpr (LN) mean = p.mean_in[row];
    } else if constexpr (LN) {
      float a[1] = {0.f};
      for (int j = tid; j < N; j += nt) a[0] = fadd(a[0], to_f(x[j]));
      block_sum<1>(a, red, bank);
      mean = div_n(a[0], N);
      float q[1] = {0.f};
      for (int j = tid; j < N; j += nt) {
        const float d = fsub(to_f(x[j]), mean);
        q[0] = ffma(d, d, q[0]);
      }
      block_sum<1>(q, red, bank);
      rstd = inv_rms(div_n(q[0], N), p.eps);
    } else {
      float a[1] = {0.f};
      for (int j = tid; j < N; j += nt) {
        float h = to_f(x[j]);
        if constexpr (OP == FADD_FWD) h = fadd(h, to_f(i1[j]));
        a[0] = ffma(h, h, a[0]);
      }
      block_sum<1>(a, red, bank);
      rstd = inv_rms(div_n(a[0], N), p.eps);
    }

    if constexpr (!BWD) {
      if (tid == 0) {
        if (p.rstd_out) p.rstd_out[row] = rstd;
        if (LN && p.mean_out) p.mean_out[row] = mean;
      }
      // Each element is read and then written by the same thread, so y may
      // alias x and h_out may alias x or the residual.
      for (int j = tid; j < N; j += nt) {
        float xf = to_f(x[j]);
        if constexpr (OP == FADD_FWD) {
          xf = fadd(xf, to_f(i1[j]));
          (static_cast<T*>(p.out1) + row * p.s_out1)[j] = from_f<T>(xf);
        }
        const float wj = fadd(to_f(wp[j]), p.offset);
        float yf;
        if constexpr (OP == LN_FWD) yf = fadd(fmul(fmul(fsub(xf, mean), rstd), wj), bp ? to_f(bp[j]) : 0.f);
        else                        yf = fmul(fmul(xf, rstd), wj);
        o0[j] = from_f<T>(yf);
      }
    } else {
      float a[NR];
#pragma unroll
      for (int i = 0; i < NR; ++i) a[i] = 0.f;
      for (int j = tid; j < N; j += nt) {
        const float xf = to_f(x[j]);
        const float g = fmul(to_f(i1[j]), fadd(to_f(wp[j]), p.offset));
        if constexpr (LN) {
          const float xh = fmul(fsub(xf, mean), rstd);
          a[0] = fadd(a[0], g);
          a[NR - 1] = ffma(g, xh, a[NR - 1]);
        } else {
          const float xh = fmul(xf, rstd);
          a[0] = ffma(g, xh, a[0]);
        }
      }
      block_sum<NR>(a, red, bank);
      const float mg = LN ? div_n(a[0], N) : 0.f;
      const float mgx = div_n(a[NR - 1], N);
      for (int j = tid; j < N; j += nt) {
        const float xf = to_f(x[j]);
        const float dyf = to_f(i1[j]);
        const float g = fmul(dyf, fadd(to_f(wp[j]), p.offset));
        float xh, dx;
        if constexpr (LN) {
          xh = fmul(fsub(xf, mean), rstd);
          dx = fmul(rstd, fsub(fsub(g, mg), fmul(xh, mgx)));
        } else {
          xh = fmul(xf, rstd);
          dx = fmul(rstd, fsub(g, fmul(xh, mgx)));
        }
        if constexpr (OP == FADD_BWD) {
          if (i2) dx = fadd(dx, to_f(i2[j]));
        }
        o0[j] = from_f<T>(dx);
        if constexpr (DW) wsw[j] = first ? fmul(dyf, xh) : ffma(dyf, xh, wsw[j]);
        if constexpr (DB) wsb[j] = first ? dyf : fadd(wsb[j], dyf);
      }
    }
    first = false;
  }
}

// ===========================================================================
// Launch logic
// ===========================================================================

// Chunks of 16 bytes each thread of the staged kernel owns (0 = too wide).
inline int staged_npt(int nchunks) {
  if (nchunks <= 256) return 1;
  if (nchunks <= 512) return 2;
  if (nchunks <= 2048) return 4;
  return 0;
}

// Allow a kernel the device's full opt-in dynamic shared memory, once per
// (kernel, device).  The attribute is an upper bound only; occupancy follows
// the size actually launched.
inline bool allow_max_smem(const void* fn, const DevInfo& di) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, bool> done;
  std::lock_guard<std::mutex> g(mu);
  auto key = std::make_pair(fn, di.dev);
  if (done.count(key)) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin) != cudaSuccess)
    return false;
  done[key] = true;
  return true;
}

// Cached occupancy query: resident CTAs per SM for (kernel, device, block, smem).
inline int cached_occupancy(const void* fn, const DevInfo& di, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, size_t>, int> cache;
  auto key = std::make_tuple(fn, di.dev, threads, smem);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  if (!allow_max_smem(fn, di)) return -1;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> g(mu);
  cache[key] = nb;
  return nb;
}

template <int OP, class T, class TW, int NPT, bool DW, bool DB>
int launch_staged(const RowParams& p, const DevInfo& di, int nin, int max_ctas, cudaStream_t st, int* grid_out) {
  constexpr int VEC = 16 / (int)sizeof(T);
  const int nchunks = p.N / VEC;
  int threads = (nchunks + NPT - 1) / NPT;
  threads = ((threads + 31) / 32) * 32;
  if (threads < 64) threads = 64;
  const size_t stage_bytes = (size_t)nin * p.N * sizeof(T);
  auto fn = staged_kernel<OP, T, TW, NPT, DW, DB>;
  const void* fp = reinterpret_cast<const void*>(fn);
  const size_t min_smem = kStagedHeader + 2 * stage_bytes;
  if (min_smem > (size_t)di.smem_optin) return NORM_ERR_UNSUPPORTED_INTERNAL;
  // Registers (and the 2-stage minimum) bound the CTAs per SM; shared memory
  // is then split evenly among them, as many stages as fit (<= kMaxStages).
  int nb = cached_occupancy(fp, di, threads, min_smem);
  if (nb < 0) return NORM_ERR_CUDA;
  if (nb == 0) return NORM_ERR_UNSUPPORTED_INTERNAL;
  int ctas = nb < max_ctas ? nb : max_ctas;
  int S = 0;
  size_t smem = 0;
  for (; ctas >= 1; --ctas) {
    size_t per_cta = (size_t)di.smem_per_sm / ctas;
    per_cta = per_cta > (size_t)di.smem_reserved + 64 ? per_cta - di.smem_reserved - 64 : 0;
    if (per_cta > (size_t)di.smem_optin) per_cta = di.smem_optin;
    if (per_cta < min_smem) continue;
    S = (int)((per_cta - kStagedHeader) / stage_bytes);
    if (S > kMaxStages) S = kMaxStages;
    // confirm `ctas` CTAs of this size are resident together
    for (; S >= 2; --S) {
      smem = kStagedHeader + (size_t)S * stage_bytes;
      const int fit = cached_occupancy(fp, di, threads, smem);
      if (fit < 0) return NORM_ERR_CUDA;
      if (fit >= ctas) break;
    }
    if (S >= 2) break;
  }
  if (ctas < 1 || S < 2) return NORM_ERR_UNSUPPORTED_INTERNAL;
  int64_t G = (int64_t)di.sms * ctas;
  if (G > p.M) G = p.M;
  if ((DW || DB) && G > di.max_partial_rows) G = di.max_partial_rows;
  fn<<<(unsigned)G, threads, smem, st>>>(p, S);
  if (cudaGetLastError() != cudaSuccess) return NORM_ERR_CUDA;
  *grid_out = (int)G;
  return NORM_OK;
}

template <int OP, class T, class TW, bool DW, bool DB>
int launch_loop(const RowParams& p, const DevInfo& di, cudaStream_t st, int* grid_out) {
  const int threads = p.N >= 4096 ? 512 : (p.N >= 1024 ? 256 : 128);
  auto fn = loop_kernel<OP, T, TW, DW, DB>;
  int nb = cached_occupancy(reinterpret_cast<const void*>(fn), di, threads, 0);
  if (nb < 0) return NORM_ERR_CUDA;
  if (nb < 1) nb = 1;
  int64_t G = (int64_t)di.sms * nb;
  if (G > p.M) G = p.M;
  if ((DW || DB) && G > di.max_partial_rows) G = di.max_partial_rows;
  fn<<<(unsigned)G, threads, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return NORM_ERR_CUDA;
  *grid_out = (int)G;
  return NORM_OK;
}

// Row kernel for one (op, types, flags): the staged path when every streamed
// row starts on a 16-byte boundary and fits, else the loop path.
template <int OP, class T, class TW, bool DW, bool DB>
int launch_rows(const RowParams& p, const DevInfo& di, bool rows_aligned, cudaStream_t st, int* grid_out) {
  constexpr int VEC = 16 / (int)sizeof(T);
  const int nin = (OP == FADD_BWD && p.in2 == nullptr) ? 2 : OpInfo<OP>::NIN;
  const int max_ctas = (DW || DB) ? 2 : 4;
  if (rows_aligned && p.N % VEC == 0 && di.force_path != 2) {
    int rc = NORM_ERR_UNSUPPORTED_INTERNAL;
    switch (staged_npt(p.N / VEC)) {
      case 1: rc = launch_staged<OP, T, TW, 1, DW, DB>(p, di, nin, max_ctas, st, grid_out); break;
      case 2: rc = launch_staged<OP, T, TW, 2, DW, DB>(p, di, nin, max_ctas, st, grid_out); break;
      case 4: rc = launch_staged<OP, T, TW, 4, DW, DB>(p, di, nin, max_ctas, st, grid_out); break;
      default: break;
    }
    if (rc != NORM_ERR_UNSUPPORTED_INTERNAL) return rc;
  }
  return launch_loop<OP, T, TW, DW, DB>(p, di, st, grid_out);
}

// Dispatch on the (dtype, w_dtype) pair.
template <int OP, bool DW, bool DB>
int launch_typed(const RowParams& p, int dtype, int wdtype, const DevInfo& di, bool al, cudaStream_t st, int* g) {
  if (dtype == NORM_F32 && wdtype == NORM_F32) return launch_rows<OP, float, float, DW, DB>(p, di, al, st, g);
  if (dtype == NORM_F16 && wdtype == NORM_F16) return launch_rows<OP, __half, __half, DW, DB>(p, di, al, st, g);
  if (dtype == NORM_BF16 && wdtype == NORM_BF16)
    return launch_rows<OP, __nv_bfloat16, __nv_bfloat16, DW, DB>(p, di, al, st, g);
  if (dtype == NORM_BF16 && wdtype == NORM_F32) return launch_rows<OP, __nv_bfloat16, float, DW, DB>(p, di, al, st, g);
  if (dtype == NORM_F16 && wdtype == NORM_F32) return launch_rows<OP, __half, float, DW, DB>(p, di, al, st, g);
  return NORM_ERR_DTYPE;
}

}  // namespace gb300norm
