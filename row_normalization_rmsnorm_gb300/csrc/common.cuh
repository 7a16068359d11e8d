// common.cuh -- shared device helpers of the row-normalisation kernels:
// element types, FP32 arithmetic with fixed rounding, warp/CTA reductions and
// the PTX wrappers for mbarriers and bulk (TMA-engine) copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gb300norm {

// ---------------------------------------------------------------------------
// Operation kinds and launch parameters
// ---------------------------------------------------------------------------
enum OpKind : int { RMS_FWD = 0, RMS_BWD = 1, LN_FWD = 2, LN_BWD = 3, FADD_FWD = 4, FADD_BWD = 5 };

// One struct for every kernel; unused fields are null / zero.
struct RowParams {
  // streamed row inputs (element strides)
  const void* in0;  int64_t s_in0;   // x (h for FADD_BWD)
  const void* in1;  int64_t s_in1;   // dy (backward) or residual (FADD_FWD)
  const void* in2;  int64_t s_in2;   // dh_out (FADD_BWD), nullable
  // row outputs
  void* out0;       int64_t s_out0;  // y (forward) or dx (backward)
  void* out1;       int64_t s_out1;  // h_out (FADD_FWD)
  // per-column parameters
  const void* w;
  const void* b;                     // LayerNorm bias, nullable
  // per-row statistics
  float* mean_out;  float* rstd_out;       // forward, nullable
  const float* mean_in; const float* rstd_in;  // backward, nullable = recompute
  // dW / dB partial rows, [gridDim.x][N] FP32
  float* ws_dw;     float* ws_db;
  int64_t M;
  int N;
  float offset;
  float eps;
  int* status;      // device status word (bounded waits that ran out)
  // test hook: each row group's producer issues no copy for its last row, so
  // the wait for that row runs out (the bounded-wait abort path, exercised)
  int hold_last;
};

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------
template <class T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__half> {
  static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <class T> __device__ __forceinline__ float to_f(T v) { return Elem<T>::to_f(v); }
template <class T> __device__ __forceinline__ T from_f(float v) { return Elem<T>::from_f(v); }

// 16 bytes of T as an array; VEC elements.
template <class T> struct Vec16 {
  static constexpr int VEC = 16 / (int)sizeof(T);
  union { uint4 u; T e[16 / sizeof(T)]; };
};

// Unpack 16 bytes of T into VEC floats (exact) and pack VEC floats back,
// rounding each to nearest-even: two elements per instruction for the
// 16-bit types.
template <class T> struct Pack16;
template <> struct Pack16<float> {
  static __device__ __forceinline__ void unpack(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ void unpack(const uint4& u, float2 (&f)[2]) {
    f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
  static __device__ __forceinline__ uint4 pack(const float2 (&f)[2]) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x), __float_as_uint(f[1].y));
  }
};
template <> struct Pack16<__nv_bfloat16> {
  static __device__ __forceinline__ void word(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
  static __device__ __forceinline__ void unpack(const uint4& u, float (&f)[8]) {
    word(u.x, f[0], f[1]); word(u.y, f[2], f[3]); word(u.z, f[4], f[5]); word(u.w, f[6], f[7]);
  }
  static __device__ __forceinline__ uint32_t two(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ uint4 pack(const float (&f)[8]) {
    return make_uint4(two(f[0], f[1]), two(f[2], f[3]), two(f[4], f[5]), two(f[6], f[7]));
  }
  static __device__ __forceinline__ void unpack(const uint4& u, float2 (&f)[4]) {
    word(u.x, f[0].x, f[0].y); word(u.y, f[1].x, f[1].y); word(u.z, f[2].x, f[2].y); word(u.w, f[3].x, f[3].y);
  }
  static __device__ __forceinline__ uint4 pack(const float2 (&f)[4]) {
    return make_uint4(two(f[0].x, f[0].y), two(f[1].x, f[1].y), two(f[2].x, f[2].y), two(f[3].x, f[3].y));
  }
};
template <> struct Pack16<__half> {
  static __device__ __forceinline__ void word(uint32_t w, float& lo, float& hi) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 f = __half22float2(h);
    lo = f.x; hi = f.y;
  }
  static __device__ __forceinline__ void unpack(const uint4& u, float (&f)[8]) {
    word(u.x, f[0], f[1]); word(u.y, f[2], f[3]); word(u.z, f[4], f[5]); word(u.w, f[6], f[7]);
  }
  static __device__ __forceinline__ uint32_t two(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ uint4 pack(const float (&f)[8]) {
    return make_uint4(two(f[0], f[1]), two(f[2], f[3]), two(f[4], f[5]), two(f[6], f[7]));
  }
  static __device__ __forceinline__ void unpack(const uint4& u, float2 (&f)[4]) {
    word(u.x, f[0].x, f[0].y); word(u.y, f[1].x, f[1].y); word(u.z, f[2].x, f[2].y); word(u.w, f[3].x, f[3].y);
  }
  static __device__ __forceinline__ uint4 pack(const float2 (&f)[4]) {
    return make_uint4(two(f[0].x, f[0].y), two(f[1].x, f[1].y), two(f[2].x, f[2].y), two(f[3].x, f[3].y));
  }
};

// ---------------------------------------------------------------------------
// FP32 arithmetic with explicit rounding.  Every value a kernel writes is
// computed through these, so the compiler cannot contract or reorder them
// differently between the trainable and the frozen instantiation of a
// kernel: the input gradient is bit-identical in both.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float ffma(float a, float b, float c) { return __fmaf_rn(a, b, c); }

// Packed pairs: one sm_100-family instruction (add / mul / fma .rn.f32x2)
// applies the operation to both lanes, each rounded exactly as the scalar
// form above, so a loop over pairs gives the bits of the loop over elements
// with half the floating-point instructions.  Unlike the scalar forms, a
// packed multiply whose result feeds a packed add may still be fused into
// one FMA by the compiler, and whether it is differs between
// instantiations.  The kernels therefore never write that pattern: where a
// product meets a sum they call ffma2 themselves.  a - b is written
// a + (-b), the same IEEE operation.
__device__ __forceinline__ float2 f2s(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// ---------------------------------------------------------------------------
// Reductions.  Butterfly shuffles give every lane the same sum (each step adds
// the same two operands on both partners); warps are combined in a fixed
// order.  `red` holds two banks of [32 warps][kMaxReduceValues] floats used
// alternately so that consecutive reductions need only one barrier each.
// ---------------------------------------------------------------------------
template <int NV>
__device__ __forceinline__ void warp_sum(float (&v)[NV]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = fadd(v[i], __shfl_xor_sync(0xffffffffu, v[i], o));
}

// Values one block_sum call may reduce; each bank has room for that many per
// warp, whatever a given call uses, so consecutive calls never share slots.
constexpr int kMaxReduceValues = 2;

// Two values reduced together: one packed add per butterfly step.
__device__ __forceinline__ void warp_sum2(float2& v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float2 t = make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
    v = fadd2(v, t);
  }
}

// A CTA-wide sum in two halves around one barrier: reduce_warps sums each
// warp's values and has lane 0 store them in bank `bank` of `red`;
// reduce_finish (after a __syncthreads) sums the warps' values.  Every warp
// reduces the same warp partials with the same butterfly, so every thread of
// the CTA ends with the same bits.  Two values go through packed adds.
template <int NV>
__device__ __forceinline__ void reduce_warps(float (&v)[NV], float* red, int bank) {
  static_assert(NV <= kMaxReduceValues, "bank size");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* r = red + bank * 32 * kMaxReduceValues;
  if constexpr (NV == 2) {
    float2 s = make_float2(v[0], v[1]);
    warp_sum2(s);
    if (lane == 0) reinterpret_cast<float2*>(r)[warp] = s;
  } else {
    warp_sum<NV>(v);
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < NV; ++i) r[warp * NV + i] = v[i];
    }
  }
}

template <int NV>
__device__ __forceinline__ void reduce_finish(float (&v)[NV], const float* red, int bank) {
  const int lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const float* r = red + bank * 32 * kMaxReduceValues;
  if constexpr (NV == 2) {
    float2 s = (lane < nw) ? reinterpret_cast<const float2*>(r)[lane] : make_float2(0.f, 0.f);
    warp_sum2(s);
    v[0] = s.x;
    v[1] = s.y;
  } else {
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = (lane < nw) ? r[lane * NV + i] : 0.f;
    warp_sum<NV>(v);
  }
}

template <int NV>
__device__ __forceinline__ void block_sum(float (&v)[NV], float* red, int& bank) {
  reduce_warps<NV>(v, red, bank);
  __syncthreads();
  reduce_finish<NV>(v, red, bank);
  bank ^= 1;
}

// Sum of VEC per-lane accumulators in a fixed tree order.
template <int VEC>
__device__ __forceinline__ float tree_sum(const float (&a)[VEC]) {
  if constexpr (VEC == 4) return fadd(fadd(a[0], a[1]), fadd(a[2], a[3]));
  else return fadd(fadd(fadd(a[0], a[1]), fadd(a[2], a[3])), fadd(fadd(a[4], a[5]), fadd(a[6], a[7])));
}
// The same sum over accumulators held as pairs (lanes 2h, 2h+1 in a[h]):
// the pairs are added lane-wise first (packed), then the two lanes.
template <int H>
__device__ __forceinline__ float2 pair_tree(const float2 (&a)[H]) {
  if constexpr (H == 2) return fadd2(a[0], a[1]);
  else return fadd2(fadd2(a[0], a[1]), fadd2(a[2], a[3]));
}
template <int H>
__device__ __forceinline__ float tree_sum(const float2 (&a)[H]) {
  const float2 t = pair_tree<H>(a);
  return fadd(t.x, t.y);
}
// Two such sums at once: (sum of a, sum of b).
template <int H>
__device__ __forceinline__ float2 tree_sum_2(const float2 (&a)[H], const float2 (&b)[H]) {
  const float2 s = pair_tree<H>(a), t = pair_tree<H>(b);
  return fadd2(make_float2(s.x, t.x), make_float2(s.y, t.y));
}

// 1/sqrt(m + eps).
__device__ __forceinline__ float inv_rms(float m, float eps) { return rsqrtf(fadd(m, eps)); }

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy PTX (sm_90+ instructions, used on sm_103a)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// try_wait suspends the calling thread until the phase completes or the
// suspend-time hint (ns) passes, so a waiting warp does not spin on the
// issue slots its neighbours need.
constexpr uint32_t kSuspendHintNs = 1000000;   // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound of any single wait for a row copy.  A copy of at most a few
// hundred KB lands in microseconds; the bound only ends a wait that would
// otherwise never finish.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Wait until the phase with the given parity of `bar` has completed, or
// until the global timer passes `deadline` (ns); false in the second case
// (the barrier is left untouched).
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  if (mbar_try_wait(bar, parity)) return true;
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() > deadline) return false;
  }
}

// The same with a limit of kWaitLimitNs from now.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_until(bar, parity, global_timer_ns() + kWaitLimitNs);
}

// try_wait with acquire semantics at cluster scope: for a phase completed by
// other CTAs' stores into this CTA's shared memory (released at cluster
// scope), so that their data is visible once the phase is seen complete.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Bounded (kWaitLimitNs) wait with cluster-scope acquire.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() > deadline) return false;
  }
}


__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy global -> shared through the TMA engine, completing `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 16-byte global store with the streaming (evict-first) hint.
__device__ __forceinline__ void st_global_cs16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Programmatic dependent launch.  Every kernel of this library is launched
// so that it may start while the previous kernel on the stream drains; it
// calls grid_dependency_wait() before its first global-memory access (which
// returns once the previous grid has completed and its writes are visible,
// at once when there is no such grid), and grid_launch_dependents() once its
// own main work is done, letting the next kernel be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters (sm_90+ instructions, used on sm_103a)
// ---------------------------------------------------------------------------
// CTAs in this CTA's cluster (1 when the kernel was not launched as a
// cluster), and this CTA's rank among them.
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives, then waits for all the
// others; shared-memory writes before it are visible to the cluster after.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address, in CTA `rank` of the cluster, of the variable at shared
// address `addr` of this CTA.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Asynchronous store of one or two floats into another CTA's shared memory,
// completing their bytes on that CTA's mbarrier.
__device__ __forceinline__ void st_async_f32(uint32_t remote, float a, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
               ::"r"(remote), "f"(a), "r"(remote_bar) : "memory");
}
__device__ __forceinline__ void st_async_f32x2(uint32_t remote, float a, float b, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(remote), "f"(a), "f"(b), "r"(remote_bar) : "memory");
}

// Status bits written to RowParams::status.
enum : int { STATUS_WAIT_TIMEOUT = 1 };

}  // namespace gb300norm
