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

// Mean of a row sum: multiplied by the FP32 reciprocal of N formed once per
// kernel (within 1.5 ulp of the quotient).
__device__ __forceinline__ float div_n(float s, float inv_n) { return fmul(s, inv_n); }

// ===========================================================================
// Staged (TMA bulk copy) kernel
// ===========================================================================
constexpr int kStagedHeader = 1024;   // bytes: S mbarriers (<= 32) + reduction banks
constexpr int kMaxStages = 16;
constexpr int kInflightUnits = 8;     // default cap on row bytes in flight per SM, x 16 KB
// The LayerNorm kernels run best with a ring of 4 stages whatever the row
// bytes in flight: measured against 5 and 6 (and the in-flight cap alone),
// the forward gains 0.5-7 % at every shape from 2048 x 4096 to 32768 x 4096
// (4096 x 4096 17.4 -> 16.4 us, 65536 x 1024 74.9 -> 69.6 us) and the
// backward up to 4 % (trainable, 8192 x 4096 40.9 -> 39.1 us), nothing
// slower; for RMSNorm and FusedAdd the cap made no difference.
constexpr int kLnMaxStages = 4;
// Where a staged instantiation keeps W' (and the bias): registers up to 4
// chunks per thread, shared memory beyond.
__host__ __device__ constexpr bool staged_wreg(int npt) { return npt <= 4; }

// Shared memory for per-column values (W', and the LayerNorm bias) when they
// are kept in shared memory rather than registers.
template <int OP>
__host__ __device__ constexpr size_t staged_col_bytes(int N, bool wreg) {
  return wreg ? 0 : ((size_t)N * 4 * (OP == LN_FWD ? 2 : 1) + 127) / 128 * 128;
}

// EXACT: the CTA's threads own exactly its nchunks chunks (threads x NPT ==
// nchunks), so no per-chunk bounds test is compiled into the row loop.
//
// CL: launched as thread-block clusters of C CTAs (C = 2, 4 or 8), the C
// CTAs of a cluster split every row of the cluster into C equal column
// slices: each streams, reduces and writes only its slice, and the CTAs
// exchange their row sums through distributed shared memory (each stores
// its sums into every peer with st.async, completing on the peer's
// mbarrier) and add them in rank order, so all CTAs of the cluster hold the
// same bits.  This serves rows that one CTA cannot take without spilling
// registers (more than 4096 chunks, or the per-column state of a wide
// backward).  The dW / dB partial row of a cluster is written slice by
// slice by its CTAs.  Without CL the cluster code is compiled out.
// Launch bounds of a staged instantiation.
//  * 512 threads, so at most 128 registers a thread, with the compiler's own
//    register target: the forwards and the trainable RMSNorm / FusedAdd
//    backwards.
//  * The LayerNorm backward with both dW and dB at 4 chunks per thread holds
//    W', dW and dB for 32 columns a thread (96 registers of state): under a
//    128-register cap it spills.  Bounded at 256 threads and one CTA per SM it
//    keeps everything in registers: at N = 8192 it runs one 256-thread CTA
//    per SM with 32 elements per thread per row, measured faster than 2
//    chunks per thread at 512 threads (71.5 vs 75.0 us at 8192 x 8192, 41.0
//    vs 43.3 us at 4096 x 8192, 53.2 vs 65.5 us at 1024 x 32768).  The
//    registers left over then hold the row's x - mean and dy from the first
//    pass to the second (KEEPB, about 210 registers in all), which saves the
//    second pass its shared-memory reads, unpacking and subtraction: another
//    3-7 % (8192 x 8192 75.7 -> 71.8 us, 4096 x 4096 28.7 -> 26.6 us).
//  * The frozen RMSNorm and LayerNorm backwards are also compiled for one
//    CTA per SM (512 threads): given more registers than the compiler's own
//    target they were measured level or faster everywhere (up to 14 %: the
//    frozen LayerNorm backward at 8192 x 4096, 30.7 -> 28.7 us), while the
//    same hint slowed the forwards.
template <int OP, bool DW, bool DB, int NPT>
struct StagedBounds {
  static constexpr bool WIDE_STATE = (OP == LN_BWD) && DW && DB && NPT == 4;
  static constexpr bool FROZEN_BWD = (OP == RMS_BWD || OP == LN_BWD) && !DW && !DB;
  static constexpr int THREADS = WIDE_STATE ? 256 : 512;
  static constexpr int MIN_CTAS = (WIDE_STATE || FROZEN_BWD) ? 1 : 0;   // 0: the compiler's choice
};

template <int OP, class T, class TW, int NPT, bool DW, bool DB, bool EXACT, bool CL>
__global__ void __launch_bounds__(StagedBounds<OP, DW, DB, NPT>::THREADS, StagedBounds<OP, DW, DB, NPT>::MIN_CTAS)
    staged_kernel(const RowParams p, const int S) {
  constexpr int VEC = 16 / (int)sizeof(T);
  constexpr int H = VEC / 2;   // element pairs per chunk
  constexpr bool LN = (OP == LN_FWD || OP == LN_BWD);
  constexpr bool BWD = OpInfo<OP>::BWD;
  // Up to 4 chunks per thread, W' (and the bias) live in registers; at 8
  // (the only staged shape for rows of 2049-4096 chunks) they move to shared
  // memory to leave the registers to the dW / dB accumulators.
  constexpr bool WREG = staged_wreg(NPT);
  // The FusedAdd forward keeps its FP32 row h in registers between passes
  // (up to 4 chunks per thread); RMSNorm and LayerNorm re-read theirs from
  // the stage (fewer registers, more resident CTAs).
  constexpr bool KEEP = (OP == FADD_FWD) && NPT <= 4;
  constexpr int NWR = WREG ? NPT : 1;
  constexpr int NB = (OP == LN_FWD && WREG) ? NPT : 1;   // bias registers
  constexpr int NDW = DW ? NPT : 1;
  constexpr int NDB = DB ? NPT : 1;
  constexpr int NX = KEEP ? NPT : 1;             // forward rows kept in registers
  constexpr int NR = (OP == LN_BWD) ? 2 : 1;     // values reduced per backward row
  // trainable LayerNorm backward at 4 chunks per thread (256 threads, one
  // CTA per SM, up to 255 registers): the row's x - mean and dy stay in
  // registers from the first pass to the second
  constexpr bool KEEPB = StagedBounds<OP, DW, DB, NPT>::WIDE_STATE;
  constexpr int NKB = KEEPB ? NPT : 1;
  using P = Pack16<T>;
  const int N = p.N;
  // cluster: C CTAs, this one's rank, and its slice of chunks (the launcher
  // makes the slices equal): chunk c of the slice is chunk col0 + c of a row
  const int ncl = CL ? (int)cluster_nctarank() : 1;
  const int crank = CL ? (int)cluster_ctarank() : 0;
  const int nchunks = N / VEC / ncl;
  const int col0 = crank * nchunks;
  const int NL = nchunks * VEC;   // columns of the slice
  const int tid = threadIdx.x, nt = blockDim.x;
  const uint32_t row_bytes = (uint32_t)nchunks * 16u;
  const int nin = (OP == FADD_BWD && p.in2 == nullptr) ? 2 : OpInfo<OP>::NIN;
  const uint32_t stage_bytes = (uint32_t)nin * row_bytes;

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + 256);
  float* wsm = reinterpret_cast<float*>(smem + kStagedHeader);   // W' [NL] (+ bias [NL]) when !WREG
  unsigned char* stages = smem + kStagedHeader + staged_col_bytes<OP>(NL, WREG);
  // abort_flag[k & 1] is raised while row k is awaited and read after row
  // k's barrier, so a thread already waiting for row k+1 cannot change what
  // the others read for row k.
  __shared__ int abort_flag[2];
  // cluster exchange: two slots (used alternately) of every rank's row sums
  // and, per slot, the mbarrier the peers' stores complete on
  __shared__ __align__(16) float xch[2][8][kMaxReduceValues];
  __shared__ __align__(8) uint64_t xbar[2];

  grid_dependency_wait();

  // Row counters of this CTA are 32-bit: the launcher guarantees that no CTA
  // owns 2^31 or more rows.
  // Rows of cluster c (c = blockIdx.x / C, one CTA per cluster without
  // clusters): c, c + G, c + 2G, ... with G clusters.
  const int G = gridDim.x / ncl;
  const int row0 = blockIdx.x / ncl;
  const int nrows = (int)((p.M - row0 + G - 1) / G);   // >= 1: the grid never exceeds M clusters
  // Copies are issued for rows issued < nrows - p.hold_last: every row, or
  // (test hook, hold_last = 1) all but the last, whose wait then runs out
  // after every earlier copy has landed.  (Read from the parameter at each
  // use rather than kept in a register.)
  const uint64_t pol = l2_policy_evict_first();
  // the streamed inputs, each from this CTA's first column (nullable ones stay null)
  auto slice = [&](const void* q) { return q ? static_cast<const char*>(q) + (size_t)col0 * 16 : nullptr; };
  const char* g0 = slice(p.in0);
  const char* g1 = slice(p.in1);
  const char* g2 = slice(p.in2);
  const float inv_n = 1.0f / (float)N;
  // Producer state (thread 0): rows of this CTA whose copies have been
  // issued, and the stage the next one goes to.  Stage and phase indices
  // advance by counting, never by dividing the row index.
  int issued = 0;
  int istage = 0;

  auto issue_next = [&]() {
    const int64_t row = row0 + (int64_t)issued * G;
    unsigned char* dst = stages + (size_t)istage * stage_bytes;
    uint64_t* bar = &bars[istage];
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, stage_bytes);
    bulk_g2s(dst, g0 + row * p.s_in0 * (int64_t)sizeof(T), row_bytes, bar, pol);
    if (nin > 1) bulk_g2s(dst + row_bytes, g1 + row * p.s_in1 * (int64_t)sizeof(T), row_bytes, bar, pol);
    if (nin > 2) bulk_g2s(dst + 2 * row_bytes, g2 + row * p.s_in2 * (int64_t)sizeof(T), row_bytes, bar, pol);
    ++issued;
    if (++istage == S) istage = 0;
  };
  // Thread 0 sets up the ring and issues the first S-1 row copies before the
  // per-column values are loaded, so the two latencies overlap.
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    if constexpr (CL) {
      mbar_init(&xbar[0], 1);
      mbar_init(&xbar[1], 1);
    }
    fence_mbar_init();
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    while (issued + p.hold_last < nrows && issued < S - 1) issue_next();
  }

  // Per-thread constant columns: W' = float(w) + offset (and the LayerNorm
  // bias) in FP32, formed once per CTA.  Elementwise values are held as
  // pairs (float2, lanes 2h and 2h+1 of a chunk) for the packed FP32
  // instructions.
  float2 wv[NWR][H];
  float2 bv[NB][H];
  const bool has_b = (OP == LN_FWD) && p.b != nullptr;
  const TW* wp = static_cast<const TW*>(p.w);
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    const int c = tid + j * nt;
#pragma unroll
    for (int h = 0; h < H; ++h) {
      float wj[2], bj[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = (col0 + c) * VEC + 2 * h + e;
        wj[e] = (c < nchunks) ? fadd(to_f(wp[col]), p.offset) : 0.f;
        bj[e] = (has_b && c < nchunks) ? to_f(static_cast<const TW*>(p.b)[col]) : 0.f;
      }
      if constexpr (WREG) {
        wv[j][h] = make_float2(wj[0], wj[1]);
        if constexpr (OP == LN_FWD) bv[j][h] = make_float2(bj[0], bj[1]);
      } else if (c < nchunks) {
        reinterpret_cast<float2*>(wsm)[c * H + h] = make_float2(wj[0], wj[1]);
        if constexpr (OP == LN_FWD) reinterpret_cast<float2*>(wsm + NL)[c * H + h] = make_float2(bj[0], bj[1]);
      }
    }
  }
  // W' (or the bias) of chunk c, slot j, into w[H]
  auto colv = [&](int j, int c, int which, float2 (&w)[H]) {
    if constexpr (WREG) {
#pragma unroll
      for (int h = 0; h < H; ++h) w[h] = which ? bv[NB > 1 ? j : 0][h] : wv[j][h];
    } else {
      const float4* q = reinterpret_cast<const float4*>(wsm + (which ? NL : 0) + c * VEC);
#pragma unroll
      for (int h = 0; h < H; h += 2) {
        const float4 t = q[h / 2];
        w[h] = make_float2(t.x, t.y); w[h + 1] = make_float2(t.z, t.w);
      }
    }
  };
  float2 dwa[NDW][H];
  float2 dba[NDB][H];
#pragma unroll
  for (int j = 0; j < NDW; ++j)
#pragma unroll
    for (int h = 0; h < H; ++h) dwa[j][h] = f2s(0.f);
#pragma unroll
  for (int j = 0; j < NDB; ++j)
#pragma unroll
    for (int h = 0; h < H; ++h) dba[j][h] = f2s(0.f);

  // ring initialised (and first copies issued) by thread 0; in a cluster,
  // every CTA's exchange barriers are initialised before any peer stores
  if constexpr (CL) cluster_barrier();
  else __syncthreads();

  // Cluster exchange of the CTA's row sums v (every thread holds them): the
  // sums of all C CTAs are added in rank order into v.  A wait that runs out
  // raises the abort flag of the next row (read after its barrier).
  int xn = 0;   // exchanges done (slot xn & 1, its use (xn >> 1) sets the phase)
  auto cluster_sum = [&](auto& v, int next_fl) {
    constexpr int NV = (int)(sizeof(v) / sizeof(float));
    const int slot = xn & 1;
    const uint32_t ph = (uint32_t)((xn >> 1) & 1);
    ++xn;
    if (tid == 0) {
      mbar_arrive_expect_tx(&xbar[slot], (uint32_t)((ncl - 1) * NV * 4));
      const uint32_t mine = smem_addr(&xch[slot][crank][0]);
      const uint32_t bar = smem_addr(&xbar[slot]);
      for (int q = 0; q < ncl; ++q) {
        if (q == crank) continue;
        if constexpr (NV == 2)
          st_async_f32x2(map_shared_rank(mine, q), v[0], v[1], map_shared_rank(bar, q));
        else
          st_async_f32(map_shared_rank(mine, q), v[0], map_shared_rank(bar, q));
      }
    }
    if (!mbar_wait_cluster_bounded(&xbar[slot], ph)) {
      atomicOr(p.status, STATUS_WAIT_TIMEOUT);
      abort_flag[next_fl] = 1;
    }
    float t[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) t[i] = 0.f;
    for (int q = 0; q < ncl; ++q) {
#pragma unroll
      for (int i = 0; i < NV; ++i) t[i] = fadd(t[i], q == crank ? v[i] : xch[slot][q][i]);
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = t[i];
  };
  // The row sums of the whole row: the CTA's (block_sum), then, in a
  // cluster, every CTA's.
  auto row_sum = [&](auto& v, int& bnk, int next_fl) {
    block_sum(v, red, bnk);
    if constexpr (CL) cluster_sum(v, next_fl);
  };


  // Saved statistics of the backward are read one row ahead, off the
  // critical path of the row being processed.
  const bool have_stats = BWD && p.rstd_in != nullptr;
  float rs_next = 0.f, mu_next = 0.f;
  if (have_stats) {
    rs_next = p.rstd_in[row0];
    if constexpr (LN) mu_next = p.mean_in[row0];
  }

  // LayerNorm forward: this thread's element count n_t (and 1 / n_t) and its
  // statistics of the row after the current one: shift, mean offset, M2.
  float ln_nt = 0.f, ln_inv_nt = 0.f, ln_c = 0.f, ln_off = 0.f, ln_m2 = 0.f;
  if constexpr (OP == LN_FWD) {
    int nv = 0;
#pragma unroll
    for (int j = 0; j < NPT; ++j) nv += (tid + j * nt < nchunks) ? 1 : 0;
    ln_nt = (float)(nv * VEC);
    ln_inv_nt = nv ? 1.0f / ln_nt : 0.f;
  }

  // ---- backward: the two passes over a staged row -----------------------
  // bwd_local: this thread's sums over its chunks of the row staged at q0 (x,
  // or h, then dy), with g = dy W': (sum g, sum g (x - mean)) for LayerNorm,
  // (0, sum g x) for RMSNorm.  sum(g xhat) = rstd sum(g (x - mean)): rstd is
  // applied once to the row total rather than to every element.
  float2 kxm[NKB][H], kdy[NKB][H];   // (KEEPB) x - mean and dy of the current row
  auto bwd_local = [&](const uint4* q0, float mean) -> float2 {
    const uint4* q1 = q0 + nchunks;
    const float2 nmean = f2s(-mean);
    float2 acc0[H], acc1[H];
#pragma unroll
    for (int h = 0; h < H; ++h) { acc0[h] = f2s(0.f); acc1[h] = f2s(0.f); }
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int c = tid + j * nt;
      if (EXACT || c < nchunks) {
        float2 xf[H], df[H], w[H];
        P::unpack(q0[c], xf);
        P::unpack(q1[c], df);
        colv(j, c, 0, w);
#pragma unroll
        for (int h = 0; h < H; ++h) {
          const float2 g = fmul2(df[h], w[h]);
          if constexpr (LN) {
            const float2 xm = fadd2(xf[h], nmean);
            acc0[h] = ffma2(df[h], w[h], acc0[h]);   // sum of g, each product unrounded
            acc1[h] = ffma2(g, xm, acc1[h]);
            if constexpr (KEEPB) { kxm[j][h] = xm; kdy[j][h] = df[h]; }
          } else {
            acc1[h] = ffma2(g, xf[h], acc1[h]);
          }
        }
      }
    }
    if constexpr (LN) return tree_sum_2<H>(acc0, acc1);
    else return make_float2(0.f, tree_sum<H>(acc1));
  };
  // bwd_out: dx of the row staged at q0 from its CTA totals tot (bwd_local's
  // sums over every thread), accumulating dW / dB.
  // dx = rstd * (g - xhat * mean(g xhat) - mean(g)) + dh, written as fused
  // multiply-adds of negated row constants; where a product meets a sum the
  // two are one fused multiply-add (dy * W' - mean(g), and the residual
  // gradient added to rstd * (...)), never a rounded product followed by an
  // add, which the compiler could fuse on its own.
  auto bwd_out = [&](const uint4* q0, int64_t row, float rstd, float mean, float2 tot) {
    const uint4* q1 = q0 + nchunks;
    const uint4* q2 = q1 + nchunks;
    const float2 rs2 = f2s(rstd);
    const float2 nmean = f2s(-mean);
    const float2 nmg = f2s(LN ? -div_n(tot.x, inv_n) : 0.f);
    const float2 nmgx = f2s(-div_n(fmul(tot.y, rstd), inv_n));
    const bool has_dh = (OP == FADD_BWD) && nin > 2;
    T* dxrow = static_cast<T*>(p.out0) + row * p.s_out0;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int c = tid + j * nt;
      if (EXACT || c < nchunks) {
        float2 xf[H], df[H], hf[H], of[H], w[H];
        if constexpr (KEEPB) {
#pragma unroll
          for (int h = 0; h < H; ++h) { xf[h] = kxm[j][h]; df[h] = kdy[j][h]; }
        } else {
          P::unpack(q0[c], xf);
          P::unpack(q1[c], df);
        }
        if (has_dh) P::unpack(q2[c], hf);
        colv(j, c, 0, w);
#pragma unroll
        for (int h = 0; h < H; ++h) {
          float2 xh, t;
          if constexpr (LN) {
            xh = fmul2(KEEPB ? xf[h] : fadd2(xf[h], nmean), rs2);
            t = ffma2(xh, nmgx, ffma2(df[h], w[h], nmg));
          } else {
            xh = fmul2(xf[h], rs2);
            t = ffma2(xh, nmgx, fmul2(df[h], w[h]));
          }
          const float2 dx = has_dh ? ffma2(rs2, t, hf[h]) : fmul2(rs2, t);
          of[h] = dx;
          if constexpr (DW) dwa[j][h] = ffma2(df[h], xh, dwa[j][h]);
          if constexpr (DB) dba[j][h] = fadd2(dba[j][h], df[h]);
        }
        st_global_cs16(dxrow + (int64_t)(col0 + c) * VEC, P::pack(of));
      }
    }
  };
  int bank = 0;
  int k = 0;
  int s = 0;            // stage of row k
  uint32_t phase = 0;   // parity of that stage's current use
  bool aborted = false;
  for (; k < nrows; ++k, (++s == S) ? (s = 0, phase ^= 1u) : 0) {
    const int64_t row = row0 + (int64_t)k * G;
    const int fl = (int)(k & 1);
    float mean = 0.f, rstd = 0.f;
    if (have_stats) {
      rstd = rs_next;
      mean = mu_next;
      if (k + 1 < nrows) {
        rs_next = p.rstd_in[row + G];
        if constexpr (LN) mu_next = p.mean_in[row + G];
      }
    }
    // (the LayerNorm forward waits for row k+1 during row k: see below)
    if ((OP != LN_FWD || k == 0) && !mbar_wait_bounded(&bars[s], phase)) {
      atomicOr(p.status, STATUS_WAIT_TIMEOUT);
      abort_flag[fl] = 1;
    }
    const uint4* r0 = reinterpret_cast<const uint4*>(stages + (size_t)s * stage_bytes);
    const uint4* r1 = r0 + nchunks;

    // After the first barrier of row k every thread has finished row k-1, so
    // its stage can take the copy of row k+S-1.
    bool refilled = false;
    auto after_first_barrier = [&]() {
      if (refilled) return;
      refilled = true;
      if (tid == 0 && !abort_flag[fl] && issued + p.hold_last < nrows) issue_next();
    };

    if constexpr (OP == LN_FWD) {
      // ---- LayerNorm forward, statistics software-pipelined -------------
      // Each thread takes, in one pass over its own elements of a row, the
      // sums S = sum(x - c) and Q = sum((x - c)^2) about a shift c that is
      // one of those elements, so its M2 = Q - S^2/n loses at most a factor
      // 1 + n to cancellation.  The CTA merges the threads exactly with the
      // pairwise update of Chan, Golub and LeVeque: M2 = sum(M2_t) +
      // sum(n_t d_t^2), d_t = (c_t - mean) + S_t / n_t, the deviation formed
      // from the small terms so that a large mean costs it nothing.  One
      // barrier per row reduces the M2 terms of row k (whose mean came from
      // the previous barrier) together with the sum of row k+1; each row is
      // read from its stage twice (statistics, output).  Rows k and k+1 are
      // resident (the ring has >= 3 stages).
      auto shifted = [&](const uint4* q0, float& c, float& su, float& sq) {
        float2 as[H], aq[H];
#pragma unroll
        for (int h = 0; h < H; ++h) { as[h] = f2s(0.f); aq[h] = f2s(0.f); }
        c = 0.f;
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          const int ci = tid + j * nt;
          if (EXACT || ci < nchunks) {
            float2 t[H];
            P::unpack(q0[ci], t);
            if (j == 0) c = t[0].x;   // the thread's first element
            const float2 nc = f2s(-c);
#pragma unroll
            for (int h = 0; h < H; ++h) {
              const float2 d = fadd2(t[h], nc);
              as[h] = fadd2(as[h], d);
              aq[h] = ffma2(d, d, aq[h]);
            }
          }
        }
        const float2 t = tree_sum_2<H>(as, aq);
        su = t.x;
        sq = t.y;
      };
      // this thread's (shift, mean offset S/n, M2) of a row from its sums
      auto local = [&](float c, float su, float sq) {
        const float so = fmul(su, ln_inv_nt);
        ln_c = c;
        ln_off = so;
        ln_m2 = fmaxf(ffma(-su, so, sq), 0.f);
      };
      if (k == 0) {
        float c0, su0, sq0;
        shifted(r0, c0, su0, sq0);
        float a[1] = {ffma(ln_nt, c0, su0)};
        row_sum(a, bank, fl ^ 1);
        after_first_barrier();
        mu_next = div_n(a[0], inv_n);
        local(c0, su0, sq0);
      }
      mean = mu_next;
      float c1 = 0.f, su1 = 0.f, sq1 = 0.f;
      if (k + 1 < nrows) {
        const int s1 = (s + 1 == S) ? 0 : s + 1;
        const uint32_t ph1 = (s + 1 == S) ? (phase ^ 1u) : phase;
        if (!mbar_wait_bounded(&bars[s1], ph1)) {
          atomicOr(p.status, STATUS_WAIT_TIMEOUT);
          abort_flag[fl] = 1;
        }
        shifted(reinterpret_cast<const uint4*>(stages + (size_t)s1 * stage_bytes), c1, su1, sq1);
      }
      const float dt = fadd(fsub(ln_c, mean), ln_off);
      float a2[2] = {ffma(fmul(ln_nt, dt), dt, ln_m2), ffma(ln_nt, c1, su1)};
      row_sum(a2, bank, fl ^ 1);
      after_first_barrier();
      rstd = inv_rms(div_n(a2[0], inv_n), p.eps);
      mu_next = div_n(a2[1], inv_n);
      local(c1, su1, sq1);
      const float2 nmean = f2s(-mean);
      if (abort_flag[fl]) { aborted = true; break; }
      if (tid == 0 && crank == 0) {
        if (p.rstd_out) p.rstd_out[row] = rstd;
        if (p.mean_out) p.mean_out[row] = mean;
      }
      const float2 rs2 = f2s(rstd);
      T* yrow = static_cast<T*>(p.out0) + row * p.s_out0;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (EXACT || c < nchunks) {
          float2 t[H], w[H], bb[H], yf[H];
          P::unpack(r0[c], t);
          colv(j, c, 0, w);
          colv(j, c, 1, bb);
#pragma unroll
          for (int h = 0; h < H; ++h) yf[h] = ffma2(fmul2(fadd2(t[h], nmean), rs2), w[h], bb[h]);
          st_global_cs16(yrow + (int64_t)(col0 + c) * VEC, P::pack(yf));
        }
      }
    } else if constexpr (!BWD) {
      // ---- forward: the row (x, or h = x + residual) in FP32 -------------
      // row value of chunk c: x, or h = x + residual (FP32, exact for 16-bit
      // inputs); kept in registers (xf) or re-read from the stage
      auto rowv = [&](int c, float2 (&o)[H]) {
        P::unpack(r0[c], o);
        if constexpr (OP == FADD_FWD) {
          float2 rf[H];
          P::unpack(r1[c], rf);
#pragma unroll
          for (int h = 0; h < H; ++h) o[h] = fadd2(o[h], rf[h]);
        }
      };
      float2 xf[NX][H];
      float2 acc[H];
#pragma unroll
      for (int h = 0; h < H; ++h) acc[h] = f2s(0.f);
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (EXACT || c < nchunks) {
          float2 t[H];
          rowv(c, t);
          if constexpr (OP == FADD_FWD) {
            // the residual stream passed on: h rounded once to T
            st_global_cs16(static_cast<T*>(p.out1) + row * p.s_out1 + (int64_t)(col0 + c) * VEC, P::pack(t));
          }
#pragma unroll
          for (int h = 0; h < H; ++h) {
            if constexpr (KEEP) xf[j][h] = t[h];
            acc[h] = ffma2(t[h], t[h], acc[h]);
          }
        } else if constexpr (KEEP) {
#pragma unroll
          for (int h = 0; h < H; ++h) xf[j][h] = f2s(0.f);
        }
      }
      float a[1] = {tree_sum<H>(acc)};
      row_sum(a, bank, fl ^ 1);
      after_first_barrier();
      rstd = inv_rms(div_n(a[0], inv_n), p.eps);
      if (abort_flag[fl]) { aborted = true; break; }
      if (tid == 0 && crank == 0 && p.rstd_out) p.rstd_out[row] = rstd;
      const float2 rs2 = f2s(rstd);
      T* yrow = static_cast<T*>(p.out0) + row * p.s_out0;
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int c = tid + j * nt;
        if (EXACT || c < nchunks) {
          float2 t[H], w[H], yf[H];
          if constexpr (KEEP) {
#pragma unroll
            for (int h = 0; h < H; ++h) t[h] = xf[j][h];
          } else {
            rowv(c, t);
          }
          colv(j, c, 0, w);
#pragma unroll
          for (int h = 0; h < H; ++h) yf[h] = fmul2(fmul2(t[h], rs2), w[h]);
          st_global_cs16(yrow + (int64_t)(col0 + c) * VEC, P::pack(yf));
        }
      }
    } else {
      // ---- backward -------------------------------------------------------
      if (!have_stats) {
        // statistics recomputed from the saved row (no saved statistics
        // given): the sum of squares for RMSNorm as in its forward; two
        // passes, mean then sum((x - mean)^2), for LayerNorm
        float2 acc[H];
#pragma unroll
        for (int h = 0; h < H; ++h) acc[h] = f2s(0.f);
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          const int c = tid + j * nt;
          if (EXACT || c < nchunks) {
            float2 xf[H];
            P::unpack(r0[c], xf);
#pragma unroll
            for (int h = 0; h < H; ++h) {
              if constexpr (LN) acc[h] = fadd2(acc[h], xf[h]);
              else              acc[h] = ffma2(xf[h], xf[h], acc[h]);
            }
          }
        }
        float a[1] = {tree_sum<H>(acc)};
        row_sum(a, bank, fl ^ 1);
        after_first_barrier();
        if constexpr (LN) {
          mean = div_n(a[0], inv_n);
          const float2 nmean = f2s(-mean);
#pragma unroll
          for (int h = 0; h < H; ++h) acc[h] = f2s(0.f);
#pragma unroll
          for (int j = 0; j < NPT; ++j) {
            const int c = tid + j * nt;
            if (EXACT || c < nchunks) {
              float2 xf[H];
              P::unpack(r0[c], xf);
#pragma unroll
              for (int h = 0; h < H; ++h) {
                const float2 d = fadd2(xf[h], nmean);
                acc[h] = ffma2(d, d, acc[h]);
              }
            }
          }
          float q[1] = {tree_sum<H>(acc)};
          row_sum(q, bank, fl ^ 1);
          rstd = inv_rms(div_n(q[0], inv_n), p.eps);
        } else {
          rstd = inv_rms(div_n(a[0], inv_n), p.eps);
        }
      }
      const float2 L = bwd_local(r0, mean);
      float a[NR];
      if constexpr (LN) { a[0] = L.x; a[NR - 1] = L.y; }
      else              { a[0] = L.y; }
      row_sum(a, bank, fl ^ 1);
      after_first_barrier();
      if (abort_flag[fl]) { aborted = true; break; }
      bwd_out(r0, row, rstd, mean, make_float2(a[0], a[NR - 1]));
    }
  }

  grid_launch_dependents();
  if (aborted) {
    // Drain of the copies still in flight into this CTA's shared memory
    // (rows k .. issued-1), all within one kWaitLimitNs from here; no
    // partial sums are written: dW / dB are not valid after a wait ran out
    // (the status word says so).
    if (tid == 0) {
      const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
      for (int kk = k; kk < issued; ++kk) {
        if (!mbar_wait_until(&bars[s], phase, deadline)) break;
        if (++s == S) { s = 0; phase ^= 1u; }
      }
    }
    // a CTA of a cluster leaves only with its peers (below)
    if constexpr (CL) cluster_barrier();
    return;
  }

  if constexpr (DW || DB) {
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int c = tid + j * nt;
      if (c < nchunks) {
        const int64_t off = (int64_t)row0 * N + (int64_t)(col0 + c) * VEC;
#pragma unroll
        for (int h = 0; h < H; h += 2) {
          if constexpr (DW)
            *reinterpret_cast<float4*>(p.ws_dw + off + 2 * h) =
                make_float4(dwa[j][h].x, dwa[j][h].y, dwa[j][h + 1].x, dwa[j][h + 1].y);
          if constexpr (DB)
            *reinterpret_cast<float4*>(p.ws_db + off + 2 * h) =
                make_float4(dba[j][h].x, dba[j][h].y, dba[j][h + 1].x, dba[j][h + 1].y);
        }
      }
    }
  }
  // No CTA of a cluster leaves while a peer may still store into its shared
  // memory: every CTA reaches a cluster barrier, whether it finished or
  // gave up.
  if constexpr (CL) cluster_barrier();
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
  __shared__ float red[2 * 32 * kMaxReduceValues];
  int bank = 0;
  const TW* wp = static_cast<const TW*>(p.w);
  const TW* bp = static_cast<const TW*>(p.b);
  const float inv_n = 1.0f / (float)N;
  grid_dependency_wait();
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
      mean = div_n(a[0], inv_n);
      float q[1] = {0.f};
      for (int j = tid; j < N; j += nt) {
        const float d = fsub(to_f(x[j]), mean);
        q[0] = ffma(d, d, q[0]);
      }
      block_sum<1>(q, red, bank);
      rstd = inv_rms(div_n(q[0], inv_n), p.eps);
    } else {
      float a[1] = {0.f};
      for (int j = tid; j < N; j += nt) {
        float h = to_f(x[j]);
        if constexpr (OP == FADD_FWD) h = fadd(h, to_f(i1[j]));
        a[0] = ffma(h, h, a[0]);
      }
      block_sum<1>(a, red, bank);
      rstd = inv_rms(div_n(a[0], inv_n), p.eps);
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
        if constexpr (OP == LN_FWD) yf = ffma(fmul(fsub(xf, mean), rstd), wj, bp ? to_f(bp[j]) : 0.f);
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
      const float mg = LN ? div_n(a[0], inv_n) : 0.f;
      const float mgx = div_n(a[NR - 1], inv_n);
      for (int j = tid; j < N; j += nt) {
        const float xf = to_f(x[j]);
        const float dyf = to_f(i1[j]);
        const float g = fmul(dyf, fadd(to_f(wp[j]), p.offset));
        float xh, dx;
        if constexpr (LN) {
          xh = fmul(fsub(xf, mean), rstd);
          dx = fmul(rstd, ffma(-xh, mgx, fsub(g, mg)));
        } else {
          xh = fmul(xf, rstd);
          dx = fmul(rstd, ffma(-xh, mgx, g));
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
  grid_launch_dependents();
}

// ===========================================================================
// Launch logic
// ===========================================================================

// Threads of a staged CTA owning NPT 16-byte chunks each (0 = too many).
inline int staged_threads(int nchunks, int npt) {
  int t = (nchunks + npt - 1) / npt;
  t = ((t + 31) / 32) * 32;
  if (t < 64) t = 64;
  return t <= 512 ? t : 0;
}

// Per-(kernel, device) facts, queried once: the kernel is allowed the
// device's full opt-in shared memory (minus its own static shared memory) as
// dynamic shared memory -- an upper bound only; occupancy follows the size
// actually launched -- and its register-spill (local memory) size is kept
// for the launch-shape choice.
struct KernelInfo {
  int max_dyn = -1;     // largest dynamic shared memory allowed, -1 = error
  int local_bytes = 0;  // local memory per thread (register spills)
  int max_threads = 0;  // largest block it can be launched with (its launch bounds)
};

inline KernelInfo kernel_info(const void* fn, const DevInfo& di) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, KernelInfo> done;
  std::lock_guard<std::mutex> g(mu);
  auto key = std::make_pair(fn, di.dev);
  auto it = done.find(key);
  if (it != done.end()) return it->second;
  KernelInfo ki;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, fn);
  if (e != cudaSuccess) { cuda_fail(e); return ki; }
  const int max_dyn = di.smem_optin - (int)attr.sharedSizeBytes;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
  if (e != cudaSuccess) { cuda_fail(e); return ki; }
  ki.max_dyn = max_dyn;
  ki.local_bytes = (int)attr.localSizeBytes;
  ki.max_threads = attr.maxThreadsPerBlock;
  done[key] = ki;
  return ki;
}

inline int allow_max_smem(const void* fn, const DevInfo& di) { return kernel_info(fn, di).max_dyn; }

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
  if (allow_max_smem(fn, di) < 0) return -1;
  int nb = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem);
  if (e != cudaSuccess) { cuda_fail(e); return -1; }
  std::lock_guard<std::mutex> g(mu);
  cache[key] = nb;
  return nb;
}

// Cached cluster occupancy: thread-block clusters of `ncl` CTAs of this
// kernel (block size, dynamic shared memory) resident on the device at once.
inline int cached_clusters(const void* fn, const DevInfo& di, int threads, size_t smem, int ncl) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, size_t, int>, int> cache;
  auto key = std::make_tuple(fn, di.dev, threads, smem, ncl);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ncl);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
  if (e != cudaSuccess) { cuda_fail(e); return -1; }
  std::lock_guard<std::mutex> g(mu);
  cache[key] = n;
  return n;
}

// One staged launch: `ncl` CTAs per row (a thread-block cluster when > 1),
// each over nchunks / ncl chunks.  *grid_out receives the number of row
// groups (CTAs without clusters, clusters with them) = the partial rows
// written when dW / dB are computed.
template <int OP, class T, class TW, int NPT, bool DW, bool DB, bool EXACT, bool CL>
int launch_staged(const RowParams& p, const DevInfo& di, int nin, int max_ctas, int ncl, cudaStream_t st,
                  int* grid_out) {
  if (CL != (ncl > 1)) return NORM_ERR_UNSUPPORTED_INTERNAL;
  constexpr int VEC = 16 / (int)sizeof(T);
  if ((p.N / VEC) % ncl) return NORM_ERR_UNSUPPORTED_INTERNAL;
  const int nchunks = p.N / VEC / ncl;   // per CTA
  const int NL = nchunks * VEC;
  const int threads = staged_threads(nchunks, NPT);
  if (threads == 0) return NORM_ERR_UNSUPPORTED_INTERNAL;
  if (EXACT && threads * NPT != nchunks) return NORM_ERR_UNSUPPORTED_INTERNAL;
  const size_t stage_bytes = (size_t)nin * NL * sizeof(T);
  auto fn = staged_kernel<OP, T, TW, NPT, DW, DB, EXACT, CL>;
  const void* fp = reinterpret_cast<const void*>(fn);
  const size_t fixed = kStagedHeader + staged_col_bytes<OP>(NL, staged_wreg(NPT));
  const int min_stages = (OP == LN_FWD) ? 3 : 2;   // the LayerNorm forward holds rows k and k+1
  const size_t min_smem = fixed + (size_t)min_stages * stage_bytes;
  const KernelInfo ki = kernel_info(fp, di);
  const int max_dyn = ki.max_dyn;
  if (max_dyn < 0) return NORM_ERR_CUDA;
  if (threads > ki.max_threads) return NORM_ERR_UNSUPPORTED_INTERNAL;
  if (min_smem > (size_t)max_dyn) return NORM_ERR_UNSUPPORTED_INTERNAL;
  // Registers (and the 2-stage minimum) bound the CTAs per SM; shared memory
  // is then split evenly among them, as many stages as fit (<= kMaxStages).
  int nb = cached_occupancy(fp, di, threads, min_smem);
  if (nb < 0) return NORM_ERR_CUDA;
  if (nb == 0) return NORM_ERR_UNSUPPORTED_INTERNAL;
  int ctas = nb < max_ctas ? nb : max_ctas;
  if (DW || DB) {
    // no more row groups per SM than the workspace has partial rows for
    const int64_t per_sm = (di.max_partial_rows * ncl + di.sms - 1) / di.sms;
    if (per_sm >= 1 && ctas > per_sm) ctas = (int)per_sm;
  }
  int S = 0;
  size_t smem = 0;
  for (; ctas >= 1; --ctas) {
    size_t per_cta = (size_t)di.smem_per_sm / ctas;
    per_cta = per_cta > (size_t)di.smem_reserved + 64 ? per_cta - di.smem_reserved - 64 : 0;
    if (per_cta > (size_t)max_dyn) per_cta = (size_t)max_dyn;
    if (per_cta < min_smem) continue;
    S = (int)((per_cta - fixed) / stage_bytes);
    if (S > kMaxStages) S = kMaxStages;
    // Rows in flight: the S-1 stages ahead of the one being reduced, in
    // every resident CTA.  Past about 128 KB per SM more of them only slows
    // the stream down (measured on 8192-wide bf16 rows), so the ring stops
    // there even where shared memory would hold more.
    const size_t inflight = (size_t)(di.tune_inflight_16k > 0 ? di.tune_inflight_16k : kInflightUnits) * 16384;
    const int s_cap = 1 + (int)(inflight / ((size_t)ctas * stage_bytes));
    if (S > s_cap) S = s_cap > min_stages ? s_cap : min_stages;
    if ((OP == LN_FWD || OP == LN_BWD) && S > kLnMaxStages) S = kLnMaxStages;
    if (di.tune_max_stages >= 2 && S > di.tune_max_stages)
      S = di.tune_max_stages > min_stages ? di.tune_max_stages : min_stages;
    // confirm `ctas` CTAs of this size are resident together
    for (; S >= min_stages; --S) {
      smem = fixed + (size_t)S * stage_bytes;
      const int fit = cached_occupancy(fp, di, threads, smem);
      if (fit < 0) return NORM_ERR_CUDA;
      if (fit >= ctas) break;
    }
    if (S >= min_stages) break;
  }
  if (ctas < 1 || S < min_stages) return NORM_ERR_UNSUPPORTED_INTERNAL;
  // row groups: one per resident CTA, or one per resident cluster
  int64_t G = (int64_t)di.sms * ctas;
  if (ncl > 1) {
    const int nc = cached_clusters(fp, di, threads, smem, ncl);
    if (nc < 0) return NORM_ERR_CUDA;
    if (nc == 0) return NORM_ERR_UNSUPPORTED_INTERNAL;
    G = nc;
  }
  if (G > p.M) G = p.M;
  if ((DW || DB) && G > di.max_partial_rows) G = di.max_partial_rows;
  // the kernel counts a row group's rows in 32 bits
  if ((p.M + G - 1) / G > (int64_t)INT32_MAX) return NORM_ERR_UNSUPPORTED_INTERNAL;
  if (launch_pdl_cluster(fn, dim3((unsigned)(G * ncl)), dim3(threads), smem, ncl, st, p, S) != NORM_OK)
    return NORM_ERR_CUDA;
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
  if (launch_pdl(fn, dim3((unsigned)G), dim3(threads), 0, st, p) != NORM_OK) return NORM_ERR_CUDA;
  *grid_out = (int)G;
  return NORM_OK;
}

constexpr int kMaxStagedSpillBytes = 64;
constexpr int kTinySpillBytes = 32;   // a spill this small counts as none

// How well one staged instantiation suits a shape: fits at all, spills
// registers, CTAs resident per SM (at the two-stage minimum), block size.
struct StagedFit {
  bool ok = false;
  bool spills = false;
  int ctas = 0;
  int threads = 0;
};

template <int OP, class T, class TW, int NPT, bool DW, bool DB, bool EXACT, bool CL>
StagedFit probe_staged(const RowParams& p, const DevInfo& di, int nin, int ncl) {
  constexpr int VEC = 16 / (int)sizeof(T);
  StagedFit f;
  const int nchunks = p.N / VEC / ncl;
  f.threads = staged_threads(nchunks, NPT);
  if (f.threads == 0) return f;
  const void* fp = reinterpret_cast<const void*>(staged_kernel<OP, T, TW, NPT, DW, DB, EXACT, CL>);
  const KernelInfo ki = kernel_info(fp, di);
  if (f.threads > ki.max_threads) return f;   // beyond the instantiation's launch bounds
  const size_t min_smem = kStagedHeader + staged_col_bytes<OP>(nchunks * VEC, staged_wreg(NPT)) +
                          (OP == LN_FWD ? 3 : 2) * (size_t)nin * nchunks * 16;
  if (ki.max_dyn < 0 || min_smem > (size_t)ki.max_dyn) return f;
  const int nb = cached_occupancy(fp, di, f.threads, min_smem);
  if (nb <= 0) return f;
  // a shape that spills more than a few registers loses to the general kernel
  if (ki.local_bytes > kMaxStagedSpillBytes) return f;
  f.ok = true;
  f.spills = ki.local_bytes > kTinySpillBytes;
  f.ctas = nb;
  return f;
}

// Row kernel for one (op, types, flags): the staged path when every streamed
// row starts on a 16-byte boundary and fits, else the loop path.  Among the
// staged shapes (1, 2, 4 or 8 chunks per thread) the choice prefers, in
// order: no register spills (a few bytes aside), at least two resident CTAs
// per SM (so one CTA's barrier overlaps another's work), at least 3/4 of the
// threads holding a chunk, every thread holding exactly its chunks (no idle
// threads in the last warp: at N = 1536 and 2560 bf16 the exact 2-chunk
// shape was up to 12 % faster than 4 chunks with a part-idle warp), and then
// 4, 2, 8, 1 chunks per thread: four
// independent chunks give each thread the most memory-level parallelism
// while W' still fits in registers (measured fastest at N = 4096 and 8192
// wherever it does not spill).
template <int OP, class T, class TW, bool DW, bool DB>
int launch_rows(const RowParams& p, const DevInfo& di, bool rows_aligned, cudaStream_t st, int* grid_out) {
  constexpr int VEC = 16 / (int)sizeof(T);
  const int nin = (OP == FADD_BWD && p.in2 == nullptr) ? 2 : OpInfo<OP>::NIN;
  // A trainable backward is further held to the partial rows its workspace
  // has (launch_staged); occupancy bounds both.
  int max_ctas = 8;
  if (di.tune_max_ctas > 0) max_ctas = di.tune_max_ctas;
  if (rows_aligned && p.N % VEC == 0 && di.force_path != 2) {
    // A backward picks its shape from the instantiation with every weight
    // gradient on, whatever it computes itself: the block size (and the
    // cluster split) fix the reduction tree, so frozen and trainable calls
    // give bit-identical dx.
    constexpr bool PDW = OpInfo<OP>::BWD;
    constexpr bool PDB = (OP == LN_BWD);
    const int nchunks_row = p.N / VEC;
    const int npts[4] = {1, 2, 4, 8};
    const int rank[4] = {1, 3, 4, 2};   // preference among chunks per thread
    // The best staged shape with `ncl` CTAs per row: index into npts (-1 if
    // none fits), whether its threads own exactly the CTA's chunks, and
    // whether it spills.  One CTA per row runs the plain instantiations
    // (exact or not); a cluster split only exact shapes of 2, 4 or 8 chunks
    // per thread.
    struct Pick { int best = -1; bool exact = false; bool spills = true; };
    auto pick = [&](int ncl) {
      Pick r;
      if (nchunks_row % ncl) return r;
      const int nchunks = nchunks_row / ncl;   // per CTA
      bool exact[4];
      StagedFit fits[4];
      for (int i = 0; i < 4; ++i) {
        const int t = staged_threads(nchunks, npts[i]);
        exact[i] = t > 0 && t * npts[i] == nchunks;
      }
      if (ncl == 1) {
#define GB300NORM_PROBE(i, n)                                                              \
  fits[i] = exact[i] ? probe_staged<OP, T, TW, n, PDW, PDB, true, false>(p, di, nin, 1)    \
                     : probe_staged<OP, T, TW, n, PDW, PDB, false, false>(p, di, nin, 1)
        GB300NORM_PROBE(0, 1); GB300NORM_PROBE(1, 2); GB300NORM_PROBE(2, 4); GB300NORM_PROBE(3, 8);
#undef GB300NORM_PROBE
      } else {
        if (exact[1]) fits[1] = probe_staged<OP, T, TW, 2, PDW, PDB, true, true>(p, di, nin, ncl);
        if (exact[2]) fits[2] = probe_staged<OP, T, TW, 4, PDW, PDB, true, true>(p, di, nin, ncl);
        if (exact[3]) fits[3] = probe_staged<OP, T, TW, 8, PDW, PDB, true, true>(p, di, nin, ncl);
      }
      long best_score = -1;
      for (int i = 0; i < 4; ++i) {
        if (!fits[i].ok) continue;
        if (di.tune_npt && npts[i] != di.tune_npt) continue;
        // the LayerNorm backward's wide-state shape (StagedBounds) needs 128
        // threads, or 64-127 threads that each hold exactly 4 chunks: at
        // N = 2048 (64 threads, exact) it was 5-12 % faster than 2 chunks per
        // thread from 8192 rows up and level below; with idle threads in its
        // last warp (N = 1536, 2560) or one warp (N = 1024) it was 8-24 %
        // slower
        if (!di.tune_npt && OP == LN_BWD && npts[i] == 4 &&
            (fits[i].threads < 64 || (fits[i].threads < 128 && !exact[i])))
          continue;
        const bool busy = 4L * nchunks >= 3L * fits[i].threads * npts[i];
        const long score = (fits[i].spills ? 0 : 1000000L) + (fits[i].ctas >= 2 ? 100000L : 0) +
                           (busy ? 10000L : 0) + (exact[i] ? 1000L : 0) + rank[i];
        if (score > best_score) { best_score = score; r.best = i; }
      }
      if (r.best >= 0) { r.exact = exact[r.best]; r.spills = fits[r.best].spills; }
      return r;
    };
    // One CTA per row where a shape fits without spilling; otherwise the
    // smallest cluster split (2, 4, 8) that does.  Splitting is measured
    // slower wherever one CTA fits: a cluster launch, its exchanges and its
    // barriers cost about 2 us, and more rows per SM in flight beat the
    // split even for a few rows.
    int ncl = 1;
    Pick pk;
    if (di.tune_cluster > 0) {
      ncl = di.tune_cluster;
      pk = pick(ncl);
    } else {
      pk = pick(1);
      for (int c = 2; c <= 8 && (pk.best < 0 || pk.spills); c *= 2) {
        const Pick q = pick(c);
        if (q.best >= 0 && !q.spills) { ncl = c; pk = q; }
      }
    }
    int rc = NORM_ERR_UNSUPPORTED_INTERNAL;
    const int npt = pk.best < 0 ? 0 : npts[pk.best];
    if (ncl == 1) {
#define GB300NORM_STAGED(n)                                                                               \
  rc = pk.exact ? launch_staged<OP, T, TW, n, DW, DB, true, false>(p, di, nin, max_ctas, 1, st, grid_out)  \
                : launch_staged<OP, T, TW, n, DW, DB, false, false>(p, di, nin, max_ctas, 1, st, grid_out)
      switch (npt) {
        case 1: GB300NORM_STAGED(1); break;
        case 2: GB300NORM_STAGED(2); break;
        case 4: GB300NORM_STAGED(4); break;
        case 8: GB300NORM_STAGED(8); break;
        default: break;
      }
#undef GB300NORM_STAGED
    } else {
      switch (npt) {
        case 2: rc = launch_staged<OP, T, TW, 2, DW, DB, true, true>(p, di, nin, max_ctas, ncl, st, grid_out); break;
        case 4: rc = launch_staged<OP, T, TW, 4, DW, DB, true, true>(p, di, nin, max_ctas, ncl, st, grid_out); break;
        case 8: rc = launch_staged<OP, T, TW, 8, DW, DB, true, true>(p, di, nin, max_ctas, ncl, st, grid_out); break;
        default: break;
      }
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
