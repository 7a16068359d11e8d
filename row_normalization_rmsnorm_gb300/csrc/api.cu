// api.cu -- the C ABI declared in include/gb300norm.h: argument validation,
// device queries, workspace layout and the launch of the row kernels plus
// the dW / dB column reduction.  No call allocates memory or synchronises
// the host (norm_device_status excepted, which is a diagnostic).
#include <atomic>
#include <cmath>
#include <mutex>

#include "launch.h"

using namespace gb300norm;

// Device status word: bounded waits that ran out set bits here.
__device__ int g_norm_status;

thread_local int t_last_cuda_error = 0;

namespace gb300norm {
std::atomic<long long> g_launches{0};   // kernels launched (norm_debug_launches)
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return NORM_ERR_CUDA;
}
}  // namespace gb300norm

namespace {

std::atomic<int> g_force_path{0};
std::atomic<int> g_tune[7] = {{0}, {0}, {0}, {0}, {0}, {0}, {0}};

int elem_size(int dt) {
  switch (dt) {
    case NORM_F32: return 4;
    case NORM_F16: return 2;
    case NORM_BF16: return 2;
    default: return 0;
  }
}

bool types_ok(int dt, int wdt) {
  return (dt == NORM_F32 && wdt == NORM_F32) || (dt == NORM_F16 && wdt == NORM_F16) ||
         (dt == NORM_BF16 && wdt == NORM_BF16) || (dt == NORM_BF16 && wdt == NORM_F32) ||
         (dt == NORM_F16 && wdt == NORM_F32);
}

// Per-device facts, queried once per device.
struct DevCache {
  std::mutex mu;
  bool ready[64] = {};
  DevInfo info[64];
  int* status[64] = {};
};
DevCache g_dev;

int get_device(DevInfo* out, int** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return cuda_fail(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> g(g_dev.mu);
  if (!g_dev.ready[dev]) {
    DevInfo di;
    di.dev = dev;
    if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
      return cuda_fail(e);
    void* st = nullptr;
    if ((e = cudaGetSymbolAddress(&st, g_norm_status)) != cudaSuccess) return cuda_fail(e);
    g_dev.info[dev] = di;
    g_dev.status[dev] = static_cast<int*>(st);
    g_dev.ready[dev] = true;
  }
  *out = g_dev.info[dev];
  out->force_path = g_force_path.load();
  out->tune_npt = g_tune[1].load();
  out->tune_max_ctas = g_tune[2].load();
  out->tune_max_stages = g_tune[3].load();
  out->tune_inflight_16k = g_tune[4].load();
  out->tune_cluster = g_tune[5].load();
  if (status) *status = g_dev.status[dev];
  return NORM_OK;
}

// ---------------------------------------------------------------------------
// Argument checks
// ---------------------------------------------------------------------------
bool finite(float v) { return std::isfinite(v); }

// A 2-D row tensor argument.
struct Mat {
  const void* p;
  int64_t stride;
};

int check_mat(const Mat& m, int64_t M, int64_t N, int es, bool required) {
  if (M == 0) return NORM_OK;
  if (!m.p) return required ? NORM_ERR_NULL : NORM_OK;
  if (m.stride < N) return NORM_ERR_STRIDE;
  // the byte extent ((M - 1) * stride + N) * es must fit in 63 bits (it is
  // formed on the host for the overlap checks and in the kernels' row offsets)
  if (M - 1 > (INT64_MAX / es - N) / m.stride) return NORM_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(m.p) % (uintptr_t)es) return NORM_ERR_ALIGN;
  return NORM_OK;
}

bool row16(const Mat& m, int64_t M, int es) {
  if (!m.p) return true;
  if (reinterpret_cast<uintptr_t>(m.p) % 16) return false;
  return M <= 1 || (m.stride * es) % 16 == 0;
}

// A byte range touched by a call, for overlap checks.
struct Span {
  uintptr_t lo = 0, hi = 0;   // [lo, hi)
  const void* p = nullptr;
  int64_t stride = 0;
  bool out = false;
  unsigned tag = 0;            // outputs may coincide exactly with inputs sharing a tag bit
};

Span mat_span(const Mat& m, int64_t M, int64_t N, int es, bool out, unsigned tag) {
  Span s;
  if (!m.p || M == 0) return s;
  s.p = m.p;
  s.stride = m.stride;
  s.lo = reinterpret_cast<uintptr_t>(m.p);
  s.hi = s.lo + (uintptr_t)(((M - 1) * m.stride + N) * es);
  s.out = out;
  s.tag = tag;
  return s;
}

Span vec_span(const void* p, int64_t n, int es, bool out) {
  Span s;
  if (!p || n == 0) return s;
  s.p = p;
  s.lo = reinterpret_cast<uintptr_t>(p);
  s.hi = s.lo + (uintptr_t)(n * es);
  s.out = out;
  return s;
}

int check_overlaps(const Span* s, int n) {
  for (int i = 0; i < n; ++i) {
    if (!s[i].out || s[i].lo == s[i].hi) continue;
    for (int j = 0; j < n; ++j) {
      if (i == j || s[j].lo == s[j].hi) continue;
      if (s[i].lo >= s[j].hi || s[j].lo >= s[i].hi) continue;
      const bool exact = !s[j].out && (s[i].tag & s[j].tag) && s[i].p == s[j].p && s[i].stride == s[j].stride;
      if (!exact) return NORM_ERR_ALIAS;
    }
  }
  return NORM_OK;
}

int check_common(int64_t M, int64_t N, float offset, float eps, int dtype, int w_dtype, const void* w) {
  if (M < 0 || N <= 0 || N > INT32_MAX) return NORM_ERR_SHAPE;
  if (!types_ok(dtype, w_dtype)) return NORM_ERR_DTYPE;
  if (!finite(offset) || !finite(eps) || eps < 0.f) return NORM_ERR_VALUE;
  if (!w) return NORM_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(w) % (uintptr_t)elem_size(w_dtype)) return NORM_ERR_ALIGN;
  return NORM_OK;
}

int check_vec_f32(const void* p) {
  return (p && reinterpret_cast<uintptr_t>(p) % 4) ? NORM_ERR_ALIGN : NORM_OK;
}

int64_t ws_bytes_needed(int64_t M, int64_t N, int sms, int nbuf) {
  return partial_rows(M, N, sms) * N * 4 * nbuf;
}

// The workspace pointer is checked before the device is queried for its size.
int check_workspace_ptr(const void* ws) {
  return (!ws || reinterpret_cast<uintptr_t>(ws) % 16) ? NORM_ERR_WORKSPACE : NORM_OK;
}

int check_workspace(const void* ws, size_t ws_bytes, int64_t need) {
  if (need == 0) return NORM_OK;
  if (!ws || reinterpret_cast<uintptr_t>(ws) % 16 || ws_bytes < (size_t)need) return NORM_ERR_WORKSPACE;
  return NORM_OK;
}

#define RETURN_IF(x)            \
  do {                          \
    int rc_ = (x);              \
    if (rc_ != NORM_OK) return rc_; \
  } while (0)

RowParams base_params(int64_t M, int64_t N, float offset, float eps, const void* w, int* status) {
  RowParams p{};
  p.M = M;
  p.N = (int)N;
  p.offset = offset;
  p.eps = eps;
  p.w = w;
  p.status = status;
  p.hold_last = g_tune[6].load();
  return p;
}

// Shared tail of the three backward calls: row kernel, then stage 2.
template <class F>
int run_bwd(RowParams& p, int64_t M, int64_t N, void* dw, void* db, int dw_dtype, void* ws, size_t ws_bytes,
            const DevInfo& di, cudaStream_t st, F&& launch_rows) {
  if (M == 0) return launch_colreduce(nullptr, dw, nullptr, db, 0, (int)N, dw_dtype, st);
  const int64_t rows = partial_rows(M, N, di.sms);
  float* wsf = static_cast<float*>(ws);
  p.ws_dw = dw ? wsf : nullptr;
  p.ws_db = db ? wsf + (dw ? rows * N : 0) : nullptr;
  int G = 0;
  RETURN_IF(launch_rows(p, &G));
  if (dw || db) RETURN_IF(launch_colreduce(p.ws_dw, dw, p.ws_db, db, G, (int)N, dw_dtype, st));
  return NORM_OK;
}

}  // namespace

extern "C" {

const char* norm_status_str(int status) {
  switch (status) {
    case NORM_OK: return "ok";
    case NORM_ERR_NULL: return "a required pointer is NULL";
    case NORM_ERR_SHAPE: return "bad shape (M < 0, N <= 0 or N too large)";
    case NORM_ERR_STRIDE: return "row stride smaller than N";
    case NORM_ERR_DTYPE: return "unsupported dtype combination";
    case NORM_ERR_WORKSPACE: return "workspace missing, too small or not 16-byte aligned";
    case NORM_ERR_ALIGN: return "pointer not aligned to its element size";
    case NORM_ERR_VALUE: return "eps must be finite and >= 0, offset finite";
    case NORM_ERR_ALIAS: return "an output overlaps another argument in a way that is not allowed";
    case NORM_ERR_CUDA: return "CUDA runtime error while querying the device or launching";
    case NORM_ERR_ARG: return "inconsistent optional arguments";
    case NORM_ERR_TOO_LARGE: return "problem too large for the library's fixed scratch (no-allocation entry point)";
    default: return "unknown status";
  }
}

int norm_version(void) { return 10000; }

int norm_last_cuda_error(void) { return t_last_cuda_error; }

const char* norm_cuda_error_string(int code) { return cudaGetErrorString(static_cast<cudaError_t>(code)); }

int norm_debug_set_path(int mode) {
  if (mode != 0 && mode != 2) return NORM_ERR_ARG;
  g_force_path.store(mode);
  return NORM_OK;
}

int64_t norm_debug_launches(int reset) {
  return reset ? (int64_t)gb300norm::g_launches.exchange(0) : (int64_t)gb300norm::g_launches.load();
}

int norm_debug_tune(int key, int value) {
  if (key < 1 || key > 6 || value < 0 || value > 64) return NORM_ERR_ARG;
  if (key == 5 && value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return NORM_ERR_ARG;
  if (key == 6 && value > 1) return NORM_ERR_ARG;
  g_tune[key].store(value);
  return NORM_OK;
}

int norm_bwd_workspace_bytes(int64_t M, int64_t N, int has_dw, int has_db, size_t* bytes) {
  if (!bytes) return NORM_ERR_NULL;
  if (M < 0 || N <= 0 || N > INT32_MAX) return NORM_ERR_SHAPE;
  const int nbuf = (has_dw ? 1 : 0) + (has_db ? 1 : 0);
  if (nbuf == 0 || M == 0) { *bytes = 0; return NORM_OK; }
  DevInfo di;
  RETURN_IF(get_device(&di, nullptr));
  *bytes = (size_t)ws_bytes_needed(M, N, di.sms, nbuf);
  return NORM_OK;
}

int norm_device_status(int reset, int* value) {
  if (!value) return NORM_ERR_NULL;
  DevInfo di;
  int* st = nullptr;
  RETURN_IF(get_device(&di, &st));
  cudaError_t e;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemcpy(value, st, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  if (reset && (e = cudaMemset(st, 0, sizeof(int))) != cudaSuccess) return cuda_fail(e);
  if (reset && (e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e);
  return NORM_OK;
}

// ---------------------------------------------------------------------------
// Sum over ranks of an M-sharded backward's dW / dB
// ---------------------------------------------------------------------------
int norm_sum_ranks(const float* parts, int64_t world, int64_t N, void* out, int out_dtype,
                   gb300norm_stream_t stream) {
  if (world < 1 || world > INT32_MAX || N <= 0 || N > INT32_MAX) return NORM_ERR_SHAPE;
  if (!parts || !out) return NORM_ERR_NULL;
  if (out_dtype != NORM_F32 && out_dtype != NORM_F16 && out_dtype != NORM_BF16) return NORM_ERR_DTYPE;
  if (reinterpret_cast<uintptr_t>(parts) % 4 || reinterpret_cast<uintptr_t>(out) % (uintptr_t)elem_size(out_dtype))
    return NORM_ERR_ALIGN;
  const Span sp[2] = {vec_span(parts, world * N, 4, false), vec_span(out, N, elem_size(out_dtype), true)};
  RETURN_IF(check_overlaps(sp, 2));
  return launch_rank_sum(parts, out, (int)world, (int)N, out_dtype, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Forward calls
// ---------------------------------------------------------------------------
int norm_rms_fwd(const void* x, int64_t x_stride, const void* w, void* y, int64_t y_stride, float* rstd, int64_t M,
                 int64_t N, float offset, float eps, int dtype, int w_dtype, gb300norm_stream_t stream) {
  RETURN_IF(check_common(M, N, offset, eps, dtype, w_dtype, w));
  const int es = elem_size(dtype), ews = elem_size(w_dtype);
  const Mat mx{x, x_stride}, my{y, y_stride};
  RETURN_IF(check_mat(mx, M, N, es, true));
  RETURN_IF(check_mat(my, M, N, es, true));
  RETURN_IF(check_vec_f32(rstd));
  const Span sp[] = {mat_span(mx, M, N, es, false, 1), mat_span(my, M, N, es, true, 1),
                     vec_span(w, N, ews, false), vec_span(rstd, M, 4, true)};
  RETURN_IF(check_overlaps(sp, 4));
  if (M == 0) return NORM_OK;
  DevInfo di;
  int* status = nullptr;
  RETURN_IF(get_device(&di, &status));
  RowParams p = base_params(M, N, offset, eps, w, status);
  p.in0 = x; p.s_in0 = x_stride;
  p.out0 = y; p.s_out0 = y_stride;
  p.rstd_out = rstd;
  const bool al = row16(mx, M, es) && row16(my, M, es);
  int G = 0;
  return launch_op_rms_fwd(p, dtype, w_dtype, di, al, reinterpret_cast<cudaStream_t>(stream), &G);
}

int norm_ln_fwd(const void* x, int64_t x_stride, const void* w, const void* b, void* y, int64_t y_stride,
                float* mean, float* rstd, int64_t M, int64_t N, float offset, float eps, int dtype, int w_dtype,
                gb300norm_stream_t stream) {
  RETURN_IF(check_common(M, N, offset, eps, dtype, w_dtype, w));
  const int es = elem_size(dtype), ews = elem_size(w_dtype);
  if (b && reinterpret_cast<uintptr_t>(b) % (uintptr_t)ews) return NORM_ERR_ALIGN;
  const Mat mx{x, x_stride}, my{y, y_stride};
  RETURN_IF(check_mat(mx, M, N, es, true));
  RETURN_IF(check_mat(my, M, N, es, true));
  RETURN_IF(check_vec_f32(rstd));
  RETURN_IF(check_vec_f32(mean));
  const Span sp[] = {mat_span(mx, M, N, es, false, 1), mat_span(my, M, N, es, true, 1),
                     vec_span(w, N, ews, false), vec_span(b, N, ews, false),
                     vec_span(mean, M, 4, true), vec_span(rstd, M, 4, true)};
  RETURN_IF(check_overlaps(sp, 6));
  if (M == 0) return NORM_OK;
  DevInfo di;
  int* status = nullptr;
  RETURN_IF(get_device(&di, &status));
  RowParams p = base_params(M, N, offset, eps, w, status);
  p.b = b;
  p.in0 = x; p.s_in0 = x_stride;
  p.out0 = y; p.s_out0 = y_stride;
  p.mean_out = mean;
  p.rstd_out = rstd;
  const bool al = row16(mx, M, es) && row16(my, M, es);
  int G = 0;
  return launch_op_ln_fwd(p, dtype, w_dtype, di, al, reinterpret_cast<cudaStream_t>(stream), &G);
}

int norm_fused_add_rms_fwd(const void* x, int64_t x_stride, const void* residual, int64_t residual_stride,
                           const void* w, void* y, int64_t y_stride, void* h_out, int64_t h_stride, float* rstd,
                           int64_t M, int64_t N, float offset, float eps, int dtype, int w_dtype,
                           gb300norm_stream_t stream) {
  RETURN_IF(check_common(M, N, offset, eps, dtype, w_dtype, w));
  const int es = elem_size(dtype), ews = elem_size(w_dtype);
  const Mat mx{x, x_stride}, mr{residual, residual_stride}, my{y, y_stride}, mh{h_out, h_stride};
  RETURN_IF(check_mat(mx, M, N, es, true));
  RETURN_IF(check_mat(mr, M, N, es, true));
  RETURN_IF(check_mat(my, M, N, es, true));
  RETURN_IF(check_mat(mh, M, N, es, true));
  RETURN_IF(check_vec_f32(rstd));
  const Span sp[] = {mat_span(mx, M, N, es, false, 1), mat_span(mr, M, N, es, false, 1),
                     mat_span(my, M, N, es, true, 1), mat_span(mh, M, N, es, true, 1),
                     vec_span(w, N, ews, false), vec_span(rstd, M, 4, true)};
  RETURN_IF(check_overlaps(sp, 6));
  if (M == 0) return NORM_OK;
  DevInfo di;
  int* status = nullptr;
  RETURN_IF(get_device(&di, &status));
  RowParams p = base_params(M, N, offset, eps, w, status);
  p.in0 = x; p.s_in0 = x_stride;
  p.in1 = residual; p.s_in1 = residual_stride;
  p.out0 = y; p.s_out0 = y_stride;
  p.out1 = h_out; p.s_out1 = h_stride;
  p.rstd_out = rstd;
  const bool al = row16(mx, M, es) && row16(mr, M, es) && row16(my, M, es) && row16(mh, M, es);
  int G = 0;
  return launch_op_fadd_fwd(p, dtype, w_dtype, di, al, reinterpret_cast<cudaStream_t>(stream), &G);
}

// ---------------------------------------------------------------------------
// Backward calls
// ---------------------------------------------------------------------------
int norm_rms_bwd(const void* dy, int64_t dy_stride, const void* x, int64_t x_stride, const void* w,
                 const float* rstd, void* dx, int64_t dx_stride, void* dw, int dw_dtype, void* workspace,
                 size_t workspace_bytes, int64_t M, int64_t N, float offset, float eps, int dtype, int w_dtype,
                 gb300norm_stream_t stream) {
  RETURN_IF(check_common(M, N, offset, eps, dtype, w_dtype, w));
  const int es = elem_size(dtype), ews = elem_size(w_dtype);
  if (dw && dw_dtype != NORM_F32 && dw_dtype != w_dtype) return NORM_ERR_DTYPE;
  const int dws = dw ? elem_size(dw_dtype) : 4;
  if (dw && reinterpret_cast<uintptr_t>(dw) % (uintptr_t)dws) return NORM_ERR_ALIGN;
  const Mat mdy{dy, dy_stride}, mx{x, x_stride}, mdx{dx, dx_stride};
  RETURN_IF(check_mat(mdy, M, N, es, true));
  RETURN_IF(check_mat(mx, M, N, es, true));
  RETURN_IF(check_mat(mdx, M, N, es, true));
  RETURN_IF(check_vec_f32(rstd));
  DevInfo di;
  int* status = nullptr;
  int64_t need = 0;
  if (dw && M > 0) {
    RETURN_IF(check_workspace_ptr(workspace));
    RETURN_IF(get_device(&di, &status));
    need = ws_bytes_needed(M, N, di.sms, 1);
  }
  RETURN_IF(check_workspace(workspace, workspace_bytes, need));
  const Span sp[] = {mat_span(mdy, M, N, es, false, 1), mat_span(mx, M, N, es, false, 0),
                     mat_span(mdx, M, N, es, true, 1), vec_span(w, N, ews, false),
                     vec_span(rstd, M, 4, false), vec_span(dw, N, dws, true),
                     vec_span(need ? workspace : nullptr, need, 1, true)};
  RETURN_IF(check_overlaps(sp, 7));
  if (!status) RETURN_IF(get_device(&di, &status));
  di.max_partial_rows = partial_rows(M, N, di.sms);
  RowParams p = base_params(M, N, offset, eps, w, status);
  p.in0 = x; p.s_in0 = x_stride;
  p.in1 = dy; p.s_in1 = dy_stride;
  p.out0 = dx; p.s_out0 = dx_stride;
  p.rstd_in = rstd;
  const bool al = row16(mx, M, es) && row16(mdy, M, es) && row16(mdx, M, es);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return run_bwd(p, M, N, dw, nullptr, dw_dtype, workspace, workspace_bytes, di, st, [&](RowParams& q, int* G) {
    return launch_op_rms_bwd(q, dtype, w_dtype, dw != nullptr, di, al, st, G);
  });
}

int norm_ln_bwd(const void* dy, int64_t dy_stride, const void* x, int64_t x_stride, const void* w,
                const float* mean, const float* rstd, void* dx, int64_t dx_stride, void* dw, void* db,
                int dw_dtype, void* workspace, size_t workspace_bytes, int64_t M, int64_t N, float offset, float eps,
                int dtype, int w_dtype, gb300norm_stream_t stream) {
  RETURN_IF(check_common(M, N, offset, eps, dtype, w_dtype, w));
  const int es = elem_size(dtype), ews = elem_size(w_dtype);
  if ((mean == nullptr) != (rstd == nullptr)) return NORM_ERR_ARG;
  if ((dw || db) && dw_dtype != NORM_F32 && dw_dtype != w_dtype) return NORM_ERR_DTYPE;
  const int dws = (dw || db) ? elem_size(dw_dtype) : 4;
  if (dw && reinterpret_cast<uintptr_t>(dw) % (uintptr_t)dws) return NORM_ERR_ALIGN;
  if (db && reinterpret_cast<uintptr_t>(db) % (uintptr_t)dws) return NORM_ERR_ALIGN;
  const Mat mdy{dy, dy_stride}, mx{x, x_stride}, mdx{dx, dx_stride};
  RETURN_IF(check_mat(mdy, M, N, es, true));
  RETURN_IF(check_mat(mx, M, N, es, true));
  RETURN_IF(check_mat(mdx, M, N, es, true));
  RETURN_IF(check_vec_f32(rstd));
  RETURN_IF(check_vec_f32(mean));
  DevInfo di;
  int* status = nullptr;
  int64_t need = 0;
  const int nbuf = (dw ? 1 : 0) + (db ? 1 : 0);
  if (nbuf && M > 0) {
    RETURN_IF(check_workspace_ptr(workspace));
    RETURN_IF(get_device(&di, &status));
    need = ws_bytes_needed(M, N, di.sms, nbuf);
  }
  RETURN_IF(check_workspace(workspace, workspace_bytes, need));
  const Span sp[] = {mat_span(mdy, M, N, es, false, 1), mat_span(mx, M, N, es, false, 0),
                     mat_span(mdx, M, N, es, true, 1), vec_span(w, N, ews, false),
                     vec_span(mean, M, 4, false), vec_span(rstd, M, 4, false),
                     vec_span(dw, N, dws, true), vec_span(db, N, dws, true),
                     vec_span(need ? workspace : nullptr, need, 1, true)};
  RETURN_IF(check_overlaps(sp, 9));
  if (!status) RETURN_IF(get_device(&di, &status));
  di.max_partial_rows = partial_rows(M, N, di.sms);
  RowParams p = base_params(M, N, offset, eps, w, status);
  p.in0 = x; p.s_in0 = x_stride;
  p.in1 = dy; p.s_in1 = dy_stride;
  p.out0 = dx; p.s_out0 = dx_stride;
  p.mean_in = mean;
  p.rstd_in = rstd;
  const bool al = row16(mx, M, es) && row16(mdy, M, es) && row16(mdx, M, es);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return run_bwd(p, M, N, dw, db, dw_dtype, workspace, workspace_bytes, di, st, [&](RowParams& q, int* G) {
    return launch_op_ln_bwd(q, dtype, w_dtype, dw != nullptr, db != nullptr, di, al, st, G);
  });
}

int norm_fused_add_rms_bwd(const void* dy, int64_t dy_stride, const void* dh_out, int64_t dh_stride, const void* h,
                           int64_t h_stride, const void* w, const float* rstd, void* dx, int64_t dx_stride, void* dw,
                           int dw_dtype, void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                           float offset, float eps, int dtype, int w_dtype, gb300norm_stream_t stream) {
  RETURN_IF(check_common(M, N, offset, eps, dtype, w_dtype, w));
  const int es = elem_size(dtype), ews = elem_size(w_dtype);
  if (dw && dw_dtype != NORM_F32 && dw_dtype != w_dtype) return NORM_ERR_DTYPE;
  const int dws = dw ? elem_size(dw_dtype) : 4;
  if (dw && reinterpret_cast<uintptr_t>(dw) % (uintptr_t)dws) return NORM_ERR_ALIGN;
  const Mat mdy{dy, dy_stride}, mdh{dh_out, dh_stride}, mh{h, h_stride}, mdx{dx, dx_stride};
  RETURN_IF(check_mat(mdy, M, N, es, true));
  RETURN_IF(check_mat(mdh, M, N, es, false));
  RETURN_IF(check_mat(mh, M, N, es, true));
  RETURN_IF(check_mat(mdx, M, N, es, true));
  RETURN_IF(check_vec_f32(rstd));
  DevInfo di;
  int* status = nullptr;
  int64_t need = 0;
  if (dw && M > 0) {
    RETURN_IF(check_workspace_ptr(workspace));
    RETURN_IF(get_device(&di, &status));
    need = ws_bytes_needed(M, N, di.sms, 1);
  }
  RETURN_IF(check_workspace(workspace, workspace_bytes, need));
  const Span sp[] = {mat_span(mdy, M, N, es, false, 1), mat_span(mdh, M, N, es, false, 1),
                     mat_span(mh, M, N, es, false, 0), mat_span(mdx, M, N, es, true, 1),
                     vec_span(w, N, ews, false), vec_span(rstd, M, 4, false),
                     vec_span(dw, N, dws, true), vec_span(need ? workspace : nullptr, need, 1, true)};
  RETURN_IF(check_overlaps(sp, 8));
  if (!status) RETURN_IF(get_device(&di, &status));
  di.max_partial_rows = partial_rows(M, N, di.sms);
  RowParams p = base_params(M, N, offset, eps, w, status);
  p.in0 = h; p.s_in0 = h_stride;
  p.in1 = dy; p.s_in1 = dy_stride;
  p.in2 = (M > 0) ? dh_out : nullptr; p.s_in2 = dh_stride;
  p.out0 = dx; p.s_out0 = dx_stride;
  p.rstd_in = rstd;
  const bool al = row16(mh, M, es) && row16(mdy, M, es) && row16(mdx, M, es) && row16(mdh, M, es);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return run_bwd(p, M, N, dw, nullptr, dw_dtype, workspace, workspace_bytes, di, st, [&](RowParams& q, int* G) {
    return launch_op_fadd_bwd(q, dtype, w_dtype, dw != nullptr, di, al, st, G);
  });
}

}  // extern "C"
