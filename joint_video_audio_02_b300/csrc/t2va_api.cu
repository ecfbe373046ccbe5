// C-ABI entry points of the joint video-audio distillation objective library.
// Argument checking, device queries and launch planning; the arithmetic lives
// in t2va_noise.cu, t2va_objective.cu and the W8A8 and fused normalisation files. Declarations and the contract of
// every entry point are in include/t2va.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "t2va_internal.cuh"
#include "t2va_w8a8.cuh"
#include "t2va_fused.cuh"

using namespace t2va;

namespace {

struct DeviceInfo {
  int sm_count = 0;
  size_t smem_optin = 0;
  size_t l2_bytes = 0;
  bool valid = false;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

bool current_device(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo& d = g_devices[dev];
  if (!d.valid) {
    int sms = 0, optin = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    d.sm_count = sms;
    d.smem_optin = (size_t)optin;
    d.l2_bytes = (size_t)l2;
    d.valid = sms > 0;
  }
  *out = d;
  return d.valid;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline bool finite(float x) { return std::isfinite(x); }

int check_geometry(int B, int M, const t2va_segment* seg) {
  if (B < 0 || M < 1 || M > kMaxM || seg == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  for (int m = 0; m < M; ++m) {
    const int64_t n = seg[m].numel, s = seg[m].sample_stride;
    if (n < 0 || s < 0) return T2VA_ERROR_INVALID_ARGUMENT;
    if (B > 1 && s < n) return T2VA_ERROR_INVALID_ARGUMENT;
    // every element offset must stay far from int64 overflow (x 8 bytes)
    const int64_t lim = INT64_MAX / 16;
    if (n > lim || (B > 1 && s > (lim - n) / (B - 1))) return T2VA_ERROR_INVALID_ARGUMENT;
  }
  return T2VA_SUCCESS;
}

int check_ptrs(int M, const t2va_segment* seg, const void* const* p) {
  if (p == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  for (int m = 0; m < M; ++m) {
    if (seg[m].numel > 0 && p[m] == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
    if (!aligned(p[m], 16)) return T2VA_ERROR_MISALIGNED;
  }
  return T2VA_SUCCESS;
}

int check_dtype(t2va_dtype dt) {
  return (dt == T2VA_FLOAT32 || dt == T2VA_BFLOAT16) ? T2VA_SUCCESS : T2VA_ERROR_UNSUPPORTED_DTYPE;
}

int check_weights(int M, const float* w) {
  if (w == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  for (int m = 0; m < M; ++m)
    if (!finite(w[m]) || w[m] < 0.f) return T2VA_ERROR_INVALID_ARGUMENT;
  return T2VA_SUCCESS;
}

int check_scalar_out(const void* p, bool required) {
  if (p == nullptr) return required ? T2VA_ERROR_INVALID_ARGUMENT : T2VA_SUCCESS;
  return aligned(p, 4) ? T2VA_SUCCESS : T2VA_ERROR_MISALIGNED;
}

#define T2VA_TRY(expr)              \
  do {                              \
    const int rc_ = (expr);         \
    if (rc_ != T2VA_SUCCESS) return rc_; \
  } while (0)

// The workspace as the objective sees it, from a caller's pointer and size: a null body
// when the pointer is null or misaligned or the size holds no header (the call then
// fails the workspace check after every argument check).
WsRef caller_workspace(void* workspace, size_t bytes) {
  WsRef w{nullptr, 0};
  if (workspace == nullptr || !aligned(workspace, 16) || bytes < kWsHeaderBytes) return w;
  w.body = reinterpret_cast<unsigned char*>(workspace) + kWsHeaderBytes;
  w.body_bytes = bytes - kWsHeaderBytes;
  return w;
}

// Shared tail of the objective entry points: the workspace check, the plan, the launch.
int run_objective(ObjectiveArgs& a, t2va_dtype dt, int mode, const WsRef& ws,
                  cudaStream_t stream) {
  DeviceInfo dev;
  if (!current_device(&dev)) return T2VA_ERROR_CUDA;
  if (ws.body == nullptr || ws.body_bytes < ws_body_bytes(a.B, a.M)) return T2VA_ERROR_WORKSPACE;
  a.partials = reinterpret_cast<float*>(ws.body);
  for (int m = 0; m < a.M; ++m) {
    const bool s_ok = a.grad_s[m] == nullptr || aligned(a.grad_s[m], 32);
    const bool d_ok = a.grad_d[m] == nullptr || aligned(a.grad_d[m], 32);
    // every full vector starts a multiple of 8 elements from the buffer's start (the
    // unaligned head of a sample is done element by element), so 32-byte aligned
    // buffers give 32-byte aligned 8-float gradient runs
    if (s_ok && d_ok) a.wide_mask |= 1u << m;
  }
  ObjectiveLaunch l;
  if (!plan_objective(a, dt, dev.sm_count, &l)) return T2VA_ERROR_INVALID_ARGUMENT;
  const cudaError_t e = launch_objective(a, dt, mode, l, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  return T2VA_SUCCESS;
}

void fill_geometry(ObjectiveArgs& a, int B, int M, const t2va_segment* seg) {
  std::memset(&a, 0, sizeof(a));
  a.B = B;
  a.M = M;
  for (int m = 0; m < M; ++m) {
    a.n[m] = seg[m].numel;
    a.stride[m] = seg[m].sample_stride;
  }
}

// Plan and launch one noising kernel writing `outputs` (NoiseOut bits). Pointers
// are checked by the caller.
int run_noise(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
              const void* const* z0, const void* const* eps, void* const* zt,
              void* const* zrf, const float* t, float* t_rf, int* status, int outputs,
              cudaStream_t stream) {
  NoiseArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = batch;
  a.M = num_modalities;
  a.t = t;
  a.t_rf = t_rf;
  a.status = status;
  const int VE = dtype == T2VA_BFLOAT16 ? 8 : 4;
  const int64_t per_cta = noise_vectors_per_cta();
  int64_t total = 0;
  for (int m = 0; m < num_modalities; ++m) {
    a.n[m] = seg[m].numel;
    a.stride[m] = seg[m].sample_stride;
    a.z0[m] = z0[m];
    a.eps[m] = eps[m];
    a.zt[m] = zt != nullptr ? zt[m] : nullptr;
    a.zrf[m] = zrf != nullptr ? zrf[m] : nullptr;
    // CTAs per (sample, modality); an empty modality gets no CTA at all
    const int64_t vec_ub = (seg[m].numel + VE - 1) / VE;
    const int64_t chunks = (vec_ub + per_cta - 1) / per_cta;
    if (chunks > INT32_MAX) return T2VA_ERROR_INVALID_ARGUMENT;
    a.chunks[m] = chunks > 0 ? (int)chunks : 1;
    a.block_off[m] = (int)total;
    total += (int64_t)batch * chunks;
    if (total > INT32_MAX) return T2VA_ERROR_INVALID_ARGUMENT;
  }
  for (int m = num_modalities; m <= kMaxM; ++m) {
    if (m < kMaxM) a.chunks[m] = 1;
    a.block_off[m] = (int)total;
  }
  // CTA b also writes t_rf[b], so a launch with t_rf has at least B CTAs
  const int64_t grid = (t_rf != nullptr && total < batch) ? batch : total;
  if (grid == 0) return T2VA_SUCCESS;
  if (launch_noise(a, dtype, outputs, (int)grid, stream) != cudaSuccess) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  return T2VA_SUCCESS;
}

}  // namespace

// The stage-3 entry points: without guidance (x0_teacher_hat_uncond and guidance
// null), x0_teacher_hat is the teacher prediction; with it, the conditional one.
int t2va::stage3_entry(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                       const void* const* z_t, const void* const* x0_teacher,
                       const void* const* x0_student, const void* const* x0_student_tangent,
                       const float* t, const void* const* zhat0,
                       const void* const* x0_teacher_hat,
                       const void* const* x0_teacher_hat_uncond, const float* guidance,
                       const void* const* x0_fake, float beta, float gamma, float eps_scm,
                       float eps_dmd, const float* weight, float lambda_scm, float lambda_dmd,
                       float* const* grad_x0_student, float* const* grad_zhat0, int accumulate,
                       float* loss, float* loss_scm, float* loss_dmd, float* norm, float* cdmd,
                       const WsRef& ws, int* status, cudaStream_t stream) {
  const int M = num_modalities;
  T2VA_TRY(check_geometry(batch, M, seg));
  T2VA_TRY(check_dtype(dtype));
  if (batch == 0) return T2VA_SUCCESS;
  for (const void* const* p : {z_t, x0_teacher, x0_student, x0_student_tangent, zhat0,
                               x0_teacher_hat, x0_fake})
    T2VA_TRY(check_ptrs(M, seg, p));
  const bool cfg = x0_teacher_hat_uncond != nullptr;
  if (cfg) {
    T2VA_TRY(check_ptrs(M, seg, x0_teacher_hat_uncond));
    if (guidance == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
    for (int m = 0; m < M; ++m)
      if (!finite(guidance[m])) return T2VA_ERROR_INVALID_ARGUMENT;
  }
  T2VA_TRY(check_ptrs(M, seg, reinterpret_cast<const void* const*>(grad_x0_student)));
  T2VA_TRY(check_ptrs(M, seg, reinterpret_cast<const void* const*>(grad_zhat0)));
  T2VA_TRY(check_scalar_out(t, true));
  T2VA_TRY(check_scalar_out(loss, true));
  for (const float* p : {loss_scm, loss_dmd, norm, cdmd}) T2VA_TRY(check_scalar_out(p, false));
  T2VA_TRY(check_scalar_out(status, true));
  T2VA_TRY(check_weights(M, weight));
  if (!finite(beta) || !(gamma >= 0.f && gamma <= 1.f) || !finite(eps_scm) || !(eps_scm > 0.f) ||
      !finite(lambda_scm) || !finite(eps_dmd) || !(eps_dmd > 0.f) || !finite(lambda_dmd))
    return T2VA_ERROR_INVALID_ARGUMENT;
  ObjectiveArgs a;
  fill_geometry(a, batch, M, seg);
  for (int m = 0; m < M; ++m) {
    a.in[kZt][m] = z_t[m];
    a.in[kXT][m] = x0_teacher[m];
    a.in[kXS][m] = x0_student[m];
    a.in[kXdot][m] = x0_student_tangent[m];
    a.in[kZh][m] = zhat0[m];
    a.in[kYT][m] = x0_teacher_hat[m];
    a.in[kYF][m] = x0_fake[m];
    if (cfg) {
      a.in[kYU][m] = x0_teacher_hat_uncond[m];
      a.cfg[m] = guidance[m];
    }
    a.grad_s[m] = grad_x0_student[m];
    a.grad_d[m] = grad_zhat0[m];
    if (grad_x0_student[m] == grad_zhat0[m]) a.alias_mask |= 1u << m;
    a.w[m] = weight[m];
  }
  a.t = t;
  a.beta = beta;
  a.gamma = gamma;
  a.eps_s = eps_scm;
  a.lam_s = lambda_scm;
  a.eps_d = eps_dmd;
  a.lam_d = lambda_dmd;
  a.accumulate = accumulate ? 1 : 0;
  a.loss = loss;
  a.loss_s = loss_scm;
  a.loss_d = loss_dmd;
  a.norm = norm;
  a.cdmd = cdmd;
  a.status = status;
  return run_objective(a, dtype, cfg ? (kModeStage3 | kModeCfg) : kModeStage3, ws, stream);
}

extern "C" {

const char* t2va_error_string(int code) {
  switch (code) {
    case T2VA_SUCCESS: return "success";
    case T2VA_ERROR_INVALID_ARGUMENT: return "invalid argument (size, scalar or null pointer)";
    case T2VA_ERROR_UNSUPPORTED_DTYPE: return "unsupported dtype (float32 and bfloat16 only)";
    case T2VA_ERROR_MISALIGNED: return "device pointer not 16-byte aligned (4-byte for scalars)";
    case T2VA_ERROR_WORKSPACE: return "workspace null, misaligned or smaller than t2va_workspace_bytes()";
    case T2VA_ERROR_CUDA: return "CUDA runtime error or kernel launch failure";
    default: return "unknown t2va error code";
  }
}

int t2va_abi_version(void) { return T2VA_ABI_VERSION; }

int t2va_objective_plan_query(int batch, int num_modalities, const t2va_segment* seg,
                              t2va_dtype dtype, int sm_count, t2va_objective_plan* out) {
  T2VA_TRY(check_geometry(batch, num_modalities, seg));
  T2VA_TRY(check_dtype(dtype));
  if (sm_count < 1 || out == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  ObjectiveArgs a;
  fill_geometry(a, batch, num_modalities, seg);
  ObjectiveLaunch l;
  if (!plan_objective(a, dtype, sm_count, &l)) return T2VA_ERROR_INVALID_ARGUMENT;
  std::memset(out, 0, sizeof(*out));
  out->grid = l.grid;
  out->threads = l.threads;
  out->vectors_per_chunk = a.vpc;
  for (int m = 0; m < num_modalities; ++m) out->chunks[m] = a.nchunk[m];
  out->outputs_modality = a.out_m;
  out->outputs_chunk = a.out_c;
  out->one_wave = (int64_t)l.grid <= 3 * (int64_t)sm_count ? 1 : 0;
  return T2VA_SUCCESS;
}

size_t t2va_workspace_bytes(int batch, int num_modalities) {
  if (batch < 0 || num_modalities < 1 || num_modalities > kMaxM) return 0;
  DeviceInfo dev;
  if (!current_device(&dev)) return 0;
  return ws_bytes(batch, num_modalities);
}

int t2va_quantize_rows(int64_t rows, int64_t cols, t2va_dtype dtype, const void* x, int64_t ld_x,
                       float eps, t2va_dtype code_dtype, void* q, int64_t ld_q, float* scale,
                       cudaStream_t stream) {
  T2VA_TRY(check_dtype(dtype));
  if (code_dtype != T2VA_INT8 && code_dtype != T2VA_BFLOAT16) return T2VA_ERROR_UNSUPPORTED_DTYPE;
  const int esz = dtype == T2VA_BFLOAT16 ? 2 : 4;
  if (rows < 0 || cols < 0 || rows > INT32_MAX || ld_x < cols || ld_q < cols || !finite(eps) ||
      !(eps > 0.f))
    return T2VA_ERROR_INVALID_ARGUMENT;
  if (rows == 0) return T2VA_SUCCESS;
  if (x == nullptr || q == nullptr || scale == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  // every input row is whole 16-byte vectors starting on a 16-byte boundary; the codes
  // of one vector (16 / element size of them) are stored together, so output rows start
  // on that boundary
  if (cols % (16 / esz) != 0 || (ld_x * esz) % 16 != 0 || ld_q % (16 / esz) != 0)
    return T2VA_ERROR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4)) return T2VA_ERROR_MISALIGNED;
  QuantArgs a;
  a.rows = rows;
  a.cols = cols;
  a.codes_bf16 = code_dtype == T2VA_BFLOAT16;
  a.x = x;
  a.ld_x = ld_x;
  a.q = q;
  a.ld_q = ld_q;
  a.scale = scale;
  a.eps = eps;
  if (launch_quantize_rows(a, dtype, stream) != cudaSuccess) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  return T2VA_SUCCESS;
}

int t2va_w8a8_linear(int64_t M, int64_t N, int64_t K, t2va_dtype code_dtype, const void* xq,
                     const float* sx, const void* wq, const float* sw, const float* bias,
                     t2va_dtype out_dtype, void* y, int* status, cudaStream_t stream) {
  T2VA_TRY(check_dtype(out_dtype));
  if (code_dtype != T2VA_INT8 && code_dtype != T2VA_BFLOAT16) return T2VA_ERROR_UNSUPPORTED_DTYPE;
  if (M < 0 || N < 0 || K < 0) return T2VA_ERROR_INVALID_ARGUMENT;
  if (M == 0 || N == 0) return T2VA_SUCCESS;
  // the guarded shapes: M, N, K multiples of 128; K small enough that no INT32 sum of
  // 127 x 127 products can overflow
  if (M % 128 != 0 || N % 128 != 0 || K % 128 != 0 || K == 0 || K > kW8a8MaxK ||
      M / gemm_tile_m() > 65535)
    return T2VA_ERROR_INVALID_ARGUMENT;
  if (xq == nullptr || sx == nullptr || wq == nullptr || sw == nullptr || y == nullptr)
    return T2VA_ERROR_INVALID_ARGUMENT;
  const bool tc = code_dtype == T2VA_BFLOAT16;
  if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(sx, 4) || !aligned(sw, 4) ||
      !aligned(bias, 4) || !aligned(y, tc ? 16 : 8) || !aligned(status, 4))
    return T2VA_ERROR_MISALIGNED;
  GemmArgs a = {};
  a.M = M;
  a.N = N;
  a.K = K;
  a.xq = reinterpret_cast<const int8_t*>(xq);
  a.sx = sx;
  a.wq = reinterpret_cast<const int8_t*>(wq);
  a.sw = sw;
  a.bias = bias;
  a.y = y;
  a.status = status;
  const cudaError_t e = tc ? launch_w8a8_tc(a, out_dtype == T2VA_BFLOAT16, stream)
                           : launch_w8a8_gemm(a, out_dtype == T2VA_BFLOAT16, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  return T2VA_SUCCESS;
}

int t2va_residual_modnorm(int64_t rows, int64_t D, int64_t rows_per_sample, t2va_dtype dtype,
                          const void* h, const void* u, const float* gate, const float* scale,
                          const float* shift, float eps, void* h_out, void* y, cudaStream_t stream) {
  T2VA_TRY(check_dtype(dtype));
  const int esz = dtype == T2VA_BFLOAT16 ? 2 : 4;
  if (rows < 0 || D < 0 || rows_per_sample < 1 || rows > (int64_t)INT32_MAX * 2 || !finite(eps) ||
      !(eps >= 0.f))
    return T2VA_ERROR_INVALID_ARGUMENT;
  if (rows == 0 || D == 0) return T2VA_SUCCESS;
  if (h == nullptr || y == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  // rows of whole 16-byte vectors; the per-sample vectors are read 4 floats at a time
  if (D % (16 / esz) != 0) return T2VA_ERROR_INVALID_ARGUMENT;
  // without a residual update there is no h' to store and no gate
  if (u == nullptr && (h_out != nullptr || gate != nullptr)) return T2VA_ERROR_INVALID_ARGUMENT;
  // y is written after its row is read: it may not be an input or h'
  if (y == h || y == u || (h_out != nullptr && (y == h_out || h_out == u))) return T2VA_ERROR_INVALID_ARGUMENT;
  for (const void* p : {h, u, static_cast<const void*>(h_out), static_cast<const void*>(y),
                        static_cast<const void*>(gate), static_cast<const void*>(scale),
                        static_cast<const void*>(shift)})
    if (!aligned(p, 16)) return T2VA_ERROR_MISALIGNED;
  FusedArgs a;
  a.rows = rows;
  a.D = D;
  a.rows_per_sample = rows_per_sample;
  a.h = h;
  a.u = u;
  a.gate = gate;
  a.scale = scale;
  a.shift = shift;
  a.eps = eps;
  a.h_out = h_out;
  a.y = y;
  if (launch_residual_modnorm(a, dtype, stream) != cudaSuccess) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  return T2VA_SUCCESS;
}

int t2va_selftest_wait_timeout(int* status, cudaStream_t stream) {
  if (status == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  if (!aligned(status, 4)) return T2VA_ERROR_MISALIGNED;
  if (launch_w8a8_tc_selftest(status, stream) != cudaSuccess) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  return T2VA_SUCCESS;
}

int t2va_workspace_init(void* workspace, size_t workspace_bytes, uint32_t /*timeout_ms*/,
                        cudaStream_t stream) {
  if (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < kWsHeaderBytes)
    return T2VA_ERROR_WORKSPACE;
  if (launch_workspace_init(workspace, workspace_bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  return T2VA_SUCCESS;
}

int t2va_noise(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
               const void* const* z0, const void* const* eps, void* const* zt,
               const float* t, int* status, cudaStream_t stream) {
  T2VA_TRY(check_geometry(batch, num_modalities, seg));
  T2VA_TRY(check_dtype(dtype));
  if (batch == 0) return T2VA_SUCCESS;
  T2VA_TRY(check_ptrs(num_modalities, seg, z0));
  T2VA_TRY(check_ptrs(num_modalities, seg, eps));
  T2VA_TRY(check_ptrs(num_modalities, seg, reinterpret_cast<const void* const*>(zt)));
  T2VA_TRY(check_scalar_out(t, true));
  T2VA_TRY(check_scalar_out(status, false));
  return run_noise(batch, num_modalities, seg, dtype, z0, eps, zt, nullptr, t, nullptr, status,
                   kNoiseZt, stream);
}

int t2va_noise_rf(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                  const void* const* z0, const void* const* eps, void* const* zt,
                  void* const* z_rf, const float* t, float* t_rf, int* status,
                  cudaStream_t stream) {
  T2VA_TRY(check_geometry(batch, num_modalities, seg));
  T2VA_TRY(check_dtype(dtype));
  if (batch == 0) return T2VA_SUCCESS;
  T2VA_TRY(check_ptrs(num_modalities, seg, z0));
  T2VA_TRY(check_ptrs(num_modalities, seg, eps));
  if (zt != nullptr)
    T2VA_TRY(check_ptrs(num_modalities, seg, reinterpret_cast<const void* const*>(zt)));
  T2VA_TRY(check_ptrs(num_modalities, seg, reinterpret_cast<const void* const*>(z_rf)));
  for (int m = 0; zt != nullptr && m < num_modalities; ++m)
    if (seg[m].numel > 0 && zt[m] == z_rf[m]) return T2VA_ERROR_INVALID_ARGUMENT;
  T2VA_TRY(check_scalar_out(t, true));
  T2VA_TRY(check_scalar_out(t_rf, false));
  T2VA_TRY(check_scalar_out(status, false));
  return run_noise(batch, num_modalities, seg, dtype, z0, eps, zt, z_rf, t, t_rf, status,
                   zt != nullptr ? (kNoiseZt | kNoiseRf) : kNoiseRf, stream);
}

int t2va_scm_objective(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                       const void* const* z_t, const void* const* x0_teacher,
                       const void* const* x0_student, const void* const* x0_student_tangent,
                       const float* t, float beta, float gamma, float eps_scm,
                       const float* weight, float lambda_scm,
                       float* const* grad_x0_student, int accumulate,
                       float* loss, float* norm,
                       void* workspace, size_t workspace_bytes, int* status,
                       cudaStream_t stream) {
  const int M = num_modalities;
  T2VA_TRY(check_geometry(batch, M, seg));
  T2VA_TRY(check_dtype(dtype));
  if (batch == 0) return T2VA_SUCCESS;
  for (const void* const* p : {z_t, x0_teacher, x0_student, x0_student_tangent})
    T2VA_TRY(check_ptrs(M, seg, p));
  T2VA_TRY(check_ptrs(M, seg, reinterpret_cast<const void* const*>(grad_x0_student)));
  T2VA_TRY(check_scalar_out(t, true));
  T2VA_TRY(check_scalar_out(loss, true));
  T2VA_TRY(check_scalar_out(norm, false));
  T2VA_TRY(check_scalar_out(status, true));
  T2VA_TRY(check_weights(M, weight));
  if (!finite(beta) || !(gamma >= 0.f && gamma <= 1.f) || !finite(eps_scm) || !(eps_scm > 0.f) ||
      !finite(lambda_scm))
    return T2VA_ERROR_INVALID_ARGUMENT;
  ObjectiveArgs a;
  fill_geometry(a, batch, M, seg);
  for (int m = 0; m < M; ++m) {
    a.in[kZt][m] = z_t[m];
    a.in[kXT][m] = x0_teacher[m];
    a.in[kXS][m] = x0_student[m];
    a.in[kXdot][m] = x0_student_tangent[m];
    a.grad_s[m] = grad_x0_student[m];
    a.w[m] = weight[m];
  }
  a.t = t;
  a.beta = beta;
  a.gamma = gamma;
  a.eps_s = eps_scm;
  a.lam_s = lambda_scm;
  a.accumulate = accumulate ? 1 : 0;
  a.loss = loss;
  a.norm = norm;
  a.status = status;
  return run_objective(a, dtype, kModeScm, caller_workspace(workspace, workspace_bytes), stream);
}

int t2va_dmd_objective(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                       const void* const* zhat0, const void* const* x0_teacher_hat,
                       const void* const* x0_fake, float eps_dmd, const float* weight,
                       float lambda_dmd, float* const* grad_zhat0, int accumulate,
                       float* loss, float* cdmd,
                       void* workspace, size_t workspace_bytes, int* status,
                       cudaStream_t stream) {
  const int M = num_modalities;
  T2VA_TRY(check_geometry(batch, M, seg));
  T2VA_TRY(check_dtype(dtype));
  if (batch == 0) return T2VA_SUCCESS;
  for (const void* const* p : {zhat0, x0_teacher_hat, x0_fake}) T2VA_TRY(check_ptrs(M, seg, p));
  T2VA_TRY(check_ptrs(M, seg, reinterpret_cast<const void* const*>(grad_zhat0)));
  T2VA_TRY(check_scalar_out(loss, true));
  T2VA_TRY(check_scalar_out(cdmd, false));
  T2VA_TRY(check_scalar_out(status, true));
  T2VA_TRY(check_weights(M, weight));
  if (!finite(eps_dmd) || !(eps_dmd > 0.f) || !finite(lambda_dmd)) return T2VA_ERROR_INVALID_ARGUMENT;
  ObjectiveArgs a;
  fill_geometry(a, batch, M, seg);
  for (int m = 0; m < M; ++m) {
    a.in[kZh][m] = zhat0[m];
    a.in[kYT][m] = x0_teacher_hat[m];
    a.in[kYF][m] = x0_fake[m];
    a.grad_d[m] = grad_zhat0[m];
    a.w[m] = weight[m];
  }
  a.eps_d = eps_dmd;
  a.lam_d = lambda_dmd;
  a.accumulate = accumulate ? 1 : 0;
  a.loss = loss;
  a.cdmd = cdmd;
  a.status = status;
  return run_objective(a, dtype, kModeDmd, caller_workspace(workspace, workspace_bytes), stream);
}

int t2va_stage3_objective(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                          const void* const* z_t, const void* const* x0_teacher,
                          const void* const* x0_student, const void* const* x0_student_tangent,
                          const float* t,
                          const void* const* zhat0, const void* const* x0_teacher_hat,
                          const void* const* x0_fake,
                          float beta, float gamma, float eps_scm, float eps_dmd,
                          const float* weight, float lambda_scm, float lambda_dmd,
                          float* const* grad_x0_student, float* const* grad_zhat0, int accumulate,
                          float* loss, float* loss_scm, float* loss_dmd, float* norm, float* cdmd,
                          void* workspace, size_t workspace_bytes, int* status,
                          cudaStream_t stream) {
  return stage3_entry(batch, num_modalities, seg, dtype, z_t, x0_teacher, x0_student,
                      x0_student_tangent, t, zhat0, x0_teacher_hat, nullptr, nullptr, x0_fake, beta,
                      gamma, eps_scm, eps_dmd, weight, lambda_scm, lambda_dmd, grad_x0_student,
                      grad_zhat0, accumulate, loss, loss_scm, loss_dmd, norm, cdmd,
                      caller_workspace(workspace, workspace_bytes), status, stream);
}

int t2va_stage3_objective_cfg(
    int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
    const void* const* z_t, const void* const* x0_teacher, const void* const* x0_student,
    const void* const* x0_student_tangent, const float* t, const void* const* zhat0,
    const void* const* x0_teacher_hat_cond, const void* const* x0_teacher_hat_uncond,
    const float* guidance, const void* const* x0_fake, float beta, float gamma, float eps_scm,
    float eps_dmd, const float* weight, float lambda_scm, float lambda_dmd,
    float* const* grad_x0_student, float* const* grad_zhat0, int accumulate, float* loss,
    float* loss_scm, float* loss_dmd, float* norm, float* cdmd, void* workspace,
    size_t workspace_bytes, int* status, cudaStream_t stream) {
  if (x0_teacher_hat_uncond == nullptr) return T2VA_ERROR_INVALID_ARGUMENT;
  return stage3_entry(batch, num_modalities, seg, dtype, z_t, x0_teacher, x0_student,
                      x0_student_tangent, t, zhat0, x0_teacher_hat_cond, x0_teacher_hat_uncond,
                      guidance, x0_fake, beta, gamma, eps_scm, eps_dmd, weight, lambda_scm,
                      lambda_dmd, grad_x0_student, grad_zhat0, accumulate, loss, loss_scm,
                      loss_dmd, norm, cdmd, caller_workspace(workspace, workspace_bytes), status,
                      stream);
}

}  // extern "C"
