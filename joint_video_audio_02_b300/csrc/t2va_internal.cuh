// Internal declarations shared by the kernels and the C-ABI layer of the
// joint video-audio distillation objective library (sm_103a).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "t2va.h"

namespace t2va {

constexpr int kMaxM = T2VA_MAX_MODALITIES;
constexpr uint32_t kWsMagic = 0x54325641u;  // "T2VA"

// ---------------------------------------------------------------------------
// Workspace layout (caller-owned device memory)
//   [0, 256)     header: written by t2va_workspace_init; no kernel reads it
//   [256, ...)   partial sums: float4 {sum g_sCM^2, sum |zhat0 - y_T|, sum g_DMD^2, 0}
//                per (sample, modality, chunk), kMaxChunks chunks per (sample, modality),
//                written by the first kernel of a call and read by the second
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t magic;
  uint32_t pad[63];
};
static_assert(sizeof(WsHeader) == 256, "header size");

constexpr size_t kWsHeaderBytes = 256;
constexpr int kQuantities = 3;  // sum g_sCM^2, sum |zhat0 - y_T|, sum g_DMD^2
constexpr int kMaxChunks = 1024;  // chunks per (sample, modality) row

inline size_t ws_body_bytes(int B, int M) { return (size_t)B * M * kMaxChunks * 16; }
inline size_t ws_bytes(int B, int M) { return kWsHeaderBytes + ws_body_bytes(B, M); }

// A workspace as the objective sees it: the partial-sum area behind the header.
struct WsRef {
  unsigned char* body;
  size_t body_bytes;
};

// Modes of the objective kernel.
enum : int { kModeScm = 1, kModeDmd = 2, kModeStage3 = 3, kModeCfg = 4 };

// Input tensor slots of the objective kernel.
// With kModeCfg, slot kYT holds the teacher's conditional prediction at the re-noised
// sample and kYU its unconditional one; the guided prediction is formed per element.
enum : int { kZt = 0, kXT = 1, kXS = 2, kXdot = 3, kZh = 4, kYT = 5, kYF = 6, kYU = 7,
             kNumInputs = 8 };

struct ObjectiveArgs {
  int B, M;
  int64_t n[kMaxM];
  int64_t stride[kMaxM];
  const void* in[kNumInputs][kMaxM];
  float* grad_s[kMaxM];
  float* grad_d[kMaxM];
  const float* t;
  float beta, gamma, eps_s, lam_s, eps_d, lam_d;
  float w[kMaxM];
  float cfg[kMaxM];            // guidance scale per modality (kModeCfg)
  int accumulate;
  uint32_t alias_mask;         // bit m: grad_d[m] == grad_s[m], write the sum once
  uint32_t wide_mask;          // bit m: the gradient buffers of m are 32-byte aligned
  float* loss;
  float* loss_s;
  float* loss_d;
  float* norm;
  float* cdmd;
  float* partials;             // float4 [B][M][kMaxChunks]
  int* status;
  // launch plan (filled by plan_objective)
  int vpc;                     // 16-byte vectors per chunk (a multiple of one CTA's batch)
  int nchunk[kMaxM];           // chunks per (sample, modality m) row
  int choff[kMaxM + 1];        // first chunk of modality m inside a sample; choff[M] = per sample
  int out_m, out_c;            // the chunk of each sample that writes the per-sample outputs
};

struct NoiseArgs {
  int B, M;
  int64_t n[kMaxM];
  int64_t stride[kMaxM];
  const void* z0[kMaxM];
  const void* eps[kMaxM];
  void* zt[kMaxM];             // TrigFlow sample (when the launch writes it)
  void* zrf[kMaxM];            // rectified-flow sample (when the launch writes it)
  int chunks[kMaxM];           // CTAs per (sample, modality)
  int block_off[kMaxM + 1];    // first CTA of each modality; block_off[M] = element CTAs
  const float* t;
  float* t_rf;                 // rectified-flow time per sample, or null
  int* status;
};

// Outputs of a noising launch.
enum NoiseOut : int { kNoiseZt = 1, kNoiseRf = 2 };

// Launchers (defined next to their kernels). They return a cudaError_t.
// `grid` is at least a.block_off[a.M], and at least a.B when a.t_rf is set.
cudaError_t launch_noise(const NoiseArgs& a, t2va_dtype dt, int outputs, int grid, cudaStream_t st);
int noise_vectors_per_cta();

struct ObjectiveLaunch {
  int grid;
  int threads;
  size_t smem;
  int grad_per;  // vectors per thread in flight in the gradient pass: 1 or 2
};
// Chooses the chunks and the grid for `a` (fills the plan fields); returns false if
// the problem is too large for the workspace layout.
bool plan_objective(ObjectiveArgs& a, t2va_dtype dt, int sm_count, ObjectiveLaunch* out);
cudaError_t launch_objective(const ObjectiveArgs& a, t2va_dtype dt, int mode,
                             const ObjectiveLaunch& l, cudaStream_t st);
cudaError_t launch_workspace_init(void* ws, size_t bytes, cudaStream_t st);

// The stage-3 entry points after their own checks (t2va_api.cu): argument validation,
// then the workspace check, then the launch. Without guidance x0_teacher_hat_uncond
// and guidance are null. A workspace whose body is null fails the workspace check.
int stage3_entry(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                 const void* const* z_t, const void* const* x0_teacher,
                 const void* const* x0_student, const void* const* x0_student_tangent,
                 const float* t, const void* const* zhat0, const void* const* x0_teacher_hat,
                 const void* const* x0_teacher_hat_uncond, const float* guidance,
                 const void* const* x0_fake, float beta, float gamma, float eps_scm,
                 float eps_dmd, const float* weight, float lambda_scm, float lambda_dmd,
                 float* const* grad_x0_student, float* const* grad_zhat0, int accumulate,
                 float* loss, float* loss_scm, float* loss_dmd, float* norm, float* cdmd,
                 const WsRef& ws, int* status, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

// 16-byte streaming load through the read-only path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ void st_stream16(void* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// bfloat16 pair (low half = element 0) -> two floats, exact.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Vector of VE elements loaded from one 16-byte chunk.
template <typename T>
struct Vec;

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int VE = 8;
  float v[8];
  __device__ __forceinline__ void from(uint4 r) {
    v[0] = bf_lo(r.x); v[1] = bf_hi(r.x);
    v[2] = bf_lo(r.y); v[3] = bf_hi(r.y);
    v[4] = bf_lo(r.z); v[5] = bf_hi(r.z);
    v[6] = bf_lo(r.w); v[7] = bf_hi(r.w);
  }
};

template <>
struct Vec<float> {
  static constexpr int VE = 4;
  float v[4];
  __device__ __forceinline__ void from(uint4 r) {
    v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
    v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
  }
};

template <typename T>
__device__ __forceinline__ float load_scalar(const void* base, int64_t e);
template <>
__device__ __forceinline__ float load_scalar<float>(const void* base, int64_t e) {
  return __ldg(reinterpret_cast<const float*>(base) + e);
}
template <>
__device__ __forceinline__ float load_scalar<__nv_bfloat16>(const void* base, int64_t e) {
  unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(base) + e);
  return __uint_as_float(((uint32_t)u) << 16);
}

// Per-sample coefficients of the sCM direction written as
//   g = kD (x0_T - x0_S) + kz z_t + kx tangent,
// which is the printed direction with F_theta - F_T = (x0_T - x0_S)/s and
// J = -c s z_t - c^2 (F_theta - F_T) - c tangent, so
//   kD = (c^2 - beta c / D) / s,  D = sqrt(1 - gamma^2 s^2),  kz = (1 - gamma) c s,  kx = c.
// Evaluated in float32 without cancellation: D^2 = (1 - gamma^2) + gamma^2 c^2 and
//   c D - 1 = -s^2 (1 + gamma^2 c^2) / (c D + 1),
//   kD = c ((c D - 1) + (1 - beta)) / (D s).
struct Coef {
  float c, s, kD, kz, kx;
  bool ok;
};

__device__ __forceinline__ Coef sample_coef(float t, float beta, float gamma) {
  Coef k;
  float s, c;
  sincosf(t, &s, &c);
  k.c = c;
  k.s = s;
  const float g2 = gamma * gamma;
  const float c2 = c * c;
  const float D = sqrtf(fmaf(g2, c2, (1.f - gamma) * (1.f + gamma)));
  const float cD = c * D;
  const float cDm1 = -(s * s) * fmaf(g2, c2, 1.f) / (cD + 1.f);
  k.kD = c * (cDm1 + (1.f - beta)) / (D * s);
  k.kz = (1.f - gamma) * c * s;
  k.kx = c;
  // 0 < t < pi/2: 1.57079637f is pi/2 rounded up, so no float lies between the bounds.
  k.ok = (t > 0.f) && (t < 1.57079637f);
  if (!k.ok) {
    const float qnan = __int_as_float(0x7fc00000);
    k.kD = k.kz = k.kx = k.s = qnan;
  }
  return k;
}

// Where the 16-byte-aligned vectors of one (sample, modality) segment start.
// Elements [0, head) and [head + nvec*VE, n) are handled one by one.
struct SegGeom {
  int64_t e0;     // first element of the sample
  int64_t head;   // scalar elements before the first aligned vector
  int64_t nvec;   // aligned vectors
  int64_t tail;   // scalar elements after the last vector
};

template <int VE>
__device__ __forceinline__ SegGeom seg_geom(int64_t n, int64_t stride, int b) {
  SegGeom g;
  g.e0 = (int64_t)b * stride;
  int64_t mis = g.e0 & (VE - 1);
  int64_t head = (VE - mis) & (VE - 1);
  g.head = head < n ? head : n;
  g.nvec = (n - g.head) / VE;
  g.tail = n - g.head - g.nvec * VE;
  return g;
}

#endif  // __CUDACC__

}  // namespace t2va
