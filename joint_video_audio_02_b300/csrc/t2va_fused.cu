// Fused gated residual + modulated RMS normalisation (TurboT2VA, section 6.3 of the
// robotworld.top/zh reading: the joint Transformer combines a normalisation with a
// modality- and timestep-dependent modulation, then a gated residual update; the pages
// name the fused patterns but print no formulas, and the standard forms are taken):
//
//   h' = h + gate * u,   y = h' / sqrt(mean(h'^2) + eps) * (1 + scale) + shift
//
// per token row of width D; gate, scale and shift are float32 vectors of width D per
// sample. h' is rounded to the latent dtype (and stored if asked), and the
// normalisation uses the rounded values, as the unfused operators would.
//
// k_residual_modnorm: 128 threads per row, two rows per CTA. Each thread keeps its four
// vectors of h' (a 4096-element bf16 row) in registers between the two passes; longer
// rows read the rest again (from the stored h', or h and u, through L2). The row's sum of
// squares is reduced by shuffles and then across the row's four warps in a fixed order,
// and the reciprocal square root is the correctly rounded one. HBM-bound: per bf16
// element 2 bytes read for h, 2 for u, 2 written for h', 2 for y.
#include "t2va_fused.cuh"

namespace t2va {
namespace {

constexpr int kFThreads = 256;
constexpr int kFTPR = 128;                 // threads per row
constexpr int kFRows = kFThreads / kFTPR;  // rows per CTA
constexpr int kFCache = 4;                 // 16-byte vectors per thread kept in registers
constexpr int kFWarpsPerRow = kFTPR / 32;

template <typename T>
struct VecT;
template <>
struct VecT<__nv_bfloat16> {
  static constexpr int VE = 8;
  static __device__ __forceinline__ void unpack(const uint4& r, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = __bfloat1622float2(h[i]);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    uint4 r;
    uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return r;
  }
};
template <>
struct VecT<float> {
  static constexpr int VE = 4;
  static __device__ __forceinline__ void unpack(const uint4& r, float* f) {
    const float* s = reinterpret_cast<const float*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = s[i];
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    uint4 r;
    float* d = reinterpret_cast<float*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = f[i];
    return r;
  }
};

// VE consecutive float32 values of a per-sample vector (32-byte or 16-byte aligned).
template <int VE>
__device__ __forceinline__ void load_vec_f32(const float* p, float* f) {
#pragma unroll
  for (int i = 0; i < VE; i += 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p + i));
    f[i] = v.x;
    f[i + 1] = v.y;
    f[i + 2] = v.z;
    f[i + 3] = v.w;
  }
}

// h' of one vector: from h and u (rounded to T and back), or h itself.
template <typename T>
__device__ __forceinline__ uint4 residual_vec(const FusedArgs& a, int64_t row, int64_t b, int64_t v) {
  using V = VecT<T>;
  constexpr int VE = V::VE;
  // a plain load: h' may be stored over h (an in-place update), so h is not read-only
  const uint4 rh = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.h) + row * a.D + v * VE);
  if (a.u == nullptr) return rh;
  float h[VE], u[VE], g[VE], o[VE];
  V::unpack(rh, h);
  V::unpack(ld_stream16(reinterpret_cast<const T*>(a.u) + row * a.D + v * VE), u);
  if (a.gate != nullptr) {
    load_vec_f32<VE>(a.gate + b * a.D + v * VE, g);
  } else {
#pragma unroll
    for (int i = 0; i < VE; ++i) g[i] = 1.f;
  }
#pragma unroll
  for (int i = 0; i < VE; ++i) o[i] = fmaf(g[i], u[i], h[i]);
  return V::pack(o);
}

template <typename T>
__global__ void __launch_bounds__(kFThreads) k_residual_modnorm(const __grid_constant__ FusedArgs a) {
  using V = VecT<T>;
  constexpr int VE = V::VE;
  __shared__ float red[kFThreads / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int t = threadIdx.x % kFTPR;
  const int64_t row = (int64_t)blockIdx.x * kFRows + threadIdx.x / kFTPR;
  const bool live = row < a.rows;
  const int64_t b = live ? row / a.rows_per_sample : 0;
  const int64_t nvec = live ? a.D / VE : 0;

  // pass 1: h' (stored if asked), and the sum of squares of its stored values
  uint4 cache[kFCache];
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < kFCache; ++c) {
    const int64_t v = (int64_t)c * kFTPR + t;
    if (v < nvec) {
      cache[c] = residual_vec<T>(a, row, b, v);
      if (a.h_out != nullptr) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.h_out) + row * a.D + v * VE) = cache[c];
      float f[VE];
      V::unpack(cache[c], f);
#pragma unroll
      for (int i = 0; i < VE; ++i) ss = fmaf(f[i], f[i], ss);
    }
  }
  for (int64_t v = (int64_t)kFCache * kFTPR + t; v < nvec; v += kFTPR) {
    const uint4 r = residual_vec<T>(a, row, b, v);
    if (a.h_out != nullptr) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.h_out) + row * a.D + v * VE) = r;
    float f[VE];
    V::unpack(r, f);
#pragma unroll
    for (int i = 0; i < VE; ++i) ss = fmaf(f[i], f[i], ss);
  }
  // the row's sum: lanes, then the row's warps in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  const int w0 = (threadIdx.x >> 5) / kFWarpsPerRow * kFWarpsPerRow;
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kFWarpsPerRow; ++w) tot += red[w0 + w];
  if (!live) return;
  const float r = __frsqrt_rn(tot / (float)a.D + a.eps);

  // pass 2: y = h' r (1 + scale) + shift, written once
  auto emit = [&](const uint4& hv, int64_t v) {
    float f[VE], sc[VE], sh[VE], o[VE];
    V::unpack(hv, f);
    if (a.scale != nullptr) {
      load_vec_f32<VE>(a.scale + b * a.D + v * VE, sc);
    } else {
#pragma unroll
      for (int i = 0; i < VE; ++i) sc[i] = 0.f;
    }
    if (a.shift != nullptr) {
      load_vec_f32<VE>(a.shift + b * a.D + v * VE, sh);
    } else {
#pragma unroll
      for (int i = 0; i < VE; ++i) sh[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < VE; ++i) o[i] = fmaf(f[i] * r, 1.f + sc[i], sh[i]);
    *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.y) + row * a.D + v * VE) = V::pack(o);
  };
#pragma unroll
  for (int c = 0; c < kFCache; ++c) {
    const int64_t v = (int64_t)c * kFTPR + t;
    if (v < nvec) emit(cache[c], v);
  }
  for (int64_t v = (int64_t)kFCache * kFTPR + t; v < nvec; v += kFTPR) {
    // beyond the registers: the stored h' if there is one, else h' formed again
    const uint4 hv = a.h_out != nullptr
                         ? *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.h_out) + row * a.D + v * VE)
                         : residual_vec<T>(a, row, b, v);
    emit(hv, v);
  }
}

}  // namespace

cudaError_t launch_residual_modnorm(const FusedArgs& a, t2va_dtype dt, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.rows + kFRows - 1) / kFRows));
  cfg.blockDim = dim3(kFThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dt == T2VA_BFLOAT16) return cudaLaunchKernelEx(&cfg, k_residual_modnorm<__nv_bfloat16>, a);
  return cudaLaunchKernelEx(&cfg, k_residual_modnorm<float>, a);
}

}  // namespace t2va
