// TrigFlow noising kernel: z_t = cos(t) z0 + sin(t) eps per modality, with one
// timestep per sample shared by all modalities (TurboT2VA, section 三 of the
// robotworld.top/zh reading: the noising equation; section 2 of the
// robotworld.top/en summary), fused with the TrigFlow -> rectified-flow wrapper
// (section 4.2 of the zh reading; Eq. 16 of the en summary): z_rf = z_t / (cos t +
// sin t) and t_rf = sin t / (cos t + sin t).
//
// HBM-bound stream: 2 reads and 1 or 2 writes per element. Each CTA owns one chunk
// of one (sample, modality) segment, so the per-sample sin/cos is computed once per
// thread and every access is a coalesced 16-byte vector; the few elements before
// the first 16-byte boundary and after the last full vector of a segment are
// done one by one by the first and last chunk. Both outputs come from the same
// loaded z0 and eps, each with one fma of float32 coefficients: cos t, sin t for
// z_t, and cos t / (cos t + sin t), sin t / (cos t + sin t) for z_rf.
#include "t2va_internal.cuh"

namespace t2va {
namespace {

// Small CTAs: 128 threads of at most 32 registers (4096 registers a CTA) fit on an SM
// beside three CTAs of the objective kernels (3 x 256 threads x 80 registers), so the
// noising of the next steps runs on every SM while an objective call streams. Measured on
// B300 in the stage-3 512x768 step: 256 threads x 4 vectors (40-56 registers) 20.84 us,
// 256 x 2 20.74 us, 128 x 4 20.95 us, 128 x 2 20.55 us; the noising alone 7.01, 7.32, 7.83
// and 7.10 us.
constexpr int kNoiseThreads = 128;
constexpr int kNoiseUnroll = 2;
constexpr int kNoiseVecPerCta = kNoiseThreads * kNoiseUnroll;
// Vectors of each input a CTA prefetches into L2 before its dependency wait: with 256
// vectors a CTA, all of them. Measured on B300 in the stage-3 512x768 step: with 256-vector
// CTAs, 64, 128 and 192 vectors gave 20.66, 20.67 and 20.52 us per step against 20.42 for
// all 256; with 1024-vector CTAs, 256, 384, 512, 640 and 1024 vectors gave 21.24, 21.21,
// 21.17, 21.15 and 21.30 us against 21.35 without.
constexpr int64_t kNoiseEarlyVec = 512;

// The noised samples are read next by the objective: their lines are stored with an
// evict_last L2 policy so that they are still there when it reads them (measured
// faster for the whole noising + objective step, on one stream or two).
__device__ __forceinline__ uint64_t policy_keep() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

template <typename T>
__device__ __forceinline__ void store_vec(void* p, const float* v);

template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16>(void* p, const float* v) {
  uint4 r;
  __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 h2 = __floats2bfloat162_rn(v[4], v[5]);
  __nv_bfloat162 h3 = __floats2bfloat162_rn(v[6], v[7]);
  r.x = *reinterpret_cast<uint32_t*>(&h0);
  r.y = *reinterpret_cast<uint32_t*>(&h1);
  r.z = *reinterpret_cast<uint32_t*>(&h2);
  r.w = *reinterpret_cast<uint32_t*>(&h3);
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(r.x), "r"(r.y),
               "r"(r.z), "r"(r.w), "l"(policy_keep())
               : "memory");
}

template <>
__device__ __forceinline__ void store_vec<float>(void* p, const float* v) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3]), "l"(policy_keep())
               : "memory");
}

template <typename T>
__device__ __forceinline__ void store_scalar(void* base, int64_t e, float v);
template <>
__device__ __forceinline__ void store_scalar<float>(void* base, int64_t e, float v) {
  reinterpret_cast<float*>(base)[e] = v;
}
template <>
__device__ __forceinline__ void store_scalar<__nv_bfloat16>(void* base, int64_t e, float v) {
  reinterpret_cast<__nv_bfloat16*>(base)[e] = __float2bfloat16_rn(v);
}

// One output element from the loaded pair and the output's two coefficients.
__device__ __forceinline__ float mix(float cz, float z, float ce, float e) {
  return fmaf(cz, z, ce * e);
}

// 16 CTAs an SM caps a thread at 32 registers; the kernel writing both z_t and z_rf gets
// 42 (12 CTAs), since at 32 it spills and ran 10.5 instead of 8.3 us.
template <typename T, int OUT>
__global__ void __launch_bounds__(kNoiseThreads, OUT == (kNoiseZt | kNoiseRf) ? 12 : 16)
    k_noise(const __grid_constant__ NoiseArgs a) {
  constexpr int VE = Vec<T>::VE;
  const int bid = blockIdx.x;

  // The HBM stream starts while the previous kernel drains: threads 0 and 1 ask L2 for
  // the first kNoiseEarlyVec vectors of this CTA's z0 and eps (a bulk prefetch returns
  // nothing to the SM and L2 is the point of coherence, so it may run before the wait).
  // Only these two threads work out the chunk here; the whole CTA does it again after
  // the wait (doing it once, for every thread, before the wait measured 0.66 us slower).
  if (threadIdx.x < 2 && bid < a.block_off[a.M]) {
    int m = 0;
#pragma unroll
    for (int i = 1; i < kMaxM; ++i)
      if (i < a.M && bid >= a.block_off[i]) m = i;
    const int local = bid - a.block_off[m];
    const int b = local / a.chunks[m];
    const SegGeom g = seg_geom<VE>(a.n[m], a.stride[m], b);
    const int64_t vbeg = (int64_t)(local - b * a.chunks[m]) * kNoiseVecPerCta;
    int64_t nv = g.nvec - vbeg;
    if (nv > kNoiseEarlyVec) nv = kNoiseEarlyVec;
    if (nv > 0) {
      const T* p = reinterpret_cast<const T*>(threadIdx.x == 0 ? a.z0[m] : a.eps[m]) + g.e0 + g.head +
                   vbeg * VE;
      uint64_t first;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(first));
      asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p),
                   "r"((uint32_t)(nv * 16)), "l"(first)
                   : "memory");
    }
  }
  // launched as a programmatic dependent of the previous kernel on the stream: no
  // load before that kernel has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  // the rectified-flow time of sample `bid`, by CTA `bid` (the grid has at least B CTAs)
  if ((OUT & kNoiseRf) && a.t_rf != nullptr && bid < a.B && threadIdx.x == 0) {
    float s, c;
    sincosf(__ldg(a.t + bid), &s, &c);
    a.t_rf[bid] = s / (c + s);
  }
  if (bid >= a.block_off[a.M]) return;  // a CTA only there for t_rf

  int m = 0;
#pragma unroll
  for (int i = 1; i < kMaxM; ++i)
    if (i < a.M && bid >= a.block_off[i]) m = i;
  const int local = bid - a.block_off[m];
  const int b = local / a.chunks[m];
  const int chunk = local - b * a.chunks[m];

  const float t = __ldg(a.t + b);
  float s, c;
  sincosf(t, &s, &c);
  if (!isfinite(t) && a.status != nullptr && threadIdx.x == 0 && chunk == 0)
    atomicOr(a.status, T2VA_STATUS_BAD_TIMESTEP);
  float cr = 0.f, sr = 0.f;
  if (OUT & kNoiseRf) {
    cr = c / (c + s);
    sr = s / (c + s);
  }

  const SegGeom g = seg_geom<VE>(a.n[m], a.stride[m], b);
  const int64_t vec0 = g.e0 + g.head;  // element index of vector 0
  const T* z0 = reinterpret_cast<const T*>(a.z0[m]);
  const T* ep = reinterpret_cast<const T*>(a.eps[m]);
  T* zt = reinterpret_cast<T*>(a.zt[m]);
  T* zr = reinterpret_cast<T*>(a.zrf[m]);

  const int64_t vbeg = (int64_t)chunk * kNoiseVecPerCta;
  uint4 rz[kNoiseUnroll], re[kNoiseUnroll];
#pragma unroll
  for (int u = 0; u < kNoiseUnroll; ++u) {
    const int64_t v = vbeg + u * kNoiseThreads + threadIdx.x;
    if (v < g.nvec) {
      rz[u] = ld_stream16(z0 + vec0 + v * VE);
      re[u] = ld_stream16(ep + vec0 + v * VE);
    }
  }
#pragma unroll
  for (int u = 0; u < kNoiseUnroll; ++u) {
    const int64_t v = vbeg + u * kNoiseThreads + threadIdx.x;
    if (v < g.nvec) {
      Vec<T> vz, ve;
      vz.from(rz[u]);
      ve.from(re[u]);
      float o[VE];
      if (OUT & kNoiseZt) {
#pragma unroll
        for (int k = 0; k < VE; ++k) o[k] = mix(c, vz.v[k], s, ve.v[k]);
        store_vec<T>(zt + vec0 + v * VE, o);
      }
      if (OUT & kNoiseRf) {
#pragma unroll
        for (int k = 0; k < VE; ++k) o[k] = mix(cr, vz.v[k], sr, ve.v[k]);
        store_vec<T>(zr + vec0 + v * VE, o);
      }
    }
  }
  // unaligned head (first chunk) and tail (last chunk): one element per thread each
  // (a one-chunk segment's thread may have one of both)
#pragma unroll
  for (int side = 0; side < 2; ++side) {
    int64_t e = -1;
    if (side == 0 && chunk == 0 && threadIdx.x < g.head) e = g.e0 + threadIdx.x;
    if (side == 1 && chunk == a.chunks[m] - 1 && threadIdx.x < g.tail)
      e = vec0 + g.nvec * VE + threadIdx.x;
    if (e >= 0) {
      const float z = load_scalar<T>(z0, e), x = load_scalar<T>(ep, e);
      if (OUT & kNoiseZt) store_scalar<T>(zt, e, mix(c, z, s, x));
      if (OUT & kNoiseRf) store_scalar<T>(zr, e, mix(cr, z, sr, x));
    }
  }
}

}  // namespace

int noise_vectors_per_cta() { return kNoiseVecPerCta; }

cudaError_t launch_noise(const NoiseArgs& a, t2va_dtype dt, int outputs, int grid,
                         cudaStream_t st) {
  // a programmatic dependent of the previous work on the stream (see k_noise)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kNoiseThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool bf = dt == T2VA_BFLOAT16;
  switch (outputs) {
    case kNoiseZt:
      return bf ? cudaLaunchKernelEx(&cfg, k_noise<__nv_bfloat16, kNoiseZt>, a)
                : cudaLaunchKernelEx(&cfg, k_noise<float, kNoiseZt>, a);
    case kNoiseRf:
      return bf ? cudaLaunchKernelEx(&cfg, k_noise<__nv_bfloat16, kNoiseRf>, a)
                : cudaLaunchKernelEx(&cfg, k_noise<float, kNoiseRf>, a);
    case kNoiseZt | kNoiseRf:
      return bf ? cudaLaunchKernelEx(&cfg, k_noise<__nv_bfloat16, kNoiseZt | kNoiseRf>, a)
                : cudaLaunchKernelEx(&cfg, k_noise<float, kNoiseZt | kNoiseRf>, a);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace t2va
