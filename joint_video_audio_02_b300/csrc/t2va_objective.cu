// Fused joint sCM / DMD / stage-3 objective kernel (TurboT2VA, robotworld.top/zh
// reading: section 3.1 joint sCM, section 四 joint DMD, section 4.1 stage-3 sum;
// robotworld.top/en summary: Eq. 6 and Eq. 11-12).
//
// Design (one persistent launch, one CTA per SM, all CTAs co-resident):
//   for every sample b, every CTA owns a contiguous slice of that sample's
//   16-byte vectors (video and audio segments back to back), so every sample is
//   spread over the whole GPU and the small audio segment never idles SMs.
//   Phase A(b): stream the slice's inputs once (16-byte loads), compute the
//     float32 directions g_sCM and g_DMD, keep them in shared memory, and
//     accumulate the per-(sample, modality) sums  sum g_sCM^2, sum |zhat0 - y_T|,
//     sum g_DMD^2. The CTA's sums go to the workspace; then the CTA arrives on
//     the sample's counter.
//   Wait(b): a bounded spin on the sample's generation word; every CTA then
//     merges the per-CTA sums itself in a fixed order (all CTAs get identical,
//     run-to-run reproducible totals).
//   Phase W(b): scale the kept directions by the per-(sample, modality) factor
//     and write the float32 gradients once.
//   With two shared-memory slots the order is A0 A1 W0 A2 W1 ... so sample b's
//   barrier is hidden behind sample b+1's reads. Vectors that do not fit in
//   shared memory are recomputed from the inputs in phase W.
// HBM traffic is therefore the algorithmic minimum whenever the direction of
// one (or two) samples fits on chip: each input read once, each gradient
// written once.
#include "t2va_internal.cuh"

namespace t2va {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 2;

struct SmemCtl {
  float red[2][kWarps][kMaxM][kQuantities];
  float tot[kMaxM][kQuantities];
  uint64_t timeout_ns;
  uint32_t gen_wait[2];
  int abort;
  int checked;
};
constexpr size_t kCtlBytes = (sizeof(SmemCtl) + 15) / 16 * 16;

template <typename T, int MODE>
struct Traits {
  static constexpr int VE = Vec<T>::VE;
  static constexpr bool kScm = (MODE & kModeScm) != 0;
  static constexpr bool kDmd = (MODE & kModeDmd) != 0;
  static constexpr int Q = (kScm ? 1 : 0) + (kDmd ? 1 : 0);
  static constexpr int P = Q * VE / 4;  // float4 pieces kept per vector
};

template <typename T, int MODE>
struct Loaded {
  uint4 r[kNumInputs];
};

template <typename T, int MODE>
__device__ __forceinline__ void load_vec(Loaded<T, MODE>& L, const ObjectiveArgs& a, int m,
                                         int64_t e) {
  using Tr = Traits<T, MODE>;
  const T* p;
  if constexpr (Tr::kScm) {
    p = reinterpret_cast<const T*>(a.in[kZt][m]); L.r[kZt] = ld_stream16(p + e);
    p = reinterpret_cast<const T*>(a.in[kXT][m]); L.r[kXT] = ld_stream16(p + e);
    p = reinterpret_cast<const T*>(a.in[kXS][m]); L.r[kXS] = ld_stream16(p + e);
    p = reinterpret_cast<const T*>(a.in[kXdot][m]); L.r[kXdot] = ld_stream16(p + e);
  }
  if constexpr (Tr::kDmd) {
    p = reinterpret_cast<const T*>(a.in[kZh][m]); L.r[kZh] = ld_stream16(p + e);
    p = reinterpret_cast<const T*>(a.in[kYT][m]); L.r[kYT] = ld_stream16(p + e);
    p = reinterpret_cast<const T*>(a.in[kYF][m]); L.r[kYF] = ld_stream16(p + e);
  }
}

// Directions of one vector: gs (sCM) and gd (DMD), and the three sums.
template <typename T, int MODE>
__device__ __forceinline__ void directions(const Loaded<T, MODE>& L, const Coef& k,
                                           float* gs, float* gd, float& sg, float& sa,
                                           float& sd) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  if constexpr (Tr::kScm) {
    Vec<T> z, xt, xs, xd;
    z.from(L.r[kZt]);
    xt.from(L.r[kXT]);
    xs.from(L.r[kXS]);
    xd.from(L.r[kXdot]);
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      const float g = fmaf(k.kD, xt.v[i] - xs.v[i], fmaf(k.kz, z.v[i], k.kx * xd.v[i]));
      gs[i] = g;
      sg = fmaf(g, g, sg);
    }
  }
  if constexpr (Tr::kDmd) {
    Vec<T> zh, yt, yf;
    zh.from(L.r[kZh]);
    yt.from(L.r[kYT]);
    yf.from(L.r[kYF]);
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      const float g = yf.v[i] - yt.v[i];
      gd[i] = g;
      sd = fmaf(g, g, sd);
      sa += fabsf(zh.v[i] - yt.v[i]);
    }
  }
}

// One element, for the unaligned head and tail of a segment.
template <typename T, int MODE>
__device__ __forceinline__ void direction_scalar(const ObjectiveArgs& a, int m, int64_t e,
                                                 const Coef& k, float& gs, float& gd) {
  using Tr = Traits<T, MODE>;
  if constexpr (Tr::kScm) {
    const float z = load_scalar<T>(a.in[kZt][m], e);
    const float xt = load_scalar<T>(a.in[kXT][m], e);
    const float xs = load_scalar<T>(a.in[kXS][m], e);
    const float xd = load_scalar<T>(a.in[kXdot][m], e);
    gs = fmaf(k.kD, xt - xs, fmaf(k.kz, z, k.kx * xd));
  }
  if constexpr (Tr::kDmd) {
    const float yt = load_scalar<T>(a.in[kYT][m], e);
    const float yf = load_scalar<T>(a.in[kYF][m], e);
    gd = yf - yt;
  }
}

template <typename T, int MODE>
__device__ __forceinline__ float abs_residual_scalar(const ObjectiveArgs& a, int m, int64_t e) {
  const float zh = load_scalar<T>(a.in[kZh][m], e);
  const float yt = load_scalar<T>(a.in[kYT][m], e);
  return fabsf(zh - yt);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

// Per-sample vector index space: modality 0's aligned vectors, then modality 1's, ...
template <int VE>
__device__ __forceinline__ int64_t sample_vectors(const ObjectiveArgs& a, int b) {
  int64_t v = 0;
  for (int m = 0; m < a.M; ++m) v += seg_geom<VE>(a.n[m], a.stride[m], b).nvec;
  return v;
}

__device__ __forceinline__ int scalar_owner(int b, int m, int M, int G) {
  return (int)(((int64_t)b * M + m) % G);
}

template <typename T, int MODE>
__device__ void phase_a(const ObjectiveArgs& a, SmemCtl& ctl, float4* slot, int b, int cta, int G) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int par = b & 1;
  const int64_t V = sample_vectors<VE>(a, b);
  const int64_t lo = V * cta / G, hi = V * (cta + 1) / G;
  const Coef k = Tr::kScm ? sample_coef(__ldg(a.t + b), a.beta, a.gamma) : Coef{};

  int64_t voff = 0;
  for (int m = 0; m < a.M; ++m) {
    float sg = 0.f, sa = 0.f, sd = 0.f;
    const SegGeom g = seg_geom<VE>(a.n[m], a.stride[m], b);
    const int64_t a0 = max(lo, voff), a1 = min(hi, voff + g.nvec);
    const int64_t ebase = g.e0 + g.head - voff * VE;  // element of vector v is ebase + v*VE
    voff += g.nvec;
    for (int64_t v = a0 + tid; v < a1; v += kThreads * kUnroll) {
      const int64_t v1 = v + kThreads;
      const bool has1 = v1 < a1;
      Loaded<T, MODE> L0, L1;
      load_vec<T, MODE>(L0, a, m, ebase + v * VE);
      if (has1) load_vec<T, MODE>(L1, a, m, ebase + v1 * VE);
      {
        float gs[VE], gd[VE];
        directions<T, MODE>(L0, k, gs, gd, sg, sa, sd);
        const int64_t pos = v - lo;
        if (pos < a.cap) {
          float4* dst = slot + pos;
          int p = 0;
          if constexpr (Tr::kScm) {
#pragma unroll
            for (int i = 0; i < VE; i += 4, ++p)
              dst[(int64_t)p * a.cap] = make_float4(gs[i], gs[i + 1], gs[i + 2], gs[i + 3]);
          }
          if constexpr (Tr::kDmd) {
#pragma unroll
            for (int i = 0; i < VE; i += 4, ++p)
              dst[(int64_t)p * a.cap] = make_float4(gd[i], gd[i + 1], gd[i + 2], gd[i + 3]);
          }
        }
      }
      if (has1) {
        float gs[VE], gd[VE];
        directions<T, MODE>(L1, k, gs, gd, sg, sa, sd);
        const int64_t pos = v1 - lo;
        if (pos < a.cap) {
          float4* dst = slot + pos;
          int p = 0;
          if constexpr (Tr::kScm) {
#pragma unroll
            for (int i = 0; i < VE; i += 4, ++p)
              dst[(int64_t)p * a.cap] = make_float4(gs[i], gs[i + 1], gs[i + 2], gs[i + 3]);
          }
          if constexpr (Tr::kDmd) {
#pragma unroll
            for (int i = 0; i < VE; i += 4, ++p)
              dst[(int64_t)p * a.cap] = make_float4(gd[i], gd[i + 1], gd[i + 2], gd[i + 3]);
          }
        }
      }
    }
    // unaligned head/tail elements of this (sample, modality): warp 0 of the owner CTA
    if (warp == 0 && cta == scalar_owner(b, m, a.M, G)) {
      int64_t e = -1;
      if (lane < g.head) e = g.e0 + lane;
      else if (lane >= 8 && lane - 8 < g.tail) e = g.e0 + g.head + g.nvec * VE + (lane - 8);
      if (e >= 0) {
        float gs = 0.f, gd = 0.f;
        direction_scalar<T, MODE>(a, m, e, k, gs, gd);
        if constexpr (Tr::kScm) sg = fmaf(gs, gs, sg);
        if constexpr (Tr::kDmd) {
          sd = fmaf(gd, gd, sd);
          sa += abs_residual_scalar<T, MODE>(a, m, e);
        }
      }
    }
    sg = warp_sum(sg);
    sa = warp_sum(sa);
    sd = warp_sum(sd);
    if (lane == 0) {
      ctl.red[par][warp][m][0] = sg;
      ctl.red[par][warp][m][1] = sa;
      ctl.red[par][warp][m][2] = sd;
    }
  }
  __syncthreads();

  // CTA sums -> workspace, then arrive on the sample's counter.
  if (warp == 0) {
    const int nq = a.M * kQuantities;
    if (tid == 0 && !ctl.checked) {
      const uint32_t magic = ld_relaxed_gpu(&a.hdr->magic);
      const uint32_t poisoned = ld_relaxed_gpu(&a.hdr->poisoned);
      ctl.timeout_ns = *reinterpret_cast<volatile uint64_t*>(&a.hdr->timeout_ns);
      ctl.checked = 1;
      if (magic != kWsMagic || poisoned != 0) {
        ctl.abort = 1;
        atomicOr(a.status, T2VA_STATUS_BAD_WORKSPACE);
      }
    }
    __syncwarp();
    const bool abort = ctl.abort != 0;
    if (!abort && lane < nq) {
      const int m = lane / kQuantities, q = lane - m * kQuantities;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += ctl.red[par][w][m][q];
      a.partials[((int64_t)(b * a.M + m) * kQuantities + q) * a.gmax + cta] = s;
      __threadfence();
    }
    __syncwarp();
    if (lane == 0 && !abort) {
      uint32_t* cnt = a.sync + (int64_t)b * 16;
      uint32_t* gen = cnt + 8;
      const uint32_t g0 = ld_relaxed_gpu(gen);
      ctl.gen_wait[par] = g0;
      __threadfence();
      const uint32_t old = atomicAdd(cnt, 1u);
      if (old == (uint32_t)(G - 1)) {
        *reinterpret_cast<volatile uint32_t*>(cnt) = 0u;
        __threadfence();
        st_release_gpu(gen, g0 + 1u);
      }
    }
  }
}

// Bounded wait for every CTA's sums of sample b, then the fixed-order merge.
template <int MODE>
__device__ bool wait_and_merge(const ObjectiveArgs& a, SmemCtl& ctl, int b, int G) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0 && !ctl.abort) {
    const uint32_t* gen = a.sync + (int64_t)b * 16 + 8;
    const uint32_t g0 = ctl.gen_wait[b & 1];
    const uint64_t start = global_timer_ns();
    while (ld_acquire_gpu(gen) == g0) {
      if (global_timer_ns() - start > ctl.timeout_ns) {
        ctl.abort = 1;
        atomicOr(a.status, T2VA_STATUS_TIMEOUT);
        atomicExch(&a.hdr->poisoned, 1u);
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (ctl.abort) return false;
  if (warp < a.M * kQuantities) {
    const int m = warp / kQuantities, q = warp - m * kQuantities;
    const float* src = a.partials + ((int64_t)(b * a.M + m) * kQuantities + q) * a.gmax;
    float s = 0.f;
    for (int i = lane; i < G; i += 32) s += __ldcg(src + i);
    s = warp_sum(s);
    if (lane == 0) ctl.tot[m][q] = s;
  }
  __syncthreads();
  return true;
}

template <typename T, int MODE>
__device__ void phase_w(const ObjectiveArgs& a, SmemCtl& ctl, const float4* slot, int b, int cta,
                        int G) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = sample_vectors<VE>(a, b);
  const int64_t lo = V * cta / G, hi = V * (cta + 1) / G;
  const Coef k = Tr::kScm ? sample_coef(__ldg(a.t + b), a.beta, a.gamma) : Coef{0, 0, 0, 0, 0, true};
  const float qnan = __int_as_float(0x7fc00000);

  int64_t voff = 0;
  for (int m = 0; m < a.M; ++m) {
    const SegGeom g = seg_geom<VE>(a.n[m], a.stride[m], b);
    // per-(sample, modality) gradient factors
    float scS = 0.f, scD = 0.f;
    if constexpr (Tr::kScm) {
      const float n = sqrtf(ctl.tot[m][0]);
      scS = 2.f * a.lam_s * a.w[m] / (k.s * (n + a.eps_s));
    }
    if constexpr (Tr::kDmd) {
      const float c = a.n[m] > 0 ? ctl.tot[m][1] / (float)a.n[m] : 0.f;
      scD = 2.f * a.lam_d * a.w[m] / (c + a.eps_d);
      if (!k.ok) scD = qnan;
    }
    const bool alias = Tr::kScm && Tr::kDmd && ((a.alias_mask >> m) & 1u);
    float* outS = a.grad_s[m];
    float* outD = a.grad_d[m];
    const int64_t a0 = max(lo, voff), a1 = min(hi, voff + g.nvec);
    const int64_t ebase = g.e0 + g.head - voff * VE;
    voff += g.nvec;
    for (int64_t v = a0 + tid; v < a1; v += kThreads * kUnroll) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t vv = v + u * kThreads;
        if (vv < a1) {
          const int64_t pos = vv - lo;
          const int64_t e = ebase + vv * VE;
          float gs[VE], gd[VE];
          if (pos < a.cap) {
            const float4* src = slot + pos;
            int p = 0;
            if constexpr (Tr::kScm) {
#pragma unroll
              for (int i = 0; i < VE; i += 4, ++p) {
                const float4 f = src[(int64_t)p * a.cap];
                gs[i] = f.x; gs[i + 1] = f.y; gs[i + 2] = f.z; gs[i + 3] = f.w;
              }
            }
            if constexpr (Tr::kDmd) {
#pragma unroll
              for (int i = 0; i < VE; i += 4, ++p) {
                const float4 f = src[(int64_t)p * a.cap];
                gd[i] = f.x; gd[i + 1] = f.y; gd[i + 2] = f.z; gd[i + 3] = f.w;
              }
            }
          } else {
            Loaded<T, MODE> L;
            load_vec<T, MODE>(L, a, m, e);
            float d0 = 0.f, d1 = 0.f, d2 = 0.f;
            directions<T, MODE>(L, k, gs, gd, d0, d1, d2);
          }
#pragma unroll
          for (int i = 0; i < VE; i += 4) {
            if (alias) {
              float4 o = make_float4(scS * gs[i] + scD * gd[i], scS * gs[i + 1] + scD * gd[i + 1],
                                     scS * gs[i + 2] + scD * gd[i + 2],
                                     scS * gs[i + 3] + scD * gd[i + 3]);
              float4* dst = reinterpret_cast<float4*>(outS + e + i);
              if (a.accumulate) {
                const float4 old = *dst;
                o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
              }
              st_stream16(dst, o);
            } else {
              if constexpr (Tr::kScm) {
                float4 o = make_float4(scS * gs[i], scS * gs[i + 1], scS * gs[i + 2], scS * gs[i + 3]);
                float4* dst = reinterpret_cast<float4*>(outS + e + i);
                if (a.accumulate) {
                  const float4 old = *dst;
                  o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
                }
                st_stream16(dst, o);
              }
              if constexpr (Tr::kDmd) {
                float4 o = make_float4(scD * gd[i], scD * gd[i + 1], scD * gd[i + 2], scD * gd[i + 3]);
                float4* dst = reinterpret_cast<float4*>(outD + e + i);
                if (a.accumulate) {
                  const float4 old = *dst;
                  o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
                }
                st_stream16(dst, o);
              }
            }
          }
        }
      }
    }
    // unaligned head/tail elements
    if (warp == 0 && cta == scalar_owner(b, m, a.M, G)) {
      int64_t e = -1;
      if (lane < g.head) e = g.e0 + lane;
      else if (lane >= 8 && lane - 8 < g.tail) e = g.e0 + g.head + g.nvec * VE + (lane - 8);
      if (e >= 0) {
        float gs = 0.f, gd = 0.f;
        direction_scalar<T, MODE>(a, m, e, k, gs, gd);
        if (alias) {
          float o = scS * gs + scD * gd;
          if (a.accumulate) o += outS[e];
          outS[e] = o;
        } else {
          if constexpr (Tr::kScm) {
            float o = scS * gs;
            if (a.accumulate) o += outS[e];
            outS[e] = o;
          }
          if constexpr (Tr::kDmd) {
            float o = scD * gd;
            if (a.accumulate) o += outD[e];
            outD[e] = o;
          }
        }
      }
    }
  }

  // per-sample outputs, written by one CTA
  if (tid == 0 && cta == (int)(b % G)) {
    float Ls = 0.f, Ld = 0.f;
    for (int m = 0; m < a.M; ++m) {
      if constexpr (Tr::kScm) {
        const float Sg = ctl.tot[m][0];
        const float n = sqrtf(Sg);
        const float d = n + a.eps_s;
        Ls += a.w[m] * (Sg / (d * d));
        if (a.norm) a.norm[(int64_t)b * a.M + m] = k.ok ? n : qnan;
      }
      if constexpr (Tr::kDmd) {
        const float c = a.n[m] > 0 ? ctl.tot[m][1] / (float)a.n[m] : 0.f;
        const float d = c + a.eps_d;
        Ld += a.w[m] * (ctl.tot[m][2] / (d * d));
        if (a.cdmd) a.cdmd[(int64_t)b * a.M + m] = k.ok ? c : qnan;
      }
    }
    Ls *= a.lam_s;
    Ld *= a.lam_d;
    if (!k.ok) {
      Ls = qnan;
      Ld = qnan;
      atomicOr(a.status, T2VA_STATUS_BAD_TIMESTEP);
    }
    a.loss[b] = (Tr::kScm ? Ls : 0.f) + (Tr::kDmd ? Ld : 0.f);
    if (a.loss_s) a.loss_s[b] = Ls;
    if (a.loss_d) a.loss_d[b] = Ld;
  }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_objective(const __grid_constant__ ObjectiveArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(smem_raw);
  float4* slots = reinterpret_cast<float4*>(smem_raw + kCtlBytes);
  using Tr = Traits<T, MODE>;
  const int64_t slot_f4 = (int64_t)a.cap * Tr::P;
  const int G = gridDim.x, cta = blockIdx.x;
  if (threadIdx.x == 0) {
    ctl.abort = 0;
    ctl.checked = 0;
  }
  __syncthreads();

  const int K = a.slots;
  for (int b = 0; b < a.B; ++b) {
    if (b >= K) __syncthreads();  // slot (b % K) was last read in W(b - K) by other threads
    phase_a<T, MODE>(a, ctl, slots + (b % K) * slot_f4, b, cta, G);
    const int wb = (K == 1) ? b : b - 1;
    if (wb >= 0) {
      if (!wait_and_merge<MODE>(a, ctl, wb, G)) return;
      phase_w<T, MODE>(a, ctl, slots + (wb % K) * slot_f4, wb, cta, G);
    }
  }
  if (K > 1 && a.B > 0) {
    const int wb = a.B - 1;
    if (!wait_and_merge<MODE>(a, ctl, wb, G)) return;
    phase_w<T, MODE>(a, ctl, slots + (wb % K) * slot_f4, wb, cta, G);
  }
}

template <typename T, int MODE>
cudaError_t launch_t(const ObjectiveArgs& a, const ObjectiveLaunch& l, cudaStream_t st) {
  auto kern = k_objective<T, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.grid);
  cfg.blockDim = dim3(l.threads);
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

__global__ void k_ws_init(uint4* ws, size_t n16, uint64_t timeout_ns, uint32_t gmax) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x)
    ws[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // block 0 also zeroed the header words above; write them after its own barrier
    WsHeader* h = reinterpret_cast<WsHeader*>(ws);
    h->timeout_ns = timeout_ns;
    h->gmax = gmax;
    h->poisoned = 0;
    __threadfence();
    h->magic = kWsMagic;
  }
}

}  // namespace

bool plan_objective(ObjectiveArgs& a, t2va_dtype dt, int mode, int sm_count, size_t smem_optin,
                    ObjectiveLaunch* out) {
  const int VE = dt == T2VA_BFLOAT16 ? 8 : 4;
  const int Q = ((mode & kModeScm) ? 1 : 0) + ((mode & kModeDmd) ? 1 : 0);
  const int P = Q * VE / 4;
  int64_t vmax = 0;
  for (int m = 0; m < a.M; ++m) vmax += (a.n[m] + VE - 1) / VE;
  int64_t G = (vmax + kThreads - 1) / kThreads;
  if (G < 1) G = 1;
  if (G > sm_count) G = sm_count;
  if (G > a.gmax) G = a.gmax;
  const int64_t per_cta = (vmax + G - 1) / G;
  const size_t bytes_per_vec = (size_t)P * 16;
  if (smem_optin <= kCtlBytes + bytes_per_vec) return false;
  const size_t budget = smem_optin - kCtlBytes;
  int slots = 1;
  int64_t cap = per_cta;
  if (a.B >= 2 && (size_t)(2 * per_cta) * bytes_per_vec <= budget) {
    slots = 2;
  } else if ((size_t)per_cta * bytes_per_vec > budget) {
    cap = (int64_t)(budget / bytes_per_vec);
  }
  if (cap < 1) cap = 1;
  a.slots = slots;
  a.cap = (int)cap;
  out->grid = (int)G;
  out->threads = kThreads;
  out->smem = kCtlBytes + (size_t)slots * cap * bytes_per_vec;
  return true;
}

cudaError_t launch_objective(const ObjectiveArgs& a, t2va_dtype dt, int mode,
                             const ObjectiveLaunch& l, cudaStream_t st) {
  if (dt == T2VA_BFLOAT16) {
    if (mode == kModeScm) return launch_t<__nv_bfloat16, kModeScm>(a, l, st);
    if (mode == kModeDmd) return launch_t<__nv_bfloat16, kModeDmd>(a, l, st);
    return launch_t<__nv_bfloat16, kModeStage3>(a, l, st);
  }
  if (mode == kModeScm) return launch_t<float, kModeScm>(a, l, st);
  if (mode == kModeDmd) return launch_t<float, kModeDmd>(a, l, st);
  return launch_t<float, kModeStage3>(a, l, st);
}

cudaError_t launch_workspace_init(void* ws, size_t bytes, uint64_t timeout_ns, uint32_t gmax,
                                  cudaStream_t st) {
  const size_t n16 = bytes / 16;
  int blocks = (int)((n16 + 255) / 256);
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  k_ws_init<<<blocks, 256, 0, st>>>(reinterpret_cast<uint4*>(ws), n16, timeout_ns, gmax);
  return cudaGetLastError();
}

}  // namespace t2va
