// Joint sCM / DMD / stage-3 objective kernels (TurboT2VA, robotworld.top/zh reading:
// section 3.1 joint sCM, section 四 joint DMD, section 4.1 stage-3 sum;
// robotworld.top/en summary: Eq. 6 and Eq. 11-12).
//
// The gradient of every (sample, modality) needs that row's norms, which need all of
// the row's elements, so the objective is two passes over the inputs, as two kernels
// on the caller's stream; the kernel boundary is the only grid-wide barrier:
//
//   k_sums  : every (sample, modality) row is cut into chunks of `vpc` 16-byte
//             vectors, one CTA per chunk (rows of every sample and modality in one
//             grid, so the small audio rows share the GPU with the video rows). Each
//             thread keeps the loads of two of its vectors in flight, computes the float32
//             directions g_sCM and g_DMD and accumulates sum g_sCM^2, sum |zhat0 - y_T|
//             and sum g_DMD^2; the CTA adds them in a fixed order and writes the
//             chunk's three partial sums to the workspace. The loads ask L2 to keep
//             the inputs. Before its dependency wait each CTA already requests the
//             first vectors of its chunk into L2 (a bulk prefetch per input).
//   k_grads : the same chunks. Each CTA starts the loads of its vectors again, except
//             zhat0 (L2 hits; L2 may drop them now), adds the row's partial sums in chunk order
//             (every CTA of a row gets bit-identical totals), derives the gradient
//             factors, recomputes the directions and writes the float32 gradients
//             once. The sample's chunk with the fewest vectors also writes the
//             per-sample outputs.
//
// HBM sees each input read once and each gradient written once when a call's inputs
// fit in L2 (126 MB on B300; the stage-3 512x768 batch of 4 reads 45 MB); larger
// calls read the inputs twice. There is no cross-CTA wait, so nothing can hang.
#include <algorithm>

#include "t2va_internal.cuh"

namespace t2va {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 2;                    // vectors per thread per batch
constexpr int kBatchVec = kThreads * kPerThread;  // vectors per CTA per batch
constexpr int64_t kMaxWaveVec = 2048;             // longest chunk of a one-wave plan
// Vectors at the start of a chunk that k_sums prefetches into L2 before its dependency
// wait, per input. Measured on B300 with caps of 192 to 384 vectors and with 1/8 to all of
// the chunk: 256 to 320 is best at every stage-3 shape tried; prefetching more, or one
// batch ahead inside the loop as well, loses. The sCM objective alone (four inputs) is
// best at 384: 10.76 against 10.90 us per 512x768 call with 320.
constexpr int64_t kEarlyVec = 320;
constexpr int64_t kEarlyVecScmOnly = 384;

template <typename T, int MODE>
struct Traits {
  static constexpr int VE = Vec<T>::VE;
  static constexpr bool kScm = (MODE & kModeScm) != 0;
  static constexpr bool kDmd = (MODE & kModeDmd) != 0;
  static constexpr bool kCfg = kDmd && (MODE & kModeCfg) != 0;
  static constexpr int k0 = kScm ? kZt : kZh;  // first input slot of the mode
  static constexpr int NIN = (kScm ? 4 : 0) + (kDmd ? 3 : 0) + (kCfg ? 1 : 0);
  // the gradient pass needs no zhat0 (it enters only the residual scale)
  static constexpr int NG = (kScm ? 4 : 0) + (kDmd ? 2 : 0) + (kCfg ? 1 : 0);
  static constexpr int kYT0 = kScm ? 4 : 0;  // position of y_T among the gradient inputs
  // resident gradient-pass CTAs per SM: three, as for the first pass, so one balanced
  // wave of chunks is one wave of both kernels
  static constexpr int kGradCtas = 3;
  // the guided stage-3 gradient pass keeps one vector per thread in flight: its seven
  // inputs spilled 96 bytes at two within 80 registers; with one it needs 72 and ran 18.0
  // instead of 18.8 us per 512x768 call on B300
  static constexpr bool kGradOneOnly = kCfg;
};

// The teacher prediction at the re-noised sample: the stored one, or with guidance
// the unconditional prediction moved s times the way to the conditional one,
// u + s (k - u), in float32 with one fma.
template <bool CFG>
__device__ __forceinline__ float teacher(float k, float u, float s) {
  if constexpr (CFG) return fmaf(s, k - u, u);
  return k;
}

// ---------------------------------------------------------------------------
// loads, cache policies, reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte streaming load through the read-only path, not kept in L1, with an L2
// eviction policy.
__device__ __forceinline__ uint4 ld16(const void* p, uint64_t policy) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(policy));
  return r;
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned start) into L2 with an
// eviction policy. It returns no data, so it may run before a dependency wait: L2 is
// the point of coherence, and a later load still sees what the previous kernel wrote.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes),
               "l"(policy)
               : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

// Sum of the CTA's three values in a fixed order: lanes, then warps. Every thread
// gets the result.
__device__ __forceinline__ float3 block_sum3(float a, float b, float c, float3 (&scratch)[kWarps]) {
  a = warp_sum(a);
  b = warp_sum(b);
  c = warp_sum(c);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) scratch[warp] = make_float3(a, b, c);
  __syncthreads();
  float3 t = make_float3(0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    t.x += scratch[w].x;
    t.y += scratch[w].y;
    t.z += scratch[w].z;
  }
  __syncthreads();  // scratch may be reused
  return t;
}

// ---------------------------------------------------------------------------
// chunks
// ---------------------------------------------------------------------------

// Chunk `blk`: sample b, modality m, chunk c of row (b, m), and the row's vectors
// [v_lo, v_hi) that it owns (aligned vectors of the segment; element 0 of vector 0
// is e_vec0).
struct Chunk {
  int b, m, c;
  int64_t e_vec0, v_lo, v_hi;
  SegGeom g;
};

template <int VE>
__device__ __forceinline__ Chunk chunk_of(const ObjectiveArgs& a, int blk) {
  Chunk k;
  const int cps = a.choff[a.M];  // chunks per sample
  k.b = blk / cps;
  const int local = blk - k.b * cps;
  k.m = 0;
#pragma unroll
  for (int i = 1; i < kMaxM; ++i)
    if (i < a.M && local >= a.choff[i]) k.m = i;
  k.c = local - a.choff[k.m];
  k.g = seg_geom<VE>(a.n[k.m], a.stride[k.m], k.b);
  k.e_vec0 = k.g.e0 + k.g.head;
  k.v_lo = (int64_t)k.c * a.vpc;
  k.v_hi = min(k.v_lo + (int64_t)a.vpc, k.g.nvec);
  return k;
}

__device__ __forceinline__ float4* row_partials(const ObjectiveArgs& a, int b, int m) {
  return reinterpret_cast<float4*>(a.partials) + ((int64_t)b * a.M + m) * kMaxChunks;
}

// The unaligned head (chunk 0) and tail (last chunk) elements of a row: at most 7 of
// each, one per thread: threads 0-6 take the head, threads 32-38 the tail.
template <int VE>
__device__ __forceinline__ int64_t edge_element(const ObjectiveArgs& a, const Chunk& k) {
  const int t = threadIdx.x;
  if (k.c == 0 && t < k.g.head) return k.g.e0 + t;
  if (k.c == a.nchunk[k.m] - 1 && t >= 32 && t - 32 < k.g.tail)
    return k.g.e0 + k.g.head + k.g.nvec * VE + (t - 32);
  return -1;
}

// ---------------------------------------------------------------------------
// per-vector arithmetic
// ---------------------------------------------------------------------------

struct Coefs {
  float kD, kz, kx, s;
  bool ok;
  float cfg;  // guidance scale of the row's modality (kModeCfg)
};

template <typename T, int MODE>
__device__ __forceinline__ Coefs coefs_of(const ObjectiveArgs& a, int b, int m) {
  Coefs c{0.f, 0.f, 0.f, 1.f, true, 1.f};
  if constexpr (Traits<T, MODE>::kScm) {
    const Coef k = sample_coef(__ldg(a.t + b), a.beta, a.gamma);
    c = Coefs{k.kD, k.kz, k.kx, k.s, k.ok, 1.f};
  }
  if constexpr (Traits<T, MODE>::kCfg) c.cfg = a.cfg[m];
  return c;
}

template <typename T, int MODE>
__device__ __forceinline__ void load_vec(uint4 (&in)[Traits<T, MODE>::NIN], const ObjectiveArgs& a,
                                         int m, int64_t e, uint64_t policy) {
  using Tr = Traits<T, MODE>;
#pragma unroll
  for (int q = 0; q < Tr::NIN; ++q)
    in[q] = ld16(reinterpret_cast<const T*>(a.in[Tr::k0 + q][m]) + e, policy);
}

// The directions of one vector from its inputs (raw 16-byte chunks, in input order
// starting at Traits::k0), and its three sums.
template <typename T, int MODE>
__device__ __forceinline__ void directions(const uint4 (&in)[Traits<T, MODE>::NIN], const Coefs& k,
                                           float* gs, float* gd, float& sg, float& sa, float& sd) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  if constexpr (Tr::kScm) {
    Vec<T> z, xt, xs, xd;
    z.from(in[kZt - Tr::k0]);
    xt.from(in[kXT - Tr::k0]);
    xs.from(in[kXS - Tr::k0]);
    xd.from(in[kXdot - Tr::k0]);
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      const float g = fmaf(k.kD, xt.v[i] - xs.v[i], fmaf(k.kz, z.v[i], k.kx * xd.v[i]));
      gs[i] = g;
      sg = fmaf(g, g, sg);
    }
  }
  if constexpr (Tr::kDmd) {
    Vec<T> zh, yt, yf, yu;
    zh.from(in[kZh - Tr::k0]);
    yt.from(in[kYT - Tr::k0]);
    yf.from(in[kYF - Tr::k0]);
    if constexpr (Tr::kCfg) yu.from(in[kYU - Tr::k0]);
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      const float y = teacher<Tr::kCfg>(yt.v[i], Tr::kCfg ? yu.v[i] : 0.f, k.cfg);
      const float g = yf.v[i] - y;
      gd[i] = g;
      sd = fmaf(g, g, sd);
      sa += fabsf(zh.v[i] - y);
    }
  }
}

// The gradient pass's inputs of one vector: the sCM inputs, then y_T and y_fake.
template <typename T, int MODE>
__device__ __forceinline__ void load_grad_vec(uint4 (&in)[Traits<T, MODE>::NG], const ObjectiveArgs& a,
                                              int m, int64_t e, uint64_t policy) {
  using Tr = Traits<T, MODE>;
  if constexpr (Tr::kScm) {
#pragma unroll
    for (int q = 0; q < 4; ++q) in[q] = ld16(reinterpret_cast<const T*>(a.in[kZt + q][m]) + e, policy);
  }
  if constexpr (Tr::kDmd) {
    in[Tr::kYT0] = ld16(reinterpret_cast<const T*>(a.in[kYT][m]) + e, policy);
    in[Tr::kYT0 + 1] = ld16(reinterpret_cast<const T*>(a.in[kYF][m]) + e, policy);
  }
  if constexpr (Tr::kCfg)
    in[Tr::kYT0 + 2] = ld16(reinterpret_cast<const T*>(a.in[kYU][m]) + e, policy);
}

// The unscaled directions of one vector from the gradient pass's inputs.
template <typename T, int MODE>
__device__ __forceinline__ void grad_directions(const uint4 (&in)[Traits<T, MODE>::NG],
                                                const Coefs& k, float* gs, float* gd) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  if constexpr (Tr::kScm) {
    Vec<T> z, xt, xs, xd;
    z.from(in[0]);
    xt.from(in[1]);
    xs.from(in[2]);
    xd.from(in[3]);
#pragma unroll
    for (int i = 0; i < VE; ++i)
      gs[i] = fmaf(k.kD, xt.v[i] - xs.v[i], fmaf(k.kz, z.v[i], k.kx * xd.v[i]));
  }
  if constexpr (Tr::kDmd) {
    Vec<T> yt, yf, yu;
    yt.from(in[Tr::kYT0]);
    yf.from(in[Tr::kYT0 + 1]);
    if constexpr (Tr::kCfg) yu.from(in[Tr::kYT0 + 2]);
#pragma unroll
    for (int i = 0; i < VE; ++i)
      gd[i] = yf.v[i] - teacher<Tr::kCfg>(yt.v[i], Tr::kCfg ? yu.v[i] : 0.f, k.cfg);
  }
}

template <typename T, int MODE>
__device__ __forceinline__ void scalar_direction(const ObjectiveArgs& a, int m, int64_t e,
                                                 const Coefs& k, float& gs, float& gd,
                                                 float& sabs) {
  using Tr = Traits<T, MODE>;
  if constexpr (Tr::kScm) {
    const float z = load_scalar<T>(a.in[kZt][m], e);
    const float xt = load_scalar<T>(a.in[kXT][m], e);
    const float xs = load_scalar<T>(a.in[kXS][m], e);
    const float xd = load_scalar<T>(a.in[kXdot][m], e);
    gs = fmaf(k.kD, xt - xs, fmaf(k.kz, z, k.kx * xd));
  }
  if constexpr (Tr::kDmd) {
    const float zh = load_scalar<T>(a.in[kZh][m], e);
    const float yu = Tr::kCfg ? load_scalar<T>(a.in[kYU][m], e) : 0.f;
    const float yt = teacher<Tr::kCfg>(load_scalar<T>(a.in[kYT][m], e), yu, k.cfg);
    const float yf = load_scalar<T>(a.in[kYF][m], e);
    gd = yf - yt;
    sabs = fabsf(zh - yt);
  }
}

// Eight consecutive gradients (32 bytes, 32-byte aligned) in one store, so every
// store instruction of a warp writes whole 32-byte sectors. The lines are marked first
// to leave L2 (the gradients are not read again here), which keeps the inputs that the
// second pass re-reads resident; measured faster than a streaming (.cs) store.
__device__ __forceinline__ void write8(float* dst, const float* v, int accumulate) {
  float o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = v[i];
  if (accumulate) {
    const float4* d = reinterpret_cast<const float4*>(dst);
    const float4 a0 = d[0], a1 = d[1];
    o[0] += a0.x; o[1] += a0.y; o[2] += a0.z; o[3] += a0.w;
    o[4] += a1.x; o[5] += a1.y; o[6] += a1.z; o[7] += a1.w;
  }
  asm volatile("st.global.L2::cache_hint.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(dst),
               "f"(o[0]), "f"(o[1]), "f"(o[2]), "f"(o[3]), "f"(o[4]), "f"(o[5]), "f"(o[6]), "f"(o[7]),
               "l"(policy_evict_first())
               : "memory");
}

__device__ __forceinline__ void write4(float* dst, const float* v, int accumulate) {
  float4 o = make_float4(v[0], v[1], v[2], v[3]);
  if (accumulate) {
    const float4 old = *reinterpret_cast<const float4*>(dst);
    o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
  }
  st_stream16(dst, o);
}

template <int VE>
__device__ __forceinline__ void write_run(float* dst, const float* v, bool wide, int accumulate) {
  if constexpr (VE == 8) {
    if (wide) {
      write8(dst, v, accumulate);
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < VE; i += 4) write4(dst + i, v + i, accumulate);
}

template <typename T, int MODE>
__device__ __forceinline__ void write_vec(const ObjectiveArgs& a, int m, int64_t e, float scS,
                                          float scD, const float* gs, const float* gd) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  const bool wide = (a.wide_mask >> m) & 1u;
  float o[VE];
  if (Tr::kScm && Tr::kDmd && ((a.alias_mask >> m) & 1u)) {
#pragma unroll
    for (int i = 0; i < VE; ++i) o[i] = scS * gs[i] + scD * gd[i];
    write_run<VE>(a.grad_s[m] + e, o, wide, a.accumulate);
    return;
  }
  if constexpr (Tr::kScm) {
#pragma unroll
    for (int i = 0; i < VE; ++i) o[i] = scS * gs[i];
    write_run<VE>(a.grad_s[m] + e, o, wide, a.accumulate);
  }
  if constexpr (Tr::kDmd) {
#pragma unroll
    for (int i = 0; i < VE; ++i) o[i] = scD * gd[i];
    write_run<VE>(a.grad_d[m] + e, o, wide, a.accumulate);
  }
}

__device__ __forceinline__ void write1(float* dst, float v, int accumulate) {
  if (accumulate) v += *dst;
  *dst = v;
}

// ---------------------------------------------------------------------------
// pass 1: partial sums per chunk
// ---------------------------------------------------------------------------

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, 3) k_sums(const __grid_constant__ ObjectiveArgs a) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  __shared__ float3 scratch[kWarps];
  const Chunk k = chunk_of<VE>(a, blockIdx.x);
  const uint64_t keep = policy_evict_last();
  // The HBM stream starts while the previous kernel drains: thread q asks L2 for the
  // chunk's first kEarlyVec vectors of input q. (Only a prefetch may run this early.)
  if (threadIdx.x < Tr::NIN && k.v_hi > k.v_lo) {
    const int64_t nv = min(k.v_hi - k.v_lo, Tr::kDmd ? kEarlyVec : kEarlyVecScmOnly);
    prefetch_l2(reinterpret_cast<const T*>(a.in[Tr::k0 + threadIdx.x][k.m]) + k.e_vec0 + k.v_lo * VE,
                (uint32_t)(nv * 16), keep);
  }
  // launched as a programmatic dependent of the previous kernel on the stream: no
  // load before that kernel has finished; the next kernel (k_grads) may launch once
  // every CTA of this one is past this point
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const Coefs cf = coefs_of<T, MODE>(a, k.b, k.m);
  // Thread t takes vectors t, t + 256, t + 512, ... of the chunk with two of them in
  // flight (buffers A and B): while it forms the directions of one, the next one's loads
  // are out, and a buffer takes the loads of the vector two steps ahead as soon as its
  // own vector is done.
  float sg = 0.f, sa = 0.f, sd = 0.f;
  uint4 A[Tr::NIN], B[Tr::NIN];
  int64_t v = k.v_lo + threadIdx.x;
  if (v < k.v_hi) load_vec<T, MODE>(A, a, k.m, k.e_vec0 + v * VE, keep);
  if (v + kThreads < k.v_hi) load_vec<T, MODE>(B, a, k.m, k.e_vec0 + (v + kThreads) * VE, keep);
  for (; v < k.v_hi; v += 2 * kThreads) {
    const int64_t v1 = v + kThreads, v2 = v + 2 * kThreads, v3 = v + 3 * kThreads;
    {
      float gs[VE], gd[VE];
      directions<T, MODE>(A, cf, gs, gd, sg, sa, sd);
    }
    if (v2 < k.v_hi) load_vec<T, MODE>(A, a, k.m, k.e_vec0 + v2 * VE, keep);
    if (v1 < k.v_hi) {
      float gs[VE], gd[VE];
      directions<T, MODE>(B, cf, gs, gd, sg, sa, sd);
    }
    if (v3 < k.v_hi) load_vec<T, MODE>(B, a, k.m, k.e_vec0 + v3 * VE, keep);
  }
  const int64_t e = edge_element<VE>(a, k);
  if (e >= 0) {
    float gs = 0.f, gd = 0.f, sabs = 0.f;
    scalar_direction<T, MODE>(a, k.m, e, cf, gs, gd, sabs);
    sg = fmaf(gs, gs, sg);
    sa += sabs;
    sd = fmaf(gd, gd, sd);
  }
  const float3 t = block_sum3(sg, sa, sd, scratch);
  if (threadIdx.x == 0) row_partials(a, k.b, k.m)[k.c] = make_float4(t.x, t.y, t.z, 0.f);
}

// ---------------------------------------------------------------------------
// pass 2: totals, gradients, per-sample outputs
// ---------------------------------------------------------------------------

// Totals of row (b, m): the chunks' partial sums added in a fixed order (thread t
// takes chunks t, t + 256, ...; then lanes; then warps), so every CTA of the row
// gets the same bits. A thread's loads go two at a time, both in flight before it adds.
__device__ __forceinline__ float3 row_totals(const ObjectiveArgs& a, int b, int m,
                                             float3 (&scratch)[kWarps]) {
  const float4* p = row_partials(a, b, m);
  const int n = a.nchunk[m];
  float x = 0.f, y = 0.f, z = 0.f;
#pragma unroll 1
  for (int c0 = threadIdx.x; c0 < n; c0 += 2 * kThreads) {
    const int c1 = c0 + kThreads;
    const float4 v0 = __ldcg(p + c0);
    const float4 v1 = c1 < n ? __ldcg(p + c1) : make_float4(0.f, 0.f, 0.f, 0.f);
    x += v0.x;
    y += v0.y;
    z += v0.z;
    if (c1 < n) {
      x += v1.x;
      y += v1.y;
      z += v1.z;
    }
  }
  return block_sum3(x, y, z, scratch);
}

// PER: vectors per thread in flight (the plan's choice; see plan_objective).
template <typename T, int MODE, int PER>
__global__ void __launch_bounds__(kThreads, Traits<T, MODE>::kGradCtas)
    k_grads(const __grid_constant__ ObjectiveArgs a) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  constexpr int kGradBatch = kThreads * PER;
  __shared__ float3 scratch[kWarps];
  const Chunk k = chunk_of<VE>(a, blockIdx.x);
  const Coefs cf = coefs_of<T, MODE>(a, k.b, k.m);
  const uint64_t drop = policy_evict_first();
  const float qnan = __int_as_float(0x7fc00000);

  // the first batch's loads (served by L2) are in flight while the totals are read
  uint4 in[PER][Tr::NG];
  int64_t base = k.v_lo;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int64_t v = base + u * kThreads + threadIdx.x;
    if (v < k.v_hi) load_grad_vec<T, MODE>(in[u], a, k.m, k.e_vec0 + v * VE, drop);
  }

  // The inputs were complete before k_sums read them (every CTA of k_sums waited for
  // its predecessor before this kernel could launch), so the loads above may run
  // ahead; the partial sums of k_sums may not be read before it has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const float3 tot = row_totals(a, k.b, k.m, scratch);
  const float n = sqrtf(tot.x);
  const float scS = Tr::kScm ? 2.f * a.lam_s * a.w[k.m] / (cf.s * (n + a.eps_s)) : 0.f;
  const float c_dmd = a.n[k.m] > 0 ? tot.y / (float)a.n[k.m] : 0.f;
  const float scD = Tr::kDmd ? (cf.ok ? 2.f * a.lam_d * a.w[k.m] / (c_dmd + a.eps_d) : qnan) : 0.f;

  for (;;) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int64_t v = base + u * kThreads + threadIdx.x;
      if (v < k.v_hi) {
        float gs[VE], gd[VE];
        grad_directions<T, MODE>(in[u], cf, gs, gd);
        write_vec<T, MODE>(a, k.m, k.e_vec0 + v * VE, scS, scD, gs, gd);
      }
    }
    base += kGradBatch;
    if (base >= k.v_hi) break;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int64_t v = base + u * kThreads + threadIdx.x;
      if (v < k.v_hi) load_grad_vec<T, MODE>(in[u], a, k.m, k.e_vec0 + v * VE, drop);
    }
  }

  const int64_t e = edge_element<VE>(a, k);
  if (e >= 0) {
    float gs = 0.f, gd = 0.f, sabs = 0.f;
    scalar_direction<T, MODE>(a, k.m, e, cf, gs, gd, sabs);
    if (Tr::kScm && Tr::kDmd && ((a.alias_mask >> k.m) & 1u)) {
      write1(a.grad_s[k.m] + e, scS * gs + scD * gd, a.accumulate);
    } else {
      if constexpr (Tr::kScm) write1(a.grad_s[k.m] + e, scS * gs, a.accumulate);
      if constexpr (Tr::kDmd) write1(a.grad_d[k.m] + e, scD * gd, a.accumulate);
    }
  }

  // per-sample outputs: by the sample's chunk with the fewest vectors (chunk out_c of
  // modality out_m, chosen by the plan; it has time to spare), from the totals of all
  // its modalities (added in the same order as everywhere else)
  if (k.m == a.out_m && k.c == a.out_c) {
    float Ls = 0.f, Ld = 0.f;
    for (int m = 0; m < a.M; ++m) {
      const float3 tm = m == k.m ? tot : row_totals(a, k.b, m, scratch);
      if (threadIdx.x == 0) {
        if constexpr (Tr::kScm) {
          const float nm = sqrtf(tm.x);
          const float d = nm + a.eps_s;
          Ls += a.w[m] * (tm.x / (d * d));
          if (a.norm) a.norm[(int64_t)k.b * a.M + m] = cf.ok ? nm : qnan;
        }
        if constexpr (Tr::kDmd) {
          const float c = a.n[m] > 0 ? tm.y / (float)a.n[m] : 0.f;
          const float d = c + a.eps_d;
          Ld += a.w[m] * (tm.z / (d * d));
          if (a.cdmd) a.cdmd[(int64_t)k.b * a.M + m] = cf.ok ? c : qnan;
        }
      }
    }
    if (threadIdx.x == 0) {
      Ls *= a.lam_s;
      Ld *= a.lam_d;
      if (!cf.ok) {
        Ls = qnan;
        Ld = qnan;
        atomicOr(a.status, T2VA_STATUS_BAD_TIMESTEP);
      }
      a.loss[k.b] = (Tr::kScm ? Ls : 0.f) + (Tr::kDmd ? Ld : 0.f);
      if (a.loss_s) a.loss_s[k.b] = Ls;
      if (a.loss_d) a.loss_d[k.b] = Ld;
    }
  }
}

// Launch as a programmatic dependent of the previous work on the stream: the kernel
// may be scheduled while that work drains, and waits for it (griddepcontrol.wait)
// before touching memory that work could have written.
template <typename K>
cudaError_t launch_pdl(K kern, int grid, cudaStream_t st, const ObjectiveArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int MODE>
cudaError_t launch_t(const ObjectiveArgs& a, const ObjectiveLaunch& l, cudaStream_t st) {
  cudaError_t e = launch_pdl(k_sums<T, MODE>, l.grid, st, a);
  if (e != cudaSuccess) return e;
  if constexpr (Traits<T, MODE>::kGradOneOnly) {
    return launch_pdl(k_grads<T, MODE, 1>, l.grid, st, a);
  } else {
    if (l.grad_per == 1) return launch_pdl(k_grads<T, MODE, 1>, l.grid, st, a);
    return launch_pdl(k_grads<T, MODE, 2>, l.grid, st, a);
  }
}

__global__ void k_ws_init(uint4* ws, size_t n16) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x)
    ws[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // block 0 zeroed the header above; write its magic after that block's barrier
  if (blockIdx.x == 0 && threadIdx.x == 0) reinterpret_cast<WsHeader*>(ws)->magic = kWsMagic;
}

}  // namespace

bool plan_objective(ObjectiveArgs& a, t2va_dtype dt, int sm_count, ObjectiveLaunch* out) {
  const int VE = dt == T2VA_BFLOAT16 ? 8 : 4;
  int64_t nvec_max = 0, grid1 = 0, total = 0;
  for (int m = 0; m < a.M; ++m) {
    const int64_t nv = (a.n[m] + VE - 1) / VE;
    nvec_max = std::max<int64_t>(nvec_max, nv);
    grid1 += std::max<int64_t>(1, (nv + kBatchVec - 1) / kBatchVec);
    total += nv;
  }
  grid1 *= a.B;
  total *= a.B;
  const int64_t sms = std::max(1, sm_count);
  const int64_t resident = 3 * sms;
  // A one-wave plan leaves about one slot in 28 free (16 of 444 on B300): the CTAs of
  // the next kernel on the stream, or of a kernel on another stream, start there while
  // this one drains. Measured on B300 against a full wave: the stage-3 512x768 step with
  // the next steps' noising beside it 21.07 -> 20.78 us, the objective alone 15.88 ->
  // 15.93 us (512x768) and 19.02 -> 18.96 us (1024x1792); 24 to 72 free slots helped the
  // step more but cost the objective 0.2 to 1.4 us.
  const int64_t wave = resident - sms / 9;
  if (total <= wave * kMaxWaveVec) {
    // One balanced wave: the shortest chunk (a multiple of 32 vectors) that gives at most
    // `wave` CTAs, so the SMs get nearly equal chunks, three on most of them (measured on
    // B300: 1024x1792 batch 1 23.2 -> 21.3 us; 512x768 batch 4 18.3).
    int64_t vpc = std::max<int64_t>(32, ((total + wave - 1) / wave + 31) / 32 * 32);
    for (;;) {
      int64_t g = 0;
      for (int m = 0; m < a.M; ++m)
        g += std::max<int64_t>(1, ((a.n[m] + VE - 1) / VE + vpc - 1) / vpc);
      if (a.B * g <= wave || vpc >= kMaxWaveVec) break;
      vpc += 32;
    }
    a.vpc = (int)vpc;
  } else {
    // Several waves: chunks of one batch of the CTA, or two when a one-batch grid would
    // need between one and four waves (each CTA's fixed costs then cover twice the
    // work); more if a row would need more chunks than the workspace holds.
    const int64_t wanted = (grid1 > resident && grid1 <= 4 * resident) ? 2 : 1;
    const int64_t batches = std::max<int64_t>(
        wanted, (nvec_max + (int64_t)kBatchVec * kMaxChunks - 1) / ((int64_t)kBatchVec * kMaxChunks));
    if (batches > INT32_MAX / kBatchVec) return false;
    a.vpc = (int)(batches * kBatchVec);
  }
  int acc = 0;
  int64_t fewest = INT64_MAX;
  for (int m = 0; m < a.M; ++m) {
    const int64_t nvec_ub = (a.n[m] + VE - 1) / VE;
    const int64_t c = std::max<int64_t>(1, (nvec_ub + a.vpc - 1) / a.vpc);  // >= 1: edges
    a.nchunk[m] = (int)c;
    a.choff[m] = acc;
    acc += (int)c;
    // the per-sample outputs go to the row's last (shortest) chunk with the fewest vectors
    const int64_t last = nvec_ub - (c - 1) * a.vpc;
    if (last < fewest) {
      fewest = last;
      a.out_m = m;
      a.out_c = (int)c - 1;
    }
  }
  for (int m = a.M; m <= kMaxM; ++m) a.choff[m] = acc;
  const int64_t grid = (int64_t)a.B * acc;
  if (grid > INT32_MAX) return false;
  out->grid = (int)grid;
  out->threads = kThreads;
  out->smem = 0;
  // Two vectors per thread in flight in the gradient pass when the call is one wave of
  // chunks longer than a vector per thread; one otherwise: with inputs beyond L2 the pass
  // re-reads them from HBM, and at one vector a thread needs about 63 registers, so four
  // CTAs fit on an SM where the later waves run. Measured on B300 (per call): 512x768
  // batch 4 15.9 us with two against 16.8 with one, 1024x1792 18.9 against 19.5; the
  // batch-16 sweep shape (multi-wave) 70.5 with one against 71.7, batch 1 7.40 against 7.56.
  out->grad_per = (grid <= wave && a.vpc > kThreads) ? 2 : 1;
  return true;
}

cudaError_t launch_objective(const ObjectiveArgs& a, t2va_dtype dt, int mode,
                             const ObjectiveLaunch& l, cudaStream_t st) {
  constexpr int kCfg3 = kModeStage3 | kModeCfg;
  if (dt == T2VA_BFLOAT16) {
    if (mode == kModeScm) return launch_t<__nv_bfloat16, kModeScm>(a, l, st);
    if (mode == kModeDmd) return launch_t<__nv_bfloat16, kModeDmd>(a, l, st);
    if (mode == kCfg3) return launch_t<__nv_bfloat16, kCfg3>(a, l, st);
    return launch_t<__nv_bfloat16, kModeStage3>(a, l, st);
  }
  if (mode == kModeScm) return launch_t<float, kModeScm>(a, l, st);
  if (mode == kModeDmd) return launch_t<float, kModeDmd>(a, l, st);
  if (mode == kCfg3) return launch_t<float, kCfg3>(a, l, st);
  return launch_t<float, kModeStage3>(a, l, st);
}

cudaError_t launch_workspace_init(void* ws, size_t bytes, cudaStream_t st) {
  const size_t n16 = bytes / 16;
  int blocks = (int)std::min<size_t>(1024, std::max<size_t>(1, (n16 + 255) / 256));
  k_ws_init<<<blocks, 256, 0, st>>>(reinterpret_cast<uint4*>(ws), n16);
  return cudaGetLastError();
}

}  // namespace t2va
