// Fused joint sCM / DMD / stage-3 objective kernel (TurboT2VA, robotworld.top/zh
// reading: section 3.1 joint sCM, section 四 joint DMD, section 4.1 stage-3 sum;
// robotworld.top/en summary: Eq. 6 and Eq. 11-12).
//
// Design (one persistent cooperative launch, one CTA of 512 threads per SM):
//   Every (sample, modality) segment is cut into G equal chunks of 16-byte vectors,
//   one per CTA, so each segment is spread over the whole GPU and the small audio
//   segment never leaves SMs idle. Inside a CTA, the chunks of one sample are laid
//   end to end in a "slot" range (each modality's chunk padded to a multiple of 32,
//   so a warp's 32 consecutive slots always belong to one modality); thread t owns
//   slots t, t + 512, ... of every sample. Samples are processed in rounds of `spr`:
//   A(r): stream the round's inputs once with 16-byte loads, keeping the next slot's
//     loads in flight while the current slot is computed (also across sample and
//     round boundaries). Compute the float32 directions g_sCM and g_DMD, keep them in
//     shared memory, and accumulate per-(sample, modality) sums of g_sCM^2,
//     |zhat0 - y_T| and g_DMD^2 per warp. The CTA then publishes its sums as 64-bit
//     words tagged with the call's epoch.
//   Merge(r): every CTA reads all CTAs' words of the round in parallel, waiting (with
//     a time limit) until every word carries this call's epoch, and adds them in a
//     fixed order: every CTA gets bit-identical totals, run to run.
//   W(r): scale the kept directions by the per-(sample, modality) factors and write
//     the float32 gradients once.
//   When all samples fit in shared memory there is one round (A, merge, W). Otherwise
//   rounds alternate between two shared-memory groups in the order A0 A1 W0 A2 W1 ...
//   so each merge is waited for behind the next round's reads. Slots that do not fit
//   in shared memory (one sample larger than the GPU's shared memory) are recomputed
//   from the inputs in W.
// HBM traffic is the algorithmic minimum whenever one sample's directions fit on
// chip: each input read once, each gradient written once. The epoch tags replace
// arrival counters, so nothing needs resetting between calls.
#include <algorithm>

#include "t2va_internal.cuh"

namespace t2va {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRound = 8;          // samples per round
constexpr uint32_t kNoWithhold = 0xFFFFFFFFu;

struct RoundCoef {
  float kD, kz, kx, s;
  int ok;
};

struct SmemCtl {
  float red[kWarps][kMaxRound][kMaxM][kQuantities];  // per-warp sums of the current round
  float scal[kMaxRound][kMaxM][kQuantities];         // unaligned head/tail sums (CTA G-1)
  float tot[2][kMaxRound][kMaxM][kQuantities];       // merged totals of a round
  float scaleS[2][kMaxRound][kMaxM];
  float scaleD[2][kMaxRound][kMaxM];
  RoundCoef coef[2][kMaxRound];
  uint64_t timeout_ns;
  uint32_t epoch;
  uint32_t withhold;
  int abort;
};
constexpr size_t kCtlBytes = (sizeof(SmemCtl) + 15) / 16 * 16;

template <typename T, int MODE>
struct Traits {
  static constexpr int VE = Vec<T>::VE;
  static constexpr bool kScm = (MODE & kModeScm) != 0;
  static constexpr bool kDmd = (MODE & kModeDmd) != 0;
  // float4 pieces of kept direction per vector
  static constexpr int kPieces = ((kScm ? 1 : 0) + (kDmd ? 1 : 0)) * VE / 4;
};

template <typename T, int MODE>
struct Loaded {
  uint4 r[kNumInputs];
};

// ---------------------------------------------------------------------------
// epoch-tagged partial sums
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_word(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t pack_word(float v, uint32_t epoch) {
  return ((uint64_t)epoch << 32) | (uint64_t)__float_as_uint(v);
}

// ---------------------------------------------------------------------------
// per-vector arithmetic
// ---------------------------------------------------------------------------

template <typename T, int MODE>
__device__ __forceinline__ void load_vec(Loaded<T, MODE>& L, const ObjectiveArgs& a, int m,
                                         int64_t e) {
  using Tr = Traits<T, MODE>;
  if constexpr (Tr::kScm) {
    L.r[kZt] = ld_stream16(reinterpret_cast<const T*>(a.in[kZt][m]) + e);
    L.r[kXT] = ld_stream16(reinterpret_cast<const T*>(a.in[kXT][m]) + e);
    L.r[kXS] = ld_stream16(reinterpret_cast<const T*>(a.in[kXS][m]) + e);
    L.r[kXdot] = ld_stream16(reinterpret_cast<const T*>(a.in[kXdot][m]) + e);
  }
  if constexpr (Tr::kDmd) {
    L.r[kZh] = ld_stream16(reinterpret_cast<const T*>(a.in[kZh][m]) + e);
    L.r[kYT] = ld_stream16(reinterpret_cast<const T*>(a.in[kYT][m]) + e);
    L.r[kYF] = ld_stream16(reinterpret_cast<const T*>(a.in[kYF][m]) + e);
  }
}

// Directions of one vector: gs (sCM) and gd (DMD), and the three sums.
template <typename T, int MODE>
__device__ __forceinline__ void directions(const Loaded<T, MODE>& L, const RoundCoef& k,
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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// slots
// ---------------------------------------------------------------------------

// One slot of a thread: sample bl of round r, slot index inside that sample.
struct Item {
  int r, bl, slot;
};

__device__ __forceinline__ int round_size(const ObjectiveArgs& a, int r) {
  return min(a.spr, a.B - r * a.spr);
}

// The thread's first slot of round r; false if it owns no slot at all (every
// thread owns the same number of slots in every sample, which may be zero).
__device__ __forceinline__ bool item_begin(Item& it, int r, const ObjectiveArgs& a) {
  it.r = r;
  it.bl = 0;
  it.slot = threadIdx.x;
  return r < a.rounds && (int)threadIdx.x < a.sample_f;
}

// The thread's next slot, in this sample, the next sample or the next round.
__device__ __forceinline__ bool item_next(Item& it, const ObjectiveArgs& a) {
  it.slot += kThreads;
  if (it.slot < a.sample_f) return true;
  it.slot = threadIdx.x;
  if (++it.bl < round_size(a, it.r)) return true;
  it.bl = 0;
  return ++it.r < a.rounds;
}

struct Where {
  int64_t e;  // first element of the vector
  int m;
  bool valid;
};

template <int VE>
__device__ __forceinline__ Where locate(const Item& it, int cta, const ObjectiveArgs& a) {
  int m = 0;
#pragma unroll
  for (int i = 1; i < kMaxM; ++i)
    if (i < a.M && it.slot >= a.choff[i]) m = i;
  const int64_t pos = it.slot - a.choff[m];
  const SegGeom g = seg_geom<VE>(a.n[m], a.stride[m], it.r * a.spr + it.bl);
  const int64_t v = (int64_t)cta * a.chunk[m] + pos;
  Where w;
  w.m = m;
  w.valid = pos < a.chunk[m] && v < g.nvec;
  w.e = g.e0 + g.head + v * VE;
  return w;
}

template <typename T, int MODE>
__device__ __forceinline__ void keep(float4* region, int64_t stride, int64_t pos, const float* gs,
                                     const float* gd) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  int p = 0;
  if constexpr (Tr::kScm) {
#pragma unroll
    for (int i = 0; i < VE; i += 4, ++p)
      region[p * stride + pos] = make_float4(gs[i], gs[i + 1], gs[i + 2], gs[i + 3]);
  }
  if constexpr (Tr::kDmd) {
#pragma unroll
    for (int i = 0; i < VE; i += 4, ++p)
      region[p * stride + pos] = make_float4(gd[i], gd[i + 1], gd[i + 2], gd[i + 3]);
  }
}

template <typename T, int MODE>
__device__ __forceinline__ void fetch(const float4* region, int64_t stride, int64_t pos, float* gs,
                                      float* gd) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  int p = 0;
  if constexpr (Tr::kScm) {
#pragma unroll
    for (int i = 0; i < VE; i += 4, ++p) {
      const float4 f = region[p * stride + pos];
      gs[i] = f.x; gs[i + 1] = f.y; gs[i + 2] = f.z; gs[i + 3] = f.w;
    }
  }
  if constexpr (Tr::kDmd) {
#pragma unroll
    for (int i = 0; i < VE; i += 4, ++p) {
      const float4 f = region[p * stride + pos];
      gd[i] = f.x; gd[i + 1] = f.y; gd[i + 2] = f.z; gd[i + 3] = f.w;
    }
  }
}

// ---------------------------------------------------------------------------
// unaligned head and tail elements
// ---------------------------------------------------------------------------

// The elements before the first 16-byte boundary and after the last full vector of
// every (sample, modality) segment of the round are handled by CTA G-1, one element
// per thread: 16 threads per segment (at most 7 head + 7 tail elements), at most
// kMaxRound * kMaxM = 32 segments. Returns the element index, or -1 if this thread
// has none; sets the segment (bl, m).
template <int VE>
__device__ __forceinline__ int64_t scalar_element(const ObjectiveArgs& a, int b0, int nb, int& bl,
                                                  int& m) {
  const int pair = threadIdx.x >> 4, lane16 = threadIdx.x & 15;
  bl = pair / a.M;
  m = pair - bl * a.M;
  if (bl >= nb) return -1;
  const SegGeom g = seg_geom<VE>(a.n[m], a.stride[m], b0 + bl);
  if (lane16 < g.head) return g.e0 + lane16;
  if (lane16 >= 8 && lane16 - 8 < g.tail) return g.e0 + g.head + g.nvec * VE + (lane16 - 8);
  return -1;
}

template <typename T, int MODE>
__device__ __forceinline__ void scalar_direction(const ObjectiveArgs& a, int m, int64_t e,
                                                 const RoundCoef& k, float& gs, float& gd,
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
    const float yt = load_scalar<T>(a.in[kYT][m], e);
    const float yf = load_scalar<T>(a.in[kYF][m], e);
    gd = yf - yt;
    sabs = fabsf(zh - yt);
  }
}

// ---------------------------------------------------------------------------
// round set-up, publication, merge
// ---------------------------------------------------------------------------

// Per-sample coefficients of round r and the head/tail sums (CTA G-1).
template <typename T, int MODE>
__device__ void round_setup(const ObjectiveArgs& a, SmemCtl& ctl, int r, int cta, int G) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  const int tid = threadIdx.x;
  const int ci = r & 1;
  const int b0 = r * a.spr;
  const int nb = round_size(a, r);
  if (tid < nb) {
    RoundCoef c{0.f, 0.f, 0.f, 1.f, 1};
    if constexpr (Tr::kScm) {
      const Coef k = sample_coef(__ldg(a.t + b0 + tid), a.beta, a.gamma);
      c = RoundCoef{k.kD, k.kz, k.kx, k.s, k.ok ? 1 : 0};
    }
    ctl.coef[ci][tid] = c;
  }
  __syncthreads();
  if (cta == G - 1) {  // block-uniform
    int bl, m;
    const int64_t e = scalar_element<VE>(a, b0, nb, bl, m);
    float gs = 0.f, gd = 0.f, sabs = 0.f;
    if (e >= 0) scalar_direction<T, MODE>(a, m, e, ctl.coef[ci][bl], gs, gd, sabs);
    const float sg = sum16(gs * gs), sa = sum16(sabs), sd = sum16(gd * gd);
    if ((tid & 15) == 0 && bl < nb) {
      ctl.scal[bl][m][0] = sg;
      ctl.scal[bl][m][1] = sa;
      ctl.scal[bl][m][2] = sd;
    }
  }
}

// After A(r): the CTA's sums of every (sample, modality, quantity) of the round, as
// epoch-tagged words. The per-warp partials are added in a fixed order.
__device__ void publish(const ObjectiveArgs& a, SmemCtl& ctl, int r, int cta, int G) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b0 = r * a.spr;
  const int nb = round_size(a, r);
  const int rows = nb * a.M * kQuantities;
  for (int u = warp; u < rows; u += kWarps) {
    const int bl = u / (a.M * kQuantities);
    const int m = (u / kQuantities) % a.M;
    const int q = u % kQuantities;
    float s = lane < kWarps ? ctl.red[lane][bl][m][q] : 0.f;
    s = warp_sum(s);
    if (lane == 0) {
      if (cta == G - 1) s += ctl.scal[bl][m][q];
      if ((uint32_t)cta != ctl.withhold)
        st_word(a.partials + (((int64_t)(b0 + bl) * a.M + m) * kQuantities + q) * a.gmax + cta,
                pack_word(s, ctl.epoch));
    }
  }
}

// Merge(r): wait (bounded) until every CTA's words of round r carry this call's epoch,
// add them in CTA order, and derive the per-(sample, modality) gradient factors. A
// warp reads the words of up to kRowsPerPass rows at once, so one round trip to L2
// serves all of them.
constexpr int kRowsPerPass = 3;
constexpr int kWordsPerLane = 5;   // CTAs 32 j + lane, j < 5: 160 CTAs per pass

template <typename T, int MODE>
__device__ bool merge(const ObjectiveArgs& a, SmemCtl& ctl, int r, int G) {
  using Tr = Traits<T, MODE>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ci = r & 1;
  const int b0 = r * a.spr;
  const int nb = round_size(a, r);
  const int rows = nb * a.M * kQuantities;
  const uint32_t E = ctl.epoch;
  const float qnan = __int_as_float(0x7fc00000);
  for (int u0 = warp; u0 < rows; u0 += kWarps * kRowsPerPass) {
    float s[kRowsPerPass];
#pragma unroll
    for (int i = 0; i < kRowsPerPass; ++i) s[i] = 0.f;
    for (int base = 0; base < G; base += 32 * kWordsPerLane) {
      uint64_t w[kRowsPerPass][kWordsPerLane];
      uint64_t start = 0;
      for (;;) {
        bool ready = true;
#pragma unroll
        for (int i = 0; i < kRowsPerPass; ++i) {
          const int u = u0 + i * kWarps;
          const uint64_t* src = a.partials + ((int64_t)b0 * a.M * kQuantities + u) * a.gmax;
#pragma unroll
          for (int j = 0; j < kWordsPerLane; ++j) {
            const int c = base + lane + 32 * j;
            w[i][j] = (u < rows && c < G) ? ld_word(src + c) : pack_word(0.f, E);
            ready &= (uint32_t)(w[i][j] >> 32) == E;
          }
        }
        if (__all_sync(0xffffffffu, ready)) break;
        const uint64_t now = global_timer_ns();
        if (start == 0) start = now;
        if (now - start > ctl.timeout_ns || *reinterpret_cast<volatile int*>(&ctl.abort)) {
          if (lane == 0 && !*reinterpret_cast<volatile int*>(&ctl.abort)) {
            ctl.abort = 1;
            atomicOr(a.status, T2VA_STATUS_TIMEOUT);
            atomicExch(&a.hdr->poisoned, 1u);
          }
          break;
        }
      }
#pragma unroll
      for (int i = 0; i < kRowsPerPass; ++i)
#pragma unroll
        for (int j = 0; j < kWordsPerLane; ++j) s[i] += __uint_as_float((uint32_t)w[i][j]);
    }
#pragma unroll
    for (int i = 0; i < kRowsPerPass; ++i) {
      const int u = u0 + i * kWarps;
      const float tot = warp_sum(s[i]);
      if (lane == 0 && u < rows) {
        const int bl = u / (a.M * kQuantities);
        const int m = (u / kQuantities) % a.M;
        const int q = u % kQuantities;
        ctl.tot[ci][bl][m][q] = tot;
        const RoundCoef& k = ctl.coef[ci][bl];
        if (Tr::kScm && q == 0) {
          const float n = sqrtf(tot);
          ctl.scaleS[ci][bl][m] = 2.f * a.lam_s * a.w[m] / (k.s * (n + a.eps_s));
        }
        if (Tr::kDmd && q == 1) {
          const float c = a.n[m] > 0 ? tot / (float)a.n[m] : 0.f;
          ctl.scaleD[ci][bl][m] = k.ok ? 2.f * a.lam_d * a.w[m] / (c + a.eps_d) : qnan;
        }
      }
    }
  }
  __syncthreads();
  return !ctl.abort;
}

// ---------------------------------------------------------------------------
// gradients
// ---------------------------------------------------------------------------

// Eight consecutive gradients (32 bytes, 32-byte aligned) in one store, so every
// store instruction of a warp writes whole 32-byte sectors.
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
  asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "f"(o[0]),
               "f"(o[1]), "f"(o[2]), "f"(o[3]), "f"(o[4]), "f"(o[5]), "f"(o[6]), "f"(o[7])
               : "memory");
}

__device__ __forceinline__ void write4(float* dst, float4 o, int accumulate) {
  float4* d = reinterpret_cast<float4*>(dst);
  if (accumulate) {
    const float4 old = *d;
    o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
  }
  st_stream16(d, o);
}

template <typename T, int MODE>
__device__ __forceinline__ void write_vec(const ObjectiveArgs& a, int m, int64_t e, float scS,
                                          float scD, const float* gs, const float* gd) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  const bool alias = Tr::kScm && Tr::kDmd && ((a.alias_mask >> m) & 1u);
  if constexpr (VE == 8) {
    if ((a.wide_mask >> m) & 1u) {  // both gradient buffers of m are 32-byte aligned
      float o[8];
      if (alias) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = scS * gs[i] + scD * gd[i];
        write8(a.grad_s[m] + e, o, a.accumulate);
        return;
      }
      if constexpr (Tr::kScm) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = scS * gs[i];
        write8(a.grad_s[m] + e, o, a.accumulate);
      }
      if constexpr (Tr::kDmd) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = scD * gd[i];
        write8(a.grad_d[m] + e, o, a.accumulate);
      }
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < VE; i += 4) {
    if (alias) {
      write4(a.grad_s[m] + e + i,
             make_float4(scS * gs[i] + scD * gd[i], scS * gs[i + 1] + scD * gd[i + 1],
                         scS * gs[i + 2] + scD * gd[i + 2], scS * gs[i + 3] + scD * gd[i + 3]),
             a.accumulate);
    } else {
      if constexpr (Tr::kScm)
        write4(a.grad_s[m] + e + i,
               make_float4(scS * gs[i], scS * gs[i + 1], scS * gs[i + 2], scS * gs[i + 3]),
               a.accumulate);
      if constexpr (Tr::kDmd)
        write4(a.grad_d[m] + e + i,
               make_float4(scD * gd[i], scD * gd[i + 1], scD * gd[i + 2], scD * gd[i + 3]),
               a.accumulate);
    }
  }
}

__device__ __forceinline__ void write1(float* dst, float v, int accumulate) {
  if (accumulate) v += *dst;
  *dst = v;
}

// W(r): the gradients of round r and its per-sample outputs.
template <typename T, int MODE>
__device__ void write_round(const ObjectiveArgs& a, SmemCtl& ctl, const float4* group, int r,
                            int cta, int G) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  const int tid = threadIdx.x;
  const int ci = r & 1;
  const int b0 = r * a.spr;
  const int nb = round_size(a, r);
  const int64_t kstride = (int64_t)a.spr * a.keep_f;
  const float qnan = __int_as_float(0x7fc00000);

  if (tid < a.sample_f) {
    for (int bl = 0; bl < nb; ++bl) {
      for (int slot = tid; slot < a.sample_f; slot += kThreads) {
        const Item it{r, bl, slot};
        const Where w = locate<VE>(it, cta, a);
        if (!w.valid) continue;
        float gs[VE], gd[VE];
        if (slot < a.keep_f) {
          fetch<T, MODE>(group, kstride, (int64_t)bl * a.keep_f + slot, gs, gd);
        } else {  // not kept on chip: recompute from the inputs
          Loaded<T, MODE> L;
          load_vec<T, MODE>(L, a, w.m, w.e);
          float d0 = 0.f, d1 = 0.f, d2 = 0.f;
          directions<T, MODE>(L, ctl.coef[ci][bl], gs, gd, d0, d1, d2);
        }
        const float scS = Tr::kScm ? ctl.scaleS[ci][bl][w.m] : 0.f;
        const float scD = Tr::kDmd ? ctl.scaleD[ci][bl][w.m] : 0.f;
        write_vec<T, MODE>(a, w.m, w.e, scS, scD, gs, gd);
      }
    }
  }

  // unaligned head/tail elements (CTA G-1)
  if (cta == G - 1) {
    int bl, m;
    const int64_t e = scalar_element<VE>(a, b0, nb, bl, m);
    if (e >= 0) {
      float gs = 0.f, gd = 0.f, sabs = 0.f;
      scalar_direction<T, MODE>(a, m, e, ctl.coef[ci][bl], gs, gd, sabs);
      const float scS = Tr::kScm ? ctl.scaleS[ci][bl][m] : 0.f;
      const float scD = Tr::kDmd ? ctl.scaleD[ci][bl][m] : 0.f;
      if (Tr::kScm && Tr::kDmd && ((a.alias_mask >> m) & 1u)) {
        write1(a.grad_s[m] + e, scS * gs + scD * gd, a.accumulate);
      } else {
        if constexpr (Tr::kScm) write1(a.grad_s[m] + e, scS * gs, a.accumulate);
        if constexpr (Tr::kDmd) write1(a.grad_d[m] + e, scD * gd, a.accumulate);
      }
    }
  }

  // per-sample outputs: sample b is written by CTA b % G
  for (int bl = tid; bl < nb; bl += kThreads) {
    const int b = b0 + bl;
    if (b % G != cta) continue;
    const RoundCoef& k = ctl.coef[ci][bl];
    float Ls = 0.f, Ld = 0.f;
    for (int m = 0; m < a.M; ++m) {
      if constexpr (Tr::kScm) {
        const float Sg = ctl.tot[ci][bl][m][0];
        const float n = sqrtf(Sg);
        const float d = n + a.eps_s;
        Ls += a.w[m] * (Sg / (d * d));
        if (a.norm) a.norm[(int64_t)b * a.M + m] = k.ok ? n : qnan;
      }
      if constexpr (Tr::kDmd) {
        const float c = a.n[m] > 0 ? ctl.tot[ci][bl][m][1] / (float)a.n[m] : 0.f;
        const float d = c + a.eps_d;
        Ld += a.w[m] * (ctl.tot[ci][bl][m][2] / (d * d));
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

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_objective(const __grid_constant__ ObjectiveArgs a) {
  using Tr = Traits<T, MODE>;
  constexpr int VE = Tr::VE;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(smem_raw);
  float4* kept = reinterpret_cast<float4*>(smem_raw + kCtlBytes);
  const int64_t kstride = (int64_t)a.spr * a.keep_f;  // float4 per piece of one group
  const int64_t group_f4 = (int64_t)Tr::kPieces * kstride;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    const uint32_t magic = ld_relaxed_gpu(&a.hdr->magic);
    const uint32_t poisoned = ld_relaxed_gpu(&a.hdr->poisoned);
    ctl.timeout_ns = *reinterpret_cast<volatile uint64_t*>(&a.hdr->timeout_ns);
    ctl.epoch = ld_relaxed_gpu(&a.hdr->epoch);
    ctl.withhold = ld_relaxed_gpu(&a.hdr->withhold_cta);
    ctl.abort = 0;
    if (magic != kWsMagic || poisoned != 0 || ctl.epoch == 0) {
      ctl.abort = 1;
      atomicOr(a.status, T2VA_STATUS_BAD_WORKSPACE);
    }
  }
  for (int u = lane; u < kMaxRound * kMaxM * kQuantities; u += 32)
    (&ctl.red[warp][0][0][0])[u] = 0.f;
  __syncthreads();
  if (ctl.abort) return;

  // the first slot's loads
  Item it;
  bool have = item_begin(it, 0, a);
  Loaded<T, MODE> Lc;
  Where wc{0, 0, false};
  if (have) {
    wc = locate<VE>(it, cta, a);
    if (wc.valid) load_vec<T, MODE>(Lc, a, wc.m, wc.e);
  }

  for (int r = 0; r < a.rounds; ++r) {
    const int ci = r & 1;
    __syncthreads();  // the previous round's W (and reads of its group) are done
    round_setup<T, MODE>(a, ctl, r, cta, G);
    __syncthreads();
    float4* group = kept + (r % a.groups) * group_f4;

    // A(r): the next slot's loads are in flight while this one is computed
    float sg = 0.f, sa = 0.f, sd = 0.f;
    while (have && it.r == r) {
      Item nx = it;
      const bool have_n = item_next(nx, a);
      Loaded<T, MODE> Ln;
      Where wn{0, 0, false};
      if (have_n) {
        wn = locate<VE>(nx, cta, a);
        if (wn.valid) load_vec<T, MODE>(Ln, a, wn.m, wn.e);
      }
      if (wc.valid) {
        float gs[VE], gd[VE];
        directions<T, MODE>(Lc, ctl.coef[ci][it.bl], gs, gd, sg, sa, sd);
        if (it.slot < a.keep_f)
          keep<T, MODE>(group, kstride, (int64_t)it.bl * a.keep_f + it.slot, gs, gd);
      }
      // a warp's slots change (sample, modality) together: flush its sums then
      if (!have_n || nx.r != r || nx.bl != it.bl || wn.m != wc.m) {
        sg = warp_sum(sg);
        sa = warp_sum(sa);
        sd = warp_sum(sd);
        if (lane == 0) {
          ctl.red[warp][it.bl][wc.m][0] += sg;
          ctl.red[warp][it.bl][wc.m][1] += sa;
          ctl.red[warp][it.bl][wc.m][2] += sd;
        }
        sg = sa = sd = 0.f;
      }
      it = nx;
      Lc = Ln;
      wc = wn;
      have = have_n;
    }
    __syncthreads();  // per-warp sums and head/tail sums complete
    publish(a, ctl, r, cta, G);
    __syncthreads();  // sums read: clear this warp's rows for the next round
    for (int u = lane; u < kMaxRound * kMaxM * kQuantities; u += 32)
      (&ctl.red[warp][0][0][0])[u] = 0.f;

    if (a.groups == 1) {
      if (!merge<T, MODE>(a, ctl, r, G)) return;
      write_round<T, MODE>(a, ctl, group, r, cta, G);
    } else if (r >= 1) {
      if (!merge<T, MODE>(a, ctl, r - 1, G)) return;
      write_round<T, MODE>(a, ctl, kept + ((r - 1) % a.groups) * group_f4, r - 1, cta, G);
    }
  }
  if (a.groups > 1 && a.rounds > 0) {
    const int r = a.rounds - 1;
    if (!merge<T, MODE>(a, ctl, r, G)) return;
    write_round<T, MODE>(a, ctl, kept + (r % a.groups) * group_f4, r, cta, G);
  }
  // Every CTA has published its last round's words, tagged with this epoch, before
  // CTA 0's last merge could finish: all of them have read the epoch, so it can move
  // on for the next call.
  if (cta == 0 && tid == 0) {
    const uint32_t next = ctl.epoch + 1u;
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(&a.hdr->epoch),
                 "r"(next == 0u ? 1u : next)
                 : "memory");
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
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA is resident: the waits always end
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
    // block 0 zeroed the header above; write its fields after that block's barrier
    WsHeader* h = reinterpret_cast<WsHeader*>(ws);
    h->timeout_ns = timeout_ns;
    h->gmax = gmax;
    h->poisoned = 0;
    h->epoch = 1;  // zeroed words carry epoch 0, so no word of a fresh workspace is final
    h->withhold_cta = kNoWithhold;
    __threadfence();
    h->magic = kWsMagic;
  }
}

}  // namespace

bool plan_objective(ObjectiveArgs& a, t2va_dtype dt, int mode, int sm_count, size_t smem_optin,
                    size_t /*l2_bytes*/, ObjectiveLaunch* out) {
  const int VE = dt == T2VA_BFLOAT16 ? 8 : 4;
  const int Q = ((mode & kModeScm) ? 1 : 0) + ((mode & kModeDmd) ? 1 : 0);
  const int64_t slot_bytes = (int64_t)Q * VE / 4 * 16;  // kept direction bytes per slot
  int64_t vtot = 0, nvec_ub[kMaxM];
  for (int m = 0; m < a.M; ++m) {
    nvec_ub[m] = (a.n[m] + VE - 1) / VE;
    vtot += nvec_ub[m];
  }
  int64_t G = (vtot + kThreads - 1) / kThreads;  // small problems use fewer CTAs
  G = std::max<int64_t>(1, std::min<int64_t>({G, (int64_t)sm_count, (int64_t)a.gmax}));
  int64_t acc = 0;
  for (int m = 0; m < a.M; ++m) {
    a.chunk[m] = (nvec_ub[m] + G - 1) / G;
    a.choff[m] = (int)std::min<int64_t>(acc, INT32_MAX);
    acc += (a.chunk[m] + 31) / 32 * 32;
    if (acc > (int64_t)1 << 30) return false;
  }
  for (int m = a.M; m < kMaxM; ++m) {
    a.chunk[m] = 0;
    a.choff[m] = (int)acc;
  }
  a.sample_f = (int)acc;
  if (smem_optin <= kCtlBytes + (size_t)32 * slot_bytes) return false;
  const int64_t budget = (int64_t)(smem_optin - kCtlBytes);
  const int64_t per_sample = a.sample_f * slot_bytes;
  a.keep_f = a.sample_f;
  if (per_sample == 0 || (a.B <= kMaxRound && a.B * per_sample <= budget)) {
    a.groups = 1;  // one round: A, merge, W
    a.spr = std::max(1, std::min(a.B, kMaxRound));
  } else if (a.B >= 2 && 2 * per_sample <= budget) {
    a.groups = 2;  // A0 A1 W0 A2 W1 ...
    const int64_t spr = std::min<int64_t>({budget / (2 * per_sample), (a.B + 1) / 2, kMaxRound});
    a.spr = (int)std::max<int64_t>(1, spr);
  } else if (per_sample <= budget) {
    a.groups = 1;
    a.spr = 1;
  } else {  // one sample's directions exceed shared memory: keep a prefix of its slots
    a.groups = 1;
    a.spr = 1;
    a.keep_f = (int)(budget / slot_bytes / 32 * 32);
  }
  a.rounds = (a.B + a.spr - 1) / a.spr;
  out->grid = (int)G;
  out->threads = kThreads;
  out->smem = kCtlBytes + (size_t)a.groups * a.spr * a.keep_f * slot_bytes;
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
  int blocks = (int)std::min<size_t>(1024, std::max<size_t>(1, (n16 + 255) / 256));
  k_ws_init<<<blocks, 256, 0, st>>>(reinterpret_cast<uint4*>(ws), n16, timeout_ns, gmax);
  return cudaGetLastError();
}

}  // namespace t2va
