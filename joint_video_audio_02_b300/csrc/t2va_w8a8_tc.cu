// Post-scale W8A8 linear on B300's fifth-generation tensor cores (TurboT2VA, section 6.2
// of the robotworld.top/zh reading): y_ij = s_i^x s_j^w sum_k x_hat_ik w_hat_jk + b_j
// with the integer sum exact.
//
// sm_103a has no INT8 form of tcgen05.mma. The codes are integers in [-127, 127], which
// bfloat16 holds exactly, and so are their products (|p| <= 16129) and every partial sum
// below 2^24 in float32. So the codes are stored as bfloat16 and contracted by
// tcgen05.mma kind::f16 (bf16 x bf16 -> f32) in chunks of 1024 along K: a chunk's sum is
// at most 1024 * 16129 < 2^24 in magnitude, hence exact in its float32 accumulator
// whatever the order of the additions, and the chunks are added as int32 by the
// epilogue. The result is the exact INT32 sum of the pages' operator.
//
// Two kernels. When N is a multiple of 256, k_w8a8_tc_wide (below) runs persistent CTAs
// over 128 x 256 tiles. Otherwise k_w8a8_tc runs one CTA per 128 x 128 output tile, 192
// threads, two CTAs per SM (one CTA's epilogue and set-up overlap the other's MMAs;
// measured 591 -> 903 TOPS at 28672 x 4096 x 4096):
//   warp 0      TMA producer: A and B tiles of 128 rows x 64 bf16 (128 bytes, swizzled
//               128B) into a 3-stage shared-memory ring, one mbarrier per stage;
//   warp 1      allocates 256 TMEM columns (two 128-column float32 accumulators)
//               and issues the MMAs from one thread: 4 x (M128 N128 K16) per stage,
//               the first MMA of each 1024-K chunk overwriting its accumulator; frees a
//               stage with tcgen05.commit, and signals a finished chunk the same way;
//   warps 2-5   epilogue: each reads its 32 TMEM lanes (rows) of a finished chunk
//               (tcgen05.ld 32x32b), adds it to int32 registers, hands the accumulator
//               back, and finally writes y = fma(float(acc), s_x s_w, b) once.
// Every mbarrier wait is bounded; a wait that runs out sets T2VA_STATUS_TIMEOUT in the
// caller's status word, the CTA drains its copies and MMAs (bounded again), frees TMEM
// and returns.
#include <cuda.h>

#include "t2va_w8a8.cuh"

namespace t2va {
namespace {

constexpr int kTM = 128, kTN = 128, kTK = 64;    // tile; kTK in bf16 elements (128 bytes)
constexpr int kTStages = 3;                      // two CTAs per SM fit
constexpr int kTThreads = 192;
constexpr int kChunkK = 1024;                    // K per exact float32 partial sum
constexpr int kStagesPerChunk = kChunkK / kTK;   // 16
constexpr int kAccSlots = 2;                     // TMEM accumulators of 128 columns
constexpr int kTmemCols = 256;                   // half of TMEM per CTA
constexpr uint32_t kTileBytes = kTM * kTK * 2;   // 16 KB per operand tile
constexpr uint32_t kStageTx = 2 * kTileBytes;
constexpr uint32_t kWaitLimit = 1u << 20;        // x 1 us suspend hint: about a second

struct TcSmem {
  uint64_t full[kTStages];
  uint64_t empty[kTStages];
  uint64_t acc_full[kAccSlots];
  uint64_t acc_empty[kAccSlots];
  uint64_t drain;
  uint64_t stall;  // never arrived on: the wait of the self-test
  uint32_t tmem_base;
  uint32_t abort;
};
constexpr size_t kTcSmem = 1024 /* alignment slack */ + (size_t)kTStages * kStageTx + 1024;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// Wait for the phase of parity `parity` to complete; false if it did not within the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(su32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte swizzle
// (rows of 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;     // leading-dimension offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;   // stride-dimension offset: one 8-row group
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor: D float32, A and B bfloat16, both K-major, M = 128, N = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTN >> 3) << 17) |
                            ((uint32_t)(kTM >> 4) << 24);

// Instruction descriptor of the wide tiles: M = 128, N = 256.
constexpr int kWN = 256;
constexpr uint32_t kIdescWide = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kWN >> 3) << 17) |
                                ((uint32_t)(kTM >> 4) << 24);

__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate,
                                     uint32_t idesc = kIdesc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive float32 columns of this warp's 32 TMEM lanes, one lane per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <bool BF16_OUT>
__global__ void __launch_bounds__(kTThreads, 2)
    k_w8a8_tc(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
              const __grid_constant__ GemmArgs a) {
  extern __shared__ unsigned char smem_raw[];
  // stages at a 1024-byte boundary (the 128-byte swizzle repeats every 1024 bytes)
  const uint32_t raw = su32(smem_raw);
  const uint32_t tiles = (raw + 1023u) & ~1023u;
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw + (tiles - raw) + kTStages * kStageTx);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * kTN, m0 = (int64_t)blockIdx.y * kTM;
  const int KT = (int)(a.K / kTK);
  const int nchunks = (KT + kStagesPerChunk - 1) / kStagesPerChunk;

  // a CTA that finds a timeout already recorded (by an earlier CTA of this launch, or a
  // launch before it) does nothing, so a failing launch ends in about one wait limit
  __shared__ uint32_t skip;
  if (threadIdx.x == 0)
    skip = (a.status != nullptr && (*reinterpret_cast<volatile int*>(a.status) & T2VA_STATUS_TIMEOUT)) ? 1u : 0u;
  __syncthreads();
  if (skip) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int j = 0; j < kAccSlots; ++j) {
      mbar_init(&sm.acc_full[j], 1);
      mbar_init(&sm.acc_empty[j], 4);
    }
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.stall, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&sm.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  volatile uint32_t* abort = &sm.abort;
  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kt = 0; kt < KT && !*abort; ++kt) {
        const int s = kt % kTStages, use = kt / kTStages;
        if (use > 0 && !mbar_wait(&sm.empty[s], (use - 1) & 1)) {
          *abort = 1;
          if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
          break;
        }
        const uint32_t sa = tiles + s * kStageTx;
        mbar_expect_tx(&sm.full[s], kStageTx);
        tma_2d(sa, &map_a, &sm.full[s], kt * kTK, (int)m0);
        tma_2d(sa + kTileBytes, &map_b, &sm.full[s], kt * kTK, (int)n0);
        issued = kt + 1;
      }
      // every copy this thread started has landed before the CTA's shared memory goes
      for (int kt = issued > kTStages ? issued - kTStages : 0; kt < issued; ++kt)
        mbar_wait(&sm.full[kt % kTStages], (kt / kTStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (a.selftest_wait && !mbar_wait(&sm.stall, 0)) {
        *abort = 1;
        if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
      }
      for (int kt = 0; kt < KT && !*abort; ++kt) {
        const int s = kt % kTStages, c = kt / kStagesPerChunk, slot = c % kAccSlots;
        const bool first = (kt % kStagesPerChunk) == 0;
        if (first && c >= kAccSlots) {
          if (!mbar_wait(&sm.acc_empty[slot], ((c / kAccSlots) - 1) & 1)) {
            *abort = 1;
            if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
            break;
          }
          tc_fence_after();
        }
        if (!mbar_wait(&sm.full[s], (kt / kTStages) & 1)) {
          *abort = 1;
          if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t sa = tiles + s * kStageTx;
        const uint64_t da = smem_desc(sa), db = smem_desc(sa + kTileBytes);
#pragma unroll
        for (int k = 0; k < kTK / 16; ++k)  // K = 16 bf16 (32 bytes) per MMA
          umma(tmem + slot * kTN, da + (uint64_t)(k * 2), db + (uint64_t)(k * 2), (first && k == 0) ? 0u : 1u);
        umma_commit(&sm.empty[s]);
        if ((kt % kStagesPerChunk) == kStagesPerChunk - 1 || kt == KT - 1) umma_commit(&sm.acc_full[slot]);
      }
      // every MMA this thread issued has finished before TMEM is freed
      umma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0);
    }
  } else {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. rows of the tile
    const int g = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * g) << 16;
    int acc[kTN];
#pragma unroll
    for (int j = 0; j < kTN; ++j) acc[j] = 0;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int slot = c % kAccSlots;
      if (!mbar_wait(&sm.acc_full[slot], (c / kAccSlots) & 1)) {
        ok = false;
        *abort = 1;
        if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < kTN / 32; ++q) {
        float v[32];
        tmem_ld32(tmem + lane_base + slot * kTN + q * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[q * 32 + i] += __float2int_rn(v[i]);  // exact integers
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[slot]);
    }
    if (ok) {
      const int64_t row = m0 + 32 * g + lane;
      const float sx = __ldg(a.sx + row);
#pragma unroll
      for (int q = 0; q < kTN / 8; ++q) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t col = n0 + q * 8 + i;
          const float b = a.bias ? __ldg(a.bias + col) : 0.f;
          y[i] = fmaf((float)acc[q * 8 + i], sx * __ldg(a.sw + col), b);
        }
        if constexpr (BF16_OUT) {
          uint4 o;
          __nv_bfloat162 h0 = __floats2bfloat162_rn(y[0], y[1]), h1 = __floats2bfloat162_rn(y[2], y[3]);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(y[4], y[5]), h3 = __floats2bfloat162_rn(y[6], y[7]);
          o.x = *reinterpret_cast<uint32_t*>(&h0);
          o.y = *reinterpret_cast<uint32_t*>(&h1);
          o.z = *reinterpret_cast<uint32_t*>(&h2);
          o.w = *reinterpret_cast<uint32_t*>(&h3);
          *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.y) + row * a.N + n0 + q * 8) = o;
        } else {
          float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) + row * a.N + n0 + q * 8);
          d[0] = make_float4(y[0], y[1], y[2], y[3]);
          d[1] = make_float4(y[4], y[5], y[6], y[7]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Wide tiles (N divisible by 256): one persistent CTA per SM walks output tiles of
// 128 x 256, tile t at rows 128 (t / (N / 256)) and columns 256 (t % (N / 256)), so the
// CTAs running at once share A row blocks and all of B through L2. An M128 N256 K16 MMA
// reads 12 KB of operands from shared memory per 128 tensor-core cycles, against 8 KB per
// 64 cycles for N = 128, so the shared-memory traffic of the operands (TMA writes plus MMA
// reads) per flop falls by a quarter (measured 1141 -> 1370 TOPS at 28672 x 4096 x 4096).
// 320 threads:
//   warp 0      TMA producer: per stage one 128 x 64 A box and two 128 x 64 B boxes (the
//               B tile's rows 0-127 and 128-255, contiguous in shared memory), 4 stages;
//   warp 1      allocates all 512 TMEM columns (two 256-column float32 accumulators,
//               used as a ring across chunks and tiles) and issues 4 x (M128 N256 K16)
//               per stage;
//   warps 2-9   epilogue: two warps per TMEM lane quadrant (rows), one per 128-column
//               half; they add each finished chunk as int32 and write the tile's y once,
//               while the MMAs of the next chunk, or of the next tile, proceed in the
//               other accumulator.
constexpr int kWStages = 4;
constexpr int kWEpiWarps = 8;
constexpr int kWThreads = 64 + 32 * kWEpiWarps;
constexpr int kWTmemCols = 2 * kWN;
constexpr uint32_t kWStageTx = kTileBytes + 2 * kTileBytes;   // A 16 KB + B 32 KB
constexpr size_t kWSmem = 1024 /* alignment slack */ + (size_t)kWStages * kWStageTx + 1024;

struct WideSmem {
  uint64_t full[kWStages];
  uint64_t empty[kWStages];
  uint64_t acc_full[kAccSlots];
  uint64_t acc_empty[kAccSlots];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
};

template <bool BF16_OUT>
__global__ void __launch_bounds__(kWThreads, 1)
    k_w8a8_tc_wide(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ GemmArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = su32(smem_raw);
  const uint32_t tiles = (raw + 1023u) & ~1023u;
  WideSmem& sm = *reinterpret_cast<WideSmem*>(smem_raw + (tiles - raw) + kWStages * kWStageTx);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = (int)(a.K / kTK);
  const int nchunks = (KT + kStagesPerChunk - 1) / kStagesPerChunk;
  const int tiles_n = (int)(a.N / kWN);
  const int ntiles = (int)(a.M / kTM) * tiles_n;

  __shared__ uint32_t skip;
  if (threadIdx.x == 0)
    skip = (a.status != nullptr && (*reinterpret_cast<volatile int*>(a.status) & T2VA_STATUS_TIMEOUT)) ? 1u : 0u;
  __syncthreads();
  if (skip) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int j = 0; j < kAccSlots; ++j) {
      mbar_init(&sm.acc_full[j], 1);
      mbar_init(&sm.acc_empty[j], kWEpiWarps);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&sm.tmem_base)),
                 "r"(kWTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  volatile uint32_t* abort = &sm.abort;
  if (warp == 0) {
    if (lane == 0) {
      int64_t g = 0, issued = 0;  // stages over all of this CTA's tiles
      for (int tile = blockIdx.x; tile < ntiles && !*abort; tile += gridDim.x) {
        const int m0 = (tile / tiles_n) * kTM, n0 = (tile % tiles_n) * kWN;
        for (int kt = 0; kt < KT && !*abort; ++kt, ++g) {
          const int s = (int)(g % kWStages);
          const int64_t use = g / kWStages;
          if (use > 0 && !mbar_wait(&sm.empty[s], (uint32_t)((use - 1) & 1))) {
            *abort = 1;
            if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
            break;
          }
          const uint32_t sa = tiles + s * kWStageTx;
          mbar_expect_tx(&sm.full[s], kWStageTx);
          tma_2d(sa, &map_a, &sm.full[s], kt * kTK, m0);
          tma_2d(sa + kTileBytes, &map_b, &sm.full[s], kt * kTK, n0);
          tma_2d(sa + 2 * kTileBytes, &map_b, &sm.full[s], kt * kTK, n0 + kTM);
          issued = g + 1;
        }
      }
      // every copy this thread started has landed before the CTA's shared memory goes
      for (int64_t q = issued > kWStages ? issued - kWStages : 0; q < issued; ++q)
        mbar_wait(&sm.full[q % kWStages], (uint32_t)((q / kWStages) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int64_t g = 0, gc0 = 0;  // stages and chunks over all of this CTA's tiles
      bool dead = false;
      for (int tile = blockIdx.x; tile < ntiles && !dead; tile += gridDim.x, gc0 += nchunks) {
        for (int kt = 0; kt < KT; ++kt, ++g) {
          if (*abort) {
            dead = true;
            break;
          }
          const int s = (int)(g % kWStages);
          const int64_t gc = gc0 + kt / kStagesPerChunk;
          const int slot = (int)(gc % kAccSlots);
          const bool first = (kt % kStagesPerChunk) == 0;
          if (first && gc >= kAccSlots) {
            if (!mbar_wait(&sm.acc_empty[slot], (uint32_t)(((gc / kAccSlots) - 1) & 1))) {
              *abort = 1;
              if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
              dead = true;
              break;
            }
            tc_fence_after();
          }
          if (!mbar_wait(&sm.full[s], (uint32_t)((g / kWStages) & 1))) {
            *abort = 1;
            if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
            dead = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + s * kWStageTx;
          const uint64_t da = smem_desc(sa), db = smem_desc(sa + kTileBytes);
#pragma unroll
          for (int k = 0; k < kTK / 16; ++k)
            umma(tmem + slot * kWN, da + (uint64_t)(k * 2), db + (uint64_t)(k * 2), (first && k == 0) ? 0u : 1u,
                 kIdescWide);
          umma_commit(&sm.empty[s]);
          if ((kt % kStagesPerChunk) == kStagesPerChunk - 1 || kt == KT - 1) umma_commit(&sm.acc_full[slot]);
        }
      }
      umma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0);
    }
  } else {
    // warp w reads TMEM lanes 32 (w % 4) .. + 31 (rows), columns 128 h .. + 127
    const int g = warp & 3, h = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(32 * g) << 16;
    int64_t gc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const int64_t m0 = (int64_t)(tile / tiles_n) * kTM, n0 = (int64_t)(tile % tiles_n) * kWN + h * kTN;
      int acc[kTN];
#pragma unroll
      for (int j = 0; j < kTN; ++j) acc[j] = 0;
      for (int c = 0; c < nchunks; ++c, ++gc) {
        const int slot = (int)(gc % kAccSlots);
        if (!mbar_wait(&sm.acc_full[slot], (uint32_t)((gc / kAccSlots) & 1))) {
          ok = false;
          *abort = 1;
          if (a.status) atomicOr(a.status, T2VA_STATUS_TIMEOUT);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < kTN / 32; ++q) {
          float v[32];
          tmem_ld32(tmem + lane_base + slot * kWN + h * kTN + q * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[q * 32 + i] += __float2int_rn(v[i]);  // exact integers
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[slot]);
      }
      if (!ok) break;
      const int64_t row = m0 + 32 * g + lane;
      const float sx = __ldg(a.sx + row);
#pragma unroll
      for (int q = 0; q < kTN / 8; ++q) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t col = n0 + q * 8 + i;
          const float b = a.bias ? __ldg(a.bias + col) : 0.f;
          y[i] = fmaf((float)acc[q * 8 + i], sx * __ldg(a.sw + col), b);
        }
        if constexpr (BF16_OUT) {
          uint4 o;
          __nv_bfloat162 h0 = __floats2bfloat162_rn(y[0], y[1]), h1 = __floats2bfloat162_rn(y[2], y[3]);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(y[4], y[5]), h3 = __floats2bfloat162_rn(y[6], y[7]);
          o.x = *reinterpret_cast<uint32_t*>(&h0);
          o.y = *reinterpret_cast<uint32_t*>(&h1);
          o.z = *reinterpret_cast<uint32_t*>(&h2);
          o.w = *reinterpret_cast<uint32_t*>(&h3);
          *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.y) + row * a.N + n0 + q * 8) = o;
        } else {
          float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) + row * a.N + n0 + q * 8);
          d[0] = make_float4(y[0], y[1], y[2], y[3]);
          d[1] = make_float4(y[4], y[5], y[6], y[7]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kWTmemCols) : "memory");
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once per process (a function-local static is
// initialised exactly once, thread-safely); null if the driver does not offer it.
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// 2-D map of a [rows][K] bf16 matrix, boxes of 128 rows x 64 elements, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {kTK, kTM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {
// buffers of the self-test launch: 128 x 128 bf16 codes (zero), scales, output
static __device__ __align__(128) __nv_bfloat16 g_st_a[128 * 128];
static __device__ __align__(128) __nv_bfloat16 g_st_b[128 * 128];
static __device__ __align__(128) float g_st_y[128 * 128];
static __device__ float g_st_s[128];
}  // namespace

cudaError_t launch_w8a8_tc_selftest(int* status, cudaStream_t st) {
  GemmArgs a = {};
  a.M = a.N = a.K = 128;
  void *pa, *pb, *py, *ps;
  if (cudaGetSymbolAddress(&pa, g_st_a) != cudaSuccess || cudaGetSymbolAddress(&pb, g_st_b) != cudaSuccess ||
      cudaGetSymbolAddress(&py, g_st_y) != cudaSuccess || cudaGetSymbolAddress(&ps, g_st_s) != cudaSuccess)
    return cudaErrorInvalidValue;
  a.xq = reinterpret_cast<const int8_t*>(pa);
  a.wq = reinterpret_cast<const int8_t*>(pb);
  a.y = py;
  a.sx = a.sw = reinterpret_cast<const float*>(ps);
  a.status = status;
  a.selftest_wait = 1;
  return launch_w8a8_tc(a, false, st);
}

// The wide persistent kernel: one CTA per SM (its shared memory admits no second one),
// at most one per tile.
static cudaError_t launch_w8a8_tc_wide(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& a, bool bf16_out,
                                cudaStream_t st) {
  // once per process, on the device current at the first call (one device per process)
  struct Setup {
    cudaError_t e;
    int sms;
  };
  static const Setup setup = [] {
    Setup r = {cudaSuccess, 0};
    int dev = 0;
    r.e = cudaGetDevice(&dev);
    if (r.e == cudaSuccess) r.e = cudaDeviceGetAttribute(&r.sms, cudaDevAttrMultiProcessorCount, dev);
    if (r.e == cudaSuccess)
      r.e = cudaFuncSetAttribute(k_w8a8_tc_wide<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmem);
    if (r.e == cudaSuccess)
      r.e = cudaFuncSetAttribute(k_w8a8_tc_wide<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmem);
    if (r.e == cudaSuccess && r.sms <= 0) r.e = cudaErrorInvalidValue;
    return r;
  }();
  if (setup.e != cudaSuccess) return setup.e;
  const int sms = setup.sms;
  const int64_t ntiles = (a.M / kTM) * (a.N / kWN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ntiles < sms ? ntiles : sms));
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = kWSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16_out) return cudaLaunchKernelEx(&cfg, k_w8a8_tc_wide<true>, ma, mb, a);
  return cudaLaunchKernelEx(&cfg, k_w8a8_tc_wide<false>, ma, mb, a);
}

cudaError_t launch_w8a8_tc(const GemmArgs& a, bool bf16_out, cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!make_map(&ma, a.xq, a.M, a.K) || !make_map(&mb, a.wq, a.N, a.K)) return cudaErrorInvalidValue;
  if (a.N % kWN == 0 && !a.selftest_wait) return launch_w8a8_tc_wide(ma, mb, a, bf16_out, st);
  static const cudaError_t smem_attr = [] {
    cudaError_t e = cudaFuncSetAttribute(k_w8a8_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_w8a8_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    return e;
  }();
  if (smem_attr != cudaSuccess) return smem_attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.N / kTN), (unsigned)(a.M / kTM));
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16_out) return cudaLaunchKernelEx(&cfg, k_w8a8_tc<true>, ma, mb, a);
  return cudaLaunchKernelEx(&cfg, k_w8a8_tc<false>, ma, mb, a);
}

}  // namespace t2va
