// Post-scale W8A8 linear operator (TurboT2VA, section 6.2 of the robotworld.top/zh
// reading, "shape-aware post-scale W8A8 linear operator"):
//
//   s_i = max(||x_i||_inf, eps) / 127,   x_hat_i = clip(rint(x_i / s_i), -127, 127)
//   y_ij = s_i^x s_j^w sum_k x_hat_ik w_hat_jk + b_j
//
// with the integer products summed exactly in INT32 over the whole K and both scales
// applied once, in the epilogue.
//
// k_quantize_rows: kTPR threads per row. The row is read once into registers (512
// vectors per row: 4096 bf16 elements; longer rows read the rest again, from L2), its
// absolute maximum is reduced by shuffles (and shared memory across the row's warps),
// and every code is rint of the
// correctly rounded float32 quotient x / s (ties to even), so the codes are bit-exact
// functions of the inputs; the quotient is formed only near a rounding boundary (see
// code_of).
//
// k_w8a8_gemm: sm_103a has no INT8 form of tcgen05.mma (ptxas rejects kind::i8 for
// this target), so the exact integer contraction runs on the warp-level INT8 MMA
// (mma.sync m16n8k32, s8 x s8 -> s32). 128 x 128 output tiles, 256 threads as 2 x 4
// warps of 64 x 32, K in steps of 64 bytes staged through a 4-deep cp.async ring in
// shared memory whose 16-byte chunks are XOR-swizzled per row pair so that ldmatrix
// reads are free of bank conflicts.
#include "t2va_w8a8.cuh"

namespace t2va {
namespace {

// ---------------------------------------------------------------------------
// per-row dynamic quantisation
// ---------------------------------------------------------------------------

constexpr int kQThreads = 256;
constexpr int kTPR = 128;                   // threads per row (measured at 28672 x 4096: 32 222 us, 64 146, 128 137, 256 138)
constexpr int kQRows = kQThreads / kTPR;    // rows per CTA
constexpr int kQCache = 512 / kTPR;         // 16-byte vectors per thread kept in registers

__device__ __forceinline__ float amax_of(const uint4& r, __nv_bfloat16) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

__device__ __forceinline__ float amax_of(const uint4& r, float) {
  const float* f = reinterpret_cast<const float*>(&r);
  return fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
}

// rint of the correctly rounded quotient x / s, clipped to [-127, 127], without a
// division for almost every element. y = x * inv with inv the correctly rounded 1 / s
// is within 3 * 2^-24 |x / s| <= 3 * 127 * 2^-24 < 2^-14 of the correctly rounded
// quotient (three roundings of relative size 2^-24 each, |x / s| <= 127). So when y
// lies more than 2^-14 from the nearest half-integer, the quotient lies on the same
// side of it and rounds to the same integer; only inside that band is the quotient
// itself formed.
__device__ __forceinline__ int code_of(float x, float s, float inv) {
  const float y = x * inv;
  float q = rintf(y);
  if (0.5f - fabsf(y - q) < 0x1p-14f) q = rintf(__fdiv_rn(x, s));
  return (int)fminf(fmaxf(q, -127.f), 127.f);
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
         ((uint32_t)(d & 0xff) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(int a, int b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn((float)a, (float)b);  // exact: |a|, |b| <= 127
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The codes of one 16-byte input vector (8 for bf16 input, 4 for float32).
template <typename T>
__device__ __forceinline__ void codes_of(const uint4& r, float s, float inv, int (&c)[16 / sizeof(T)]);

template <>
__device__ __forceinline__ void codes_of<__nv_bfloat16>(const uint4& r, float s, float inv, int (&c)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    c[2 * i] = code_of(f.x, s, inv);
    c[2 * i + 1] = code_of(f.y, s, inv);
  }
}

template <>
__device__ __forceinline__ void codes_of<float>(const uint4& r, float s, float inv, int (&c)[4]) {
  const float* f = reinterpret_cast<const float*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = code_of(f[i], s, inv);
}

// Store the codes of input vector v of a row: int8 (8 or 4 bytes) or bfloat16 integers
// (16 or 8 bytes).
template <typename T, bool BF16_CODES>
__device__ __forceinline__ void store_codes(const uint4& r, float s, float inv, void* q, int64_t v) {
  constexpr int VE = 16 / sizeof(T);
  int c[VE];
  codes_of<T>(r, s, inv, c);
  if constexpr (BF16_CODES) {
    __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(q) + v * VE;
    if constexpr (VE == 8)
      *reinterpret_cast<uint4*>(d) = make_uint4(pack_bf16(c[0], c[1]), pack_bf16(c[2], c[3]),
                                                pack_bf16(c[4], c[5]), pack_bf16(c[6], c[7]));
    else
      *reinterpret_cast<uint2*>(d) = make_uint2(pack_bf16(c[0], c[1]), pack_bf16(c[2], c[3]));
  } else {
    int8_t* d = reinterpret_cast<int8_t*>(q) + v * VE;
    if constexpr (VE == 8)
      *reinterpret_cast<uint2*>(d) = make_uint2(pack4(c[0], c[1], c[2], c[3]), pack4(c[4], c[5], c[6], c[7]));
    else
      *reinterpret_cast<uint32_t*>(d) = pack4(c[0], c[1], c[2], c[3]);
  }
}

template <typename T, bool BF16_CODES>
__global__ void __launch_bounds__(kQThreads) k_quantize_rows(const __grid_constant__ QuantArgs a) {
  constexpr int VE = 16 / sizeof(T);
  constexpr int kWarpsPerRow = kTPR >= 32 ? kTPR / 32 : 1;
  __shared__ float red[kQThreads / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int t = threadIdx.x % kTPR;
  const int64_t row = (int64_t)blockIdx.x * kQRows + threadIdx.x / kTPR;
  const bool live = row < a.rows;
  const T* x = reinterpret_cast<const T*>(a.x) + (live ? row : 0) * a.ld_x;
  const int64_t nvec = live ? a.cols / VE : 0;
  uint4 cache[kQCache];
  float m = 0.f;
#pragma unroll
  for (int c = 0; c < kQCache; ++c) {
    const int64_t v = (int64_t)c * kTPR + t;
    if (v < nvec) {
      cache[c] = ld_stream16(x + v * VE);
      m = fmaxf(m, amax_of(cache[c], T()));
    }
  }
  for (int64_t v = (int64_t)kQCache * kTPR + t; v < nvec; v += kTPR)
    m = fmaxf(m, amax_of(*reinterpret_cast<const uint4*>(x + v * VE), T()));
  // the row's maximum (max is exact, so the order of the reduction does not matter):
  // lanes of the row's threads within a warp, then the row's warps through shared memory
#pragma unroll
  for (int o = (kTPR < 32 ? kTPR : 32) / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if constexpr (kWarpsPerRow > 1) {
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    const int w0 = (threadIdx.x >> 5) / kWarpsPerRow * kWarpsPerRow;
#pragma unroll
    for (int w = 0; w < kWarpsPerRow; ++w) m = fmaxf(m, red[w0 + w]);
  }
  if (!live) return;
  const float s = __fdiv_rn(fmaxf(m, a.eps), 127.f);
  const float inv = __frcp_rn(s);
  void* q = BF16_CODES ? (void*)(reinterpret_cast<__nv_bfloat16*>(a.q) + row * a.ld_q)
                       : (void*)(reinterpret_cast<int8_t*>(a.q) + row * a.ld_q);
#pragma unroll
  for (int c = 0; c < kQCache; ++c) {
    const int64_t v = (int64_t)c * kTPR + t;
    if (v < nvec) store_codes<T, BF16_CODES>(cache[c], s, inv, q, v);
  }
  for (int64_t v = (int64_t)kQCache * kTPR + t; v < nvec; v += kTPR)
    store_codes<T, BF16_CODES>(*reinterpret_cast<const uint4*>(x + v * VE), s, inv, q, v);
  if (t == 0) a.scale[row] = s;
}

// ---------------------------------------------------------------------------
// INT8 GEMM with the post-scale epilogue
// ---------------------------------------------------------------------------

constexpr int kBM = 128, kBN = 128, kBK = 64;  // kBK in int8 elements (bytes)
constexpr int kGThreads = 256;
constexpr int kStages = 4;
constexpr int kTileBytes = kBM * kBK;                    // one operand tile, 8 KB
constexpr int kStageBytes = 2 * kTileBytes;              // A and B
constexpr int kGemmSmem = kStages * kStageBytes;         // 64 KB

// Byte offset of 16-byte chunk `c` (0..3) of row `r` of a [128][64] int8 tile.
__device__ __forceinline__ int swz(int r, int c) { return r * kBK + ((c ^ ((r >> 1) & 3)) << 4); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copies of K-step `ks` of this CTA's A rows [m0, m0+128) and B rows [n0, n0+128) into
// stage `st`: 2 x 512 chunks of 16 bytes, 4 per thread.
__device__ __forceinline__ void load_stage(const GemmArgs& a, uint32_t smem, int st, int64_t m0,
                                           int64_t n0, int ks) {
  const uint32_t base = smem + st * kStageBytes;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int id = i * kGThreads + threadIdx.x;  // 0..511
    const int r = id >> 2, c = id & 3;
    const int64_t k = (int64_t)ks * kBK + c * 16;
    cp_async16(base + swz(r, c), a.xq + (m0 + r) * a.K + k);
    cp_async16(base + kTileBytes + swz(r, c), a.wq + (n0 + r) * a.K + k);
  }
}

template <bool BF16_OUT>
__global__ void __launch_bounds__(kGThreads) k_w8a8_gemm(const __grid_constant__ GemmArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const uint32_t smem = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const int64_t n0 = (int64_t)blockIdx.x * kBN, m0 = (int64_t)blockIdx.y * kBM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp >> 2, wn = warp & 3;  // warp tile: rows wm*64.., cols wn*32..
  const int KT = (int)(a.K / kBK);

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < KT) load_stage(a, smem, s, m0, n0, s);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  // ldmatrix row/chunk of this lane: A (x4 = rows 0-15 x chunks 0-1 of a 16 x 32 slice),
  // B (x4 = n rows 0-15 x chunks 0-1 of a 16 x 32 slice: two n8 tiles)
  const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8, a_chk = lane >> 4;
  const int b_row = (lane & 7) + ((lane >> 4) & 1) * 8, b_chk = (lane >> 3) & 1;

  for (int kt = 0; kt < KT; ++kt) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 2) : "memory");
    __syncthreads();
    // refill the stage consumed one step ago (every warp is past it after the barrier)
    const int nk = kt + kStages - 1;
    if (nk < KT) load_stage(a, smem, nk % kStages, m0, n0, nk);
    asm volatile("cp.async.commit_group;" ::: "memory");

    const uint32_t sa = smem + (kt % kStages) * kStageBytes, sb = sa + kTileBytes;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {  // two k32 slices of the 64-byte step
      uint32_t af[4][4], bf[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = wm * 64 + i * 16 + a_row;
        ldsm_x4(sa + swz(r, kk * 2 + a_chk), af[i][0], af[i][1], af[i][2], af[i][3]);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = wn * 32 + j * 16 + b_row;
        ldsm_x4(sb + swz(r, kk * 2 + b_chk), bf[2 * j][0], bf[2 * j][1], bf[2 * j + 1][0],
                bf[2 * j + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");

  // epilogue: y = float(acc) * (s_x s_w) + b, written once
  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t row = m0 + wm * 64 + i * 16 + g + h * 8;
      const float sx = __ldg(a.sx + row);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t col = n0 + wn * 32 + j * 8 + t4 * 2;
        const float s0 = sx * __ldg(a.sw + col), s1 = sx * __ldg(a.sw + col + 1);
        const float b0 = a.bias ? __ldg(a.bias + col) : 0.f, b1 = a.bias ? __ldg(a.bias + col + 1) : 0.f;
        const float y0 = fmaf((float)acc[i][j][2 * h], s0, b0);
        const float y1 = fmaf((float)acc[i][j][2 * h + 1], s1, b1);
        if constexpr (BF16_OUT) {
          *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(a.y) + row * a.N + col) =
              __floats2bfloat162_rn(y0, y1);
        } else {
          *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.y) + row * a.N + col) = make_float2(y0, y1);
        }
      }
    }
  }
}

template <typename K, typename A>
cudaError_t launch_pdl_args(K kern, dim3 grid, int threads, size_t smem, cudaStream_t st, const A& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t launch_quantize_rows(const QuantArgs& a, t2va_dtype dt, cudaStream_t st) {
  const dim3 grid((unsigned)((a.rows + kQRows - 1) / kQRows));
  if (dt == T2VA_BFLOAT16)
    return a.codes_bf16 ? launch_pdl_args(k_quantize_rows<__nv_bfloat16, true>, grid, kQThreads, 0, st, a)
                        : launch_pdl_args(k_quantize_rows<__nv_bfloat16, false>, grid, kQThreads, 0, st, a);
  return a.codes_bf16 ? launch_pdl_args(k_quantize_rows<float, true>, grid, kQThreads, 0, st, a)
                      : launch_pdl_args(k_quantize_rows<float, false>, grid, kQThreads, 0, st, a);
}

int gemm_tile_m() { return kBM; }
int gemm_tile_n() { return kBN; }
int gemm_tile_k() { return kBK; }

cudaError_t launch_w8a8_gemm(const GemmArgs& a, bool bf16_out, cudaStream_t st) {
  // once per process (a function-local static is initialised exactly once, thread-safely)
  static const cudaError_t smem_attr = [] {
    cudaError_t e = cudaFuncSetAttribute(k_w8a8_gemm<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_w8a8_gemm<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    return e;
  }();
  if (smem_attr != cudaSuccess) return smem_attr;
  const dim3 grid((unsigned)(a.N / kBN), (unsigned)(a.M / kBM));
  if (bf16_out) return launch_pdl_args(k_w8a8_gemm<true>, grid, kGThreads, kGemmSmem, st, a);
  return launch_pdl_args(k_w8a8_gemm<false>, grid, kGThreads, kGemmSmem, st, a);
}

}  // namespace t2va
