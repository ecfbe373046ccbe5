// Declarations shared by the W8A8 kernels (t2va_w8a8.cu, t2va_w8a8_tc.cu) and the C ABI.
#pragma once

#include "t2va_internal.cuh"

namespace t2va {

// Per-row dynamic quantisation (t2va_w8a8.cu).
struct QuantArgs {
  int64_t rows, cols;
  bool codes_bf16;             // codes stored as bfloat16 integers instead of int8
  const void* x;               // bf16 or float32 [rows][ld_x]
  int64_t ld_x;                // elements
  void* q;                     // [rows][ld_q] codes
  int64_t ld_q;                // code elements
  float* scale;                // [rows]
  float eps;
};

// INT8 GEMM with the post-scale epilogue (t2va_w8a8.cu): y[M][N] from xq[M][K] and
// wq[N][K], both K-contiguous.
constexpr int64_t kW8a8MaxK = 131072;  // 131072 * 127 * 127 < 2^31

struct GemmArgs {
  int64_t M, N, K;
  const int8_t* xq;            // int8 codes, or bfloat16 codes for the tensor-core path
  const float* sx;
  const int8_t* wq;            // as xq
  const float* sw;
  const float* bias;           // [N] or null
  void* y;                     // bf16 or float32 [M][N]
  int* status;                 // device status word or null (tensor-core path)
  int selftest_wait;           // tensor-core path: first wait on a barrier nothing arrives on
};

cudaError_t launch_quantize_rows(const QuantArgs& a, t2va_dtype dt, cudaStream_t st);
cudaError_t launch_w8a8_gemm(const GemmArgs& a, bool bf16_out, cudaStream_t st);
cudaError_t launch_w8a8_tc(const GemmArgs& a, bool bf16_out, cudaStream_t st);
// One 128 x 128 x 128 tensor-core launch on library-owned buffers whose MMA thread first
// waits on a barrier that nothing arrives on (a test of the bounded waits).
cudaError_t launch_w8a8_tc_selftest(int* status, cudaStream_t st);
int gemm_tile_m();
int gemm_tile_n();
int gemm_tile_k();

}  // namespace t2va
