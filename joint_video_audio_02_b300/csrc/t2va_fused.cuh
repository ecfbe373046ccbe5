// Declarations shared by the fused residual + normalisation kernel (t2va_fused.cu) and
// the C ABI.
#pragma once

#include "t2va_internal.cuh"

namespace t2va {

struct FusedArgs {
  int64_t rows, D;             // token rows of D contiguous elements
  int64_t rows_per_sample;     // row r belongs to sample r / rows_per_sample
  const void* h;               // [rows][D] latent dtype
  const void* u;               // [rows][D] or null (no residual update)
  const float* gate;           // [samples][D] or null (1)
  const float* scale;          // [samples][D] or null (0)
  const float* shift;          // [samples][D] or null (0)
  float eps;
  void* h_out;                 // [rows][D] or null (h' not stored)
  void* y;                     // [rows][D]
};

cudaError_t launch_residual_modnorm(const FusedArgs& a, t2va_dtype dt, cudaStream_t st);

}  // namespace t2va
