// Allocation-free variant of the stage-3 objective entry point.
//
// Some callers cannot call cudaMalloc, or any routine that allocates: code that
// runs inside another runtime's memory pool or under a custom allocator that
// owns all device memory, plugins that get only the inputs and outputs from
// their host, and hosts that forbid allocation once set-up is over. They cannot
// provide the caller-owned workspace that t2va_stage3_objective needs. This
// entry point uses instead a scratch array of fixed size that belongs to the
// library: a file-scope __device__ array, held by every GPU that loads the
// library until the process exits. The caller still passes every input and
// output buffer.
//
// Host code cannot use the array's name as a device address: on the host it
// names a host-side stand-in. So the first call on each device, with that
// device current, asks the runtime for the array's device address
// (cudaGetSymbolAddress) and keeps it; later calls on that device reuse it. A
// device reset (cudaDeviceReset) unloads the module and invalidates that address:
// a process that resets a device must not call this entry point afterwards.
#include <mutex>

#include "t2va_internal.cuh"

using namespace t2va;

namespace {

static_assert(T2VA_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

// The scratch array. Every call on a device shares it.
static __device__ __align__(256) unsigned char g_scratch[T2VA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_dev[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_scratch on the current device, looked up once per device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return T2VA_ERROR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return T2VA_ERROR_CUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return T2VA_SUCCESS;
}

}  // namespace

extern "C" int t2va_stage3_objective_noalloc(
    int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
    const void* const* z_t, const void* const* x0_teacher, const void* const* x0_student,
    const void* const* x0_student_tangent, const float* t, const void* const* zhat0,
    const void* const* x0_teacher_hat, const void* const* x0_fake, float beta, float gamma,
    float eps_scm, float eps_dmd, const float* weight, float lambda_scm, float lambda_dmd,
    float* const* grad_x0_student, float* const* grad_zhat0, int accumulate, float* loss,
    float* loss_scm, float* loss_dmd, float* norm, float* cdmd, int* status,
    cudaStream_t stream) {
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != T2VA_SUCCESS) return rc;
  // the scratch is the workspace's partial-sum area (no header is needed)
  const WsRef ws{reinterpret_cast<unsigned char*>(scratch), (size_t)T2VA_NOALLOC_SCRATCH_BYTES};
  // The same checks, in the same order, as t2va_stage3_objective: every argument check,
  // then the scratch must hold what this batch needs (else T2VA_ERROR_WORKSPACE), and
  // nothing is enqueued on an error. The scratch keeps what the last call left there;
  // that is harmless, because the call's first kernel writes every partial sum its
  // second kernel reads.
  return stage3_entry(batch, num_modalities, seg, dtype, z_t, x0_teacher, x0_student,
                      x0_student_tangent, t, zhat0, x0_teacher_hat, nullptr, nullptr, x0_fake,
                      beta, gamma, eps_scm, eps_dmd, weight, lambda_scm, lambda_dmd,
                      grad_x0_student, grad_zhat0, accumulate, loss, loss_scm, loss_dmd, norm,
                      cdmd, ws, status, stream);
}
