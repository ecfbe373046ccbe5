/*
 * t2va.h - C ABI of the joint video-audio distillation objective library
 * (TurboT2VA joint sCM + DMD objective; NVIDIA B300, sm_103a).
 *
 * The library computes, on the GPU, one data-parallel step of TurboT2VA's
 * distillation objective over paired video and audio latents that share one
 * timestep per sample: TrigFlow noising, the joint sCM direction with its
 * per-sample, per-modality L2 normalisation, the DMD term with its
 * residual-scale normaliser, the per-sample losses and the float32 gradients
 * with respect to the student outputs. Next to it: the TrigFlow -> rectified-flow
 * wrapper fused into the noising, the DMD teacher guided per modality, and from the
 * inference stack the post-scale W8A8 linear and the fused residual + modulated RMS
 * normalisation.
 *
 * Sources (cited per entry point below):
 *   [zh] "TurboT2VA：分数正则化一致性蒸馏加速 19B 视频音频联合生成，四步采样
 *        20.1×、H20 上全栈 54.67×" (robotworld.top/zh/papers/paper-2608.24674),
 *        sections 三, 3.1, 四, 4.1, 4.2, 6.2, 6.3, 七 (the only page printing the
 *        equations).
 *   [en] "TurboT2VA: Score-Regularized Consistency Distillation for Fast
 *        Large-Scale Text-to-Video-Audio Generation"
 *        (robotworld.top/en/papers/paper-2608.24674): Eq. 6 (per-modality L2
 *        normalisation), Eq. 11-12 (DMD residual-scale normaliser), Eq. 16
 *        (TrigFlow -> rectified-flow wrapper).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - A batch holds `batch` samples; each sample has `num_modalities` latents
 *   (modality 0 = video, 1 = audio in the paper; up to T2VA_MAX_MODALITIES).
 * - Latent m of sample b is seg[m].numel contiguous elements starting at
 *   element b * seg[m].sample_stride of each per-modality buffer. All buffers of
 *   one modality (inputs and float32 gradients) share this geometry; the
 *   element order inside a sample is irrelevant (the objective reduces over all
 *   elements of a sample and modality).
 * - Pointer arrays (`const void* const* x`) are HOST arrays of num_modalities
 *   DEVICE pointers. Every device pointer must be 16-byte aligned. Scalars `t`
 *   (per-sample timesteps, float32 [batch]) and the outputs are DEVICE pointers.
 *   `weight` is a HOST array of num_modalities floats (w_m).
 * - Inputs are float32 or bfloat16 (`dtype`); arithmetic is float32 with
 *   float32 accumulation; gradients are written in float32.
 * - The caller owns every buffer and the stream. The library allocates no
 *   device memory (it has two static device arrays: the scratch of
 *   t2va_stage3_objective_noalloc and the buffers of t2va_selftest_wait_timeout),
 *   keeps no state across calls, and never synchronises the host: calls are
 *   asynchronous on `stream`. Outputs must not overlap inputs unless an entry
 *   point says so.
 * - Return value: T2VA_SUCCESS or a synchronous error code (argument checks,
 *   launch failure); nothing is enqueued when an error is returned. Problems
 *   found on the device set bits in the caller's device int `*status`
 *   (OR-ed, never cleared by the library).
 * - Tails and per-sample offsets that are not multiples of the 16-byte vector
 *   width are handled, not rejected.
 */
#ifndef T2VA_H
#define T2VA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define T2VA_ABI_VERSION 3  /* 2: t2va_noise_rf, t2va_stage3_objective_cfg, W8A8, t2va_residual_modnorm;
                               3: t2va_objective_plan_query */
#define T2VA_MAX_MODALITIES 4

typedef enum t2va_dtype {
  T2VA_FLOAT32 = 0,
  T2VA_BFLOAT16 = 1,
  T2VA_INT8 = 2       /* W8A8 codes only */
} t2va_dtype;

/* Geometry of one modality: elements per sample and the distance (in elements)
 * between the first elements of consecutive samples (>= numel when batch > 1). */
typedef struct t2va_segment {
  int64_t numel;
  int64_t sample_stride;
} t2va_segment;

/* Synchronous return codes. */
enum {
  T2VA_SUCCESS = 0,
  T2VA_ERROR_INVALID_ARGUMENT = 1,  /* bad size, scalar or null pointer          */
  T2VA_ERROR_UNSUPPORTED_DTYPE = 2, /* a dtype the entry point does not take        */
  T2VA_ERROR_MISALIGNED = 3,        /* a device pointer breaks its alignment rule  */
  T2VA_ERROR_WORKSPACE = 4,         /* workspace null, misaligned or too small     */
  T2VA_ERROR_CUDA = 5               /* a CUDA runtime call or launch failed        */
};

/* Device status bits, OR-ed into *status by the kernels. */
#define T2VA_STATUS_BAD_TIMESTEP 0x1  /* a sample's t is outside (0, pi/2): its outputs are NaN    */
/* A bounded pipeline wait of the tensor-core W8A8 kernel ran out (its output is
 * incomplete). No objective kernel waits on another CTA, so the objective never sets it. */
#define T2VA_STATUS_TIMEOUT 0x2
/* Never set: no kernel reads the workspace header (the bit keeps its value for ABI
 * compatibility). */
#define T2VA_STATUS_BAD_WORKSPACE 0x4

/* Static description of a return code (never NULL). */
const char* t2va_error_string(int code);

/* T2VA_ABI_VERSION of the loaded library. */
int t2va_abi_version(void);

/* Bytes of workspace needed by the objective entry points for up to `batch`
 * samples of `num_modalities` modalities: 256 bytes plus 16 KiB per (sample,
 * modality). An objective call is two kernels on `stream` (both programmatic
 * dependents of the work before them); the first writes
 * per-chunk partial sums into the workspace and the second reads them, so the
 * workspace needs no initialisation and keeps nothing between calls. Calls that
 * may run concurrently need distinct workspaces. Returns 0 on invalid arguments
 * or if no device can be queried. */
size_t t2va_workspace_bytes(int batch, int num_modalities);

/* The launch plan of an objective call (t2va_scm_objective, t2va_dmd_objective and the
 * t2va_stage3_objective family) for these sizes on a GPU with `sm_count` SMs. Host
 * arithmetic only: no device is touched and nothing is enqueued, so it runs without a
 * GPU. The plan depends only on the arguments given here.
 *
 * Each (sample, modality) row is cut into chunks of `vectors_per_chunk` 16-byte
 * vectors (8 bfloat16 or 4 float32 elements; the unaligned head and tail elements of a
 * sample go to its first and last chunk); both kernels of a call launch one CTA per
 * chunk of every row of every sample.
 *   grid               CTAs per kernel: batch * sum_m chunks[m]
 *   threads            threads per CTA
 *   vectors_per_chunk  16-byte vectors per chunk
 *   chunks[m]          chunks per row of modality m, 1 ... 1024 (entries past
 *                      num_modalities are 0)
 *   outputs_modality, outputs_chunk
 *                      the chunk of every sample whose CTA also writes the per-sample
 *                      outputs (loss, norm, cdmd): the shortest last chunk of a row
 *   one_wave           1 when the grid fits in one wave of three CTAs per SM
 * Returns T2VA_SUCCESS, T2VA_ERROR_INVALID_ARGUMENT (a geometry the objective entry
 * points reject, sm_count < 1, a null `out`, or sizes no plan covers) or
 * T2VA_ERROR_UNSUPPORTED_DTYPE. */
typedef struct t2va_objective_plan {
  int grid;
  int threads;
  int vectors_per_chunk;
  int chunks[T2VA_MAX_MODALITIES];
  int outputs_modality;
  int outputs_chunk;
  int one_wave;
} t2va_objective_plan;

int t2va_objective_plan_query(int batch, int num_modalities, const t2va_segment* seg,
                              t2va_dtype dtype, int sm_count, t2va_objective_plan* out);

/* Zero a workspace (16-byte aligned device memory of `workspace_bytes`) on
 * `stream` and write its header. Optional: the objective entry points do not
 * depend on the workspace's contents. `timeout_ms` is ignored (kept for ABI
 * compatibility). */
int t2va_workspace_init(void* workspace, size_t workspace_bytes, uint32_t timeout_ms,
                        cudaStream_t stream);

/* TrigFlow noising  ([zh] section 三, the noising equation; [en] section 2):
 *   z_t^m = cos(t_b) * z0^m + sin(t_b) * eps^m    for every modality m,
 * with one shared t_b per sample and independent eps per modality. z0, eps and
 * zt have the same dtype; zt may be the same buffer as z0 or eps (in place).
 * Results are rounded to the output dtype (round to nearest even); every finite
 * t is accepted. `status` may be NULL; a non-finite t sets
 * T2VA_STATUS_BAD_TIMESTEP. Reads 2 and writes 1 element per latent element. */
int t2va_noise(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
               const void* const* z0, const void* const* eps, void* const* zt,
               const float* t, int* status, cudaStream_t stream);

/* TrigFlow noising fused with the TrigFlow -> rectified-flow wrapper
 * ([zh] 4.2; [en] Eq. 16), for a backbone trained in the rectified-flow
 * parameterisation:
 *   z_t^m  = cos(t_b) z0^m + sin(t_b) eps^m                  (as t2va_noise),
 *   z_rf^m = z_t^m / (cos t_b + sin t_b),
 *   t_rf[b] = sin t_b / (cos t_b + sin t_b),
 * so z_rf = (1 - t_rf) z0 + t_rf eps. Both latents come from one read of z0 and
 * eps, each rounded once from float32 arithmetic to the latent dtype.
 * `zt` may be NULL (only z_rf is written); `z_rf` is required; a zt[m] that is the
 * same buffer as z_rf[m] is an error; either may be the same buffer as z0 or eps
 * (in place). `t_rf` (device float [batch]) may be NULL. Every finite t is
 * accepted (t in [0, pi/2] keeps cos t + sin t >= 1); `status` may be NULL; a
 * non-finite t sets T2VA_STATUS_BAD_TIMESTEP. Reads 2 and writes 1 or 2 elements
 * per latent element. */
int t2va_noise_rf(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                  const void* const* z0, const void* const* eps, void* const* zt,
                  void* const* z_rf, const float* t, float* t_rf, int* status,
                  cudaStream_t stream);

/* Joint sCM objective  ([zh] 3.1; [en] Eq. 6). Per sample b and modality m,
 * with c = cos t_b, s = sin t_b and elementwise
 *   F_T = (c z_t - x0_teacher)/s,  F_theta = (c z_t - x0_student)/s,
 *   J   = c s (dF_theta/dt + dF_theta/dz^v F_T^v + dF_theta/dz^a F_T^a)
 *         assembled from `x0_student_tangent`, the tangent of the student x0
 *         prediction along (dt, dz^v, dz^a) = (1, F_T^v, F_T^a),
 *   g   = -beta c / sqrt(1 - gamma^2 s^2) (sg(F_theta) - F_T) - gamma c s z_t - J,
 *   g_bar = g / (||g||_2 + eps_scm)    (norm over the sample's elements of m),
 *   r   = F_theta - sg(F_theta) - g_bar,
 * it writes
 *   loss[b] = lambda_scm * sum_m weight[m] ||r_m||^2          (device float [batch]),
 *   norm[b*M + m] = ||g_m||_2      (device float [batch*M], may be NULL),
 *   grad_x0_student[m] = d(sum_b loss[b]) / d x0_student = 2 lambda w_m g_bar / s
 *     (float32, same geometry as the inputs; added to the buffer's contents
 *      when `accumulate` is non-zero, overwritten otherwise).
 * The whole g_bar is a stop-gradient target. Requires beta finite,
 * 0 <= gamma <= 1, eps_scm > 0, weight[m] >= 0. A sample with t outside
 * (0, pi/2) gets NaN outputs and sets T2VA_STATUS_BAD_TIMESTEP. `workspace`
 * must hold t2va_workspace_bytes(batch, M) bytes (16-byte aligned). `status`
 * is required. Runs as two kernels on `stream` (sums, then gradients); each
 * input is read from HBM once when the call's inputs fit in L2, else twice. */
int t2va_scm_objective(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                       const void* const* z_t, const void* const* x0_teacher,
                       const void* const* x0_student, const void* const* x0_student_tangent,
                       const float* t, float beta, float gamma, float eps_scm,
                       const float* weight, float lambda_scm,
                       float* const* grad_x0_student, int accumulate,
                       float* loss, float* norm,
                       void* workspace, size_t workspace_bytes, int* status,
                       cudaStream_t stream);

/* Joint DMD objective  ([zh] 四; [en] Eq. 11-12). On the re-noised on-policy
 * sample, with y_T = x0_teacher_hat and y_fake = x0_fake (the teacher and
 * fake-score x0 predictions at zhat_t):
 *   g = y_fake - y_T,  c_m = (1/N_m) sum_i |zhat0_i - y_T,i|,
 *   g_bar = g / (c_m + eps_dmd),  Delta = zhat0 - sg(zhat0 - g_bar),
 *   loss[b] = lambda_dmd * sum_m weight[m] sum_i Delta_i^2   (a sum over elements),
 *   cdmd[b*M + m] = c_m  (may be NULL),
 *   grad_zhat0[m] = 2 lambda_dmd w_m g_bar (float32; `accumulate` as above).
 * A modality with numel 0 contributes 0 and reports c_m = 0. Requires
 * eps_dmd > 0, weight[m] >= 0. Does not depend on t. */
int t2va_dmd_objective(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                       const void* const* zhat0, const void* const* x0_teacher_hat,
                       const void* const* x0_fake, float eps_dmd, const float* weight,
                       float lambda_dmd, float* const* grad_zhat0, int accumulate,
                       float* loss, float* cdmd,
                       void* workspace, size_t workspace_bytes, int* status,
                       cudaStream_t stream);

/* Stage-3 objective  ([zh] 4.1; [en] section 3):
 *   loss[b] = lambda_scm L_sCM,b + lambda_dmd L_DMD,b
 * over the same batch and the same per-sample t, with both terms as defined
 * above and one set of weights w_m. Two kernels on `stream`: the first reads the
 * seven inputs for the sums, the second reads them again (from L2 when they fit
 * there) and writes both gradients once. `loss_scm` and `loss_dmd` (device float
 * [batch], each already multiplied by its lambda) may be NULL, as may `norm`
 * and `cdmd`. If grad_zhat0[m] == grad_x0_student[m] (the caller's on-policy
 * sample is the student output itself), the two gradients are summed into
 * that one buffer. A sample with t outside (0, pi/2) gets NaN in every output. */
int t2va_stage3_objective(int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
                          const void* const* z_t, const void* const* x0_teacher,
                          const void* const* x0_student, const void* const* x0_student_tangent,
                          const float* t,
                          const void* const* zhat0, const void* const* x0_teacher_hat,
                          const void* const* x0_fake,
                          float beta, float gamma, float eps_scm, float eps_dmd,
                          const float* weight, float lambda_scm, float lambda_dmd,
                          float* const* grad_x0_student, float* const* grad_zhat0, int accumulate,
                          float* loss, float* loss_scm, float* loss_dmd, float* norm, float* cdmd,
                          void* workspace, size_t workspace_bytes, int* status,
                          cudaStream_t stream);

/* Stage-3 objective with a guided teacher ([zh] 四 and 七; [en] section 3: the
 * teacher prediction of the DMD term is computed with classifier-free guidance,
 * at a scale per modality, 3.0 for video and 5.0 for audio in the paper's
 * training). Per element, in float32,
 *   y_T = u + guidance[m] (k - u),   k = x0_teacher_hat_cond, u = x0_teacher_hat_uncond,
 * and then exactly t2va_stage3_objective with x0_teacher_hat = y_T. `guidance`
 * is a host array of num_modalities finite floats; x0_teacher_hat_uncond has
 * the geometry of the other latents. The guided prediction is never stored:
 * each pass reads k and u (eight inputs for the sums, seven for the gradients). */
int t2va_stage3_objective_cfg(
    int batch, int num_modalities, const t2va_segment* seg, t2va_dtype dtype,
    const void* const* z_t, const void* const* x0_teacher, const void* const* x0_student,
    const void* const* x0_student_tangent, const float* t, const void* const* zhat0,
    const void* const* x0_teacher_hat_cond, const void* const* x0_teacher_hat_uncond,
    const float* guidance, const void* const* x0_fake, float beta, float gamma, float eps_scm,
    float eps_dmd, const float* weight, float lambda_scm, float lambda_dmd,
    float* const* grad_x0_student, float* const* grad_zhat0, int accumulate, float* loss,
    float* loss_scm, float* loss_dmd, float* norm, float* cdmd, void* workspace,
    size_t workspace_bytes, int* status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Post-scale W8A8 linear  ([zh] 6.2; [en] section 6): static per-output-channel
 * weight quantisation, dynamic per-row activation quantisation, an exact INT32
 * sum over the whole K, and both scales applied once, after the sum:
 *   s_i = max(||x_i||_inf, eps) / 127,  x_hat_i = clip(round(x_i / s_i), -127, 127),
 *   y_ij = s_i^x s_j^w sum_k x_hat_ik w_hat_jk + b_j.
 * --------------------------------------------------------------------------- */

/* Quantise `rows` rows of `cols` elements (bfloat16 or float32, row i at
 * x + i * ld_x elements) into codes (row i at q + i * ld_q code elements) and float32
 * scales scale[i] = max(amax_i, eps) / 127. Each code is rint of the correctly rounded
 * float32 quotient x / s (ties to even), clipped to [-127, 127], so codes are exact
 * functions of the inputs. `code_dtype` is T2VA_INT8 (one byte per code) or
 * T2VA_BFLOAT16 (the same integers stored as bfloat16, exact, for the tensor-core
 * contraction below). Use it for the activations before every linear and once for each
 * weight matrix (rows = output channels). Requires eps > 0, cols a multiple of 16
 * bytes of input (8 bf16 or 4 float32 elements), ld_x * element size a multiple of 16,
 * ld_q a multiple of the codes written per input vector (16 / element size), x and q
 * 16-byte aligned. 128 threads per row: reads each input once (rows longer than 8 KiB
 * are read a second time, from L2). One kernel on `stream`. */
int t2va_quantize_rows(int64_t rows, int64_t cols, t2va_dtype dtype, const void* x, int64_t ld_x,
                       float eps, t2va_dtype code_dtype, void* q, int64_t ld_q, float* scale,
                       cudaStream_t stream);

/* y[M][N] (row-major, bfloat16 or float32 per `out_dtype`) from activation codes
 * xq[M][K] with scales sx[M] and weight codes wq[N][K] with scales sw[N] (both
 * K-contiguous, of `code_dtype`), and an optional bias[N] (NULL for none). The integer
 * sum is exact; the epilogue is y = fma(float(acc), sx_i * sw_j, b_j) in float32,
 * rounded once to `out_dtype`. Shapes are guarded as in the paper: M, N and K must be
 * multiples of 128 (else T2VA_ERROR_INVALID_ARGUMENT; the caller keeps its own BF16
 * linear for other shapes), and K <= 131072 so that no INT32 sum can overflow.
 *   - T2VA_INT8 codes: the warp-level INT8 MMA (mma.sync m16n8k32 s8). sm_103a has no
 *     INT8 form of the fifth-generation tensor-core MMA.
 *   - T2VA_BFLOAT16 codes: tcgen05.mma (bf16 x bf16 -> f32 in TMEM), K summed in chunks
 *     of 1024 whose float32 sums stay below 2^24 and are therefore exact integers, the
 *     chunks added as int32. Same result, at the bf16 tensor-core rate: 128 x 256 tiles
 *     on one persistent CTA per SM when N is a multiple of 256, else 128 x 128 tiles.
 *     Needs y 16-byte aligned. Its pipeline waits are bounded: a wait that runs out sets
 *     T2VA_STATUS_TIMEOUT in `status` (may be NULL) and leaves y incomplete.
 * One kernel on `stream`. */
int t2va_w8a8_linear(int64_t M, int64_t N, int64_t K, t2va_dtype code_dtype, const void* xq,
                     const float* sx, const void* wq, const float* sw, const float* bias,
                     t2va_dtype out_dtype, void* y, int* status, cudaStream_t stream);

/* Fused gated residual update + modulated RMS normalisation  ([zh] 6.3: the joint
 * Transformer combines a normalisation with a modality- and timestep-dependent
 * modulation, then a gated residual update; the pages print no formulas, and the
 * standard diffusion-Transformer forms are taken). Per token row r of D contiguous
 * elements, with sample b = r / rows_per_sample:
 *   h'[r] = h[r] + gate[b] * u[r]                          (if u is given; else h' = h)
 *   y[r]  = h'[r] / sqrt(mean(h'[r]^2) + eps) * (1 + scale[b]) + shift[b]
 * h' is rounded to `dtype` and the normalisation uses the rounded values. gate, scale
 * and shift are float32 [samples][D] device arrays, each may be NULL (gate 1, scale 0,
 * shift 0; gate only with u). h' is stored in `h_out` if it is not NULL (h_out may be
 * h, an in-place update; it needs u). y may not be h, u or h_out. Requires D a multiple
 * of 16 bytes of elements, rows_per_sample >= 1, eps >= 0, every pointer 16-byte
 * aligned. One kernel on `stream`, 128 threads per row; reads h (and u) once and writes
 * h' and y once. */
int t2va_residual_modnorm(int64_t rows, int64_t D, int64_t rows_per_sample, t2va_dtype dtype,
                          const void* h, const void* u, const float* gate, const float* scale,
                          const float* shift, float eps, void* h_out, void* y, cudaStream_t stream);

/* Self-test of the tensor-core W8A8 kernel's bounded waits: one 128 x 128 x 128 launch on
 * library-owned buffers whose MMA thread first waits on an mbarrier that nothing arrives
 * on. The wait runs out after about a second; the kernel then sets
 * T2VA_STATUS_TIMEOUT in *status (a device int), drains its copies, frees its TMEM and
 * returns, and the context stays usable. A tensor-core W8A8 launch given a status word
 * that already holds T2VA_STATUS_TIMEOUT does nothing, so clear it before reusing it. */
int t2va_selftest_wait_timeout(int* status, cudaStream_t stream);

/* Bytes of the library's own scratch array used by
 * t2va_stage3_objective_noalloc (1 MiB). Every GPU on which the library's module
 * is loaded holds this much device memory until the process exits. */
#define T2VA_NOALLOC_SCRATCH_BYTES (1u << 20)

/* The stage-3 objective without a caller-provided workspace.
 *
 * The paper has no counterpart: this entry point is for callers that cannot
 * allocate device memory. Examples are code that runs inside another runtime's
 * memory pool or under an allocator that owns all device memory, plugins that
 * get only their inputs and outputs from a host, and hosts that forbid
 * allocation after set-up. Such callers cannot provide the workspace that
 * t2va_stage3_objective needs.
 *
 * The arguments, outputs and results are those of t2va_stage3_objective,
 * without `workspace` and `workspace_bytes`. In their place the call uses a
 * scratch array owned by the library: T2VA_NOALLOC_SCRATCH_BYTES of static
 * device memory per GPU. The call allocates nothing: no cudaMalloc, no cudaFree
 * and no allocating library routine.
 *
 * - Limit: the partial sums of the call (16 KiB per sample and modality, the
 *   workspace that t2va_workspace_bytes counts without its 256-byte header) must
 *   fit in the scratch, so at most 32 samples of 2 modalities per call. A larger
 *   batch returns T2VA_ERROR_WORKSPACE, and nothing is enqueued.
 * - First call: the first call on each device, with that device current, looks
 *   up the scratch's device address (cudaGetSymbolAddress) and keeps it. Under
 *   CUDA's lazy module loading that lookup is also what loads the library's module
 *   and its 1 MiB array onto the device, so the first call can fail with
 *   T2VA_ERROR_CUDA when device memory is exhausted: make it during set-up, before
 *   the host's allocator takes the memory and before any stream capture on that
 *   device. A device reset (cudaDeviceReset) unloads the module and invalidates
 *   the kept address: do not call this entry point again after one.
 * - Sharing: every call on a device shares the one scratch array. A call's first
 *   kernel writes the partial sums its second kernel reads, so the array needs no
 *   clearing, but calls that overlap on the GPU (on different streams or from
 *   different host threads) race on it and give wrong results. Order them on one
 *   stream, or use t2va_stage3_objective with one workspace per concurrent call.
 * - Errors: argument errors are those of t2va_stage3_objective, returned before
 *   anything is enqueued. T2VA_ERROR_CUDA means the scratch's address could not
 *   be obtained. */
int t2va_stage3_objective_noalloc(int batch, int num_modalities, const t2va_segment* seg,
                                  t2va_dtype dtype, const void* const* z_t,
                                  const void* const* x0_teacher, const void* const* x0_student,
                                  const void* const* x0_student_tangent, const float* t,
                                  const void* const* zhat0, const void* const* x0_teacher_hat,
                                  const void* const* x0_fake, float beta, float gamma,
                                  float eps_scm, float eps_dmd, const float* weight,
                                  float lambda_scm, float lambda_dmd,
                                  float* const* grad_x0_student, float* const* grad_zhat0,
                                  int accumulate, float* loss, float* loss_scm, float* loss_dmd,
                                  float* norm, float* cdmd, int* status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* T2VA_H */
