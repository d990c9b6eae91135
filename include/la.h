/*
 * la.h -- C ABI of the GB300 (sm_103a) fused linear-attention library (libla.so).
 *
 * The operation (module neuralops.core.triton_kernels.linear_attn, functions `fwd` and
 * `bwd`; feature list in that module's docstring: feature maps elu+1 and relu, chunked
 * causal streaming, bidirectional parallel reduction, cosFormer cos/sin modulation):
 *
 *   a_i^p = w_i^p phi(q_i),  b_j^p = w_j^p phi(k_j)
 *   S_i^p = sum_{j in J(i)} b_j^p v_j^T,  z_i^p = sum_{j in J(i)} b_j^p
 *   out_i = (sum_p (a_i^p)^T S_i^p) / (sum_p a_i^p . z_i^p + eps)
 *
 * J(i) = {j <= i} (causal) or all j (bidirectional); phi(x) = elu(x) + 1, relu(x) or x;
 * without position weights there is one term p with w = 1, with them there are two:
 * w^cos = cos_weight and w^sin = sin_weight.  la_bwd returns the exact gradient of la_fwd
 * (the page's `bwd` differentiates `fwd`).
 *
 * Grouped-query attention (module neuralops.core.triton_kernels.gqa, `fwd`/`bwd`): with
 * Hkv key/value heads and Hq = n_rep * Hkv query heads, query head h reads key/value head
 * h / n_rep, and dk, dv are the sums over the n_rep query heads of each group.  The
 * expanded key/value tensors are never formed.
 *
 * Layout: q, out, grad_out, dq are contiguous [B, Hq, N, D]; k, v, dk, dv are contiguous
 * [B, Hkv, N, D] (row-major, D fastest); la_fwd_strided and la_bwd_strided take inputs with
 * other strides (D still contiguous).  la_fwd_v and la_bwd_v take a value width Dv of its
 * own: v, dv [B, Hkv, N, Dv] and out, grad_out [B, Hq, N, Dv] (`fwd` takes v as a tensor of
 * its own and reads only q's head dimension; the state S = sum b v^T is then D x Dv).  Elements are float32 (LA_F32) or
 * bfloat16 (LA_BF16); outputs use the input type.  Arithmetic is float32 accumulation in
 * both cases (bfloat16 tensor-core operands on the LA_BF16 fast path).  cos_weight and
 * sin_weight are float32 device vectors of length N, indexed by position, applied to
 * phi(q_i) and phi(k_i); give both or neither.
 *
 * Ownership: every pointer is caller-owned device memory (except where a function says
 * host).  The library allocates no device memory: scratch comes from the caller's
 * workspace of at least la_workspace_size() bytes, 256-byte aligned.  Outputs are fully
 * overwritten, never accumulated into.  The workspace must not be shared by calls that
 * can run at the same time.
 *
 * Execution: la_fwd and la_bwd only enqueue kernels on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and return; they never synchronise.  Kernels are launched with
 * programmatic stream serialization, so a kernel's blocks may be placed while the previous
 * kernel's last blocks finish; each kernel waits for the work before it on the stream to
 * complete (griddepcontrol.wait) before it touches memory, so stream order holds as for
 * plain launches.  Their status covers
 * argument checks and launch errors.  Errors found by a kernel while it runs (a bounded
 * wait that ran out) are latched in a device word that la_get_status() reads.
 *
 * Errors: no exception crosses this ABI and no kernel traps.
 *   LA_ERR_ARG          null required pointer, B, Hq, Hkv, N or D <= 0, Hq % Hkv != 0,
 *                       eps negative or not finite, unknown dtype or phi, exactly one of
 *                       cos_weight / sin_weight given, sizes whose element count
 *                       overflows 64 bits
 *   LA_ERR_UNSUPPORTED  D (or Dv) not in {32, 64, 128}
 *   LA_ERR_ALIGN        a pointer that is not 16-byte aligned (workspace: 256-byte)
 *   LA_ERR_WORKSPACE    ws_bytes < la_workspace_size(...) or workspace NULL while needed;
 *                       (from la_get_status) la_bwd_from_fwd got a workspace that another
 *                       la_fwd call wrote
 *   LA_ERR_CUDA         a CUDA launch or runtime error (see la_last_cuda_error())
 *   LA_ERR_TIMEOUT      (from la_get_status) a kernel's bounded wait ran out
 * All argument checks run on the host before any CUDA call.
 */
#ifndef LA_H
#define LA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_ARG = 1,
    LA_ERR_UNSUPPORTED = 2,
    LA_ERR_ALIGN = 3,
    LA_ERR_CUDA = 4,
    LA_ERR_TIMEOUT = 5,
    LA_ERR_WORKSPACE = 6
} la_status;

/* Feature map phi: elu(x) + 1 with alpha = 1, max(x, 0), or x itself (identity: the
 * caller's q and k are the features; the linear_attn page lists the maps as non-negative,
 * so identity expects non-negative q and k: with signed features the denominator can
 * vanish and the result is ill-conditioned or non-finite). */
typedef enum { LA_PHI_ELU1 = 0, LA_PHI_RELU = 1, LA_PHI_IDENTITY = 2 } la_phi;

/* Element type of q, k, v, grad_out and of every output. */
typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

/* Which kernel family a call with these arguments runs. */
typedef enum { LA_PATH_SIMT = 0, LA_PATH_TCGEN05 = 1 } la_path;

/* Element strides of a [B, H, N, D] input along B, H and N; its last dimension (D) is
 * contiguous.  E.g. q taken from a fused [B, N, 3, H, D] projection as qkv[:, :, 0]
 * permuted to [B, H, N, D]: b = 3 N H D, h = D, n = 3 H D. */
typedef struct {
    long long b, h, n;
} la_strides;

/* Bytes of workspace that la_fwd (is_bwd = 0) or la_bwd (is_bwd = 1) needs for these
 * sizes.  Host-only, never fails: returns 0 for arguments la_fwd / la_bwd would reject.
 * has_weights: 1 when cos_weight and sin_weight are given. */
size_t la_workspace_size(int B, int Hq, int Hkv, int N, int D, la_dtype dtype, int is_causal,
                         int has_weights, int is_bwd);

/* Kernel family chosen for these arguments (host-only; for tests and reports): the
 * tensor-core kernels (LA_PATH_TCGEN05) for bfloat16 at D = 64 or 128 with n_rep = Hq / Hkv
 * in {1, 2, 4, 8}, forward and backward (with cos/sin weights as two passes, one per term);
 * the CUDA-core kernels (LA_PATH_SIMT) otherwise. */
la_path la_kernel_path(int B, int Hq, int Hkv, int N, int D, la_dtype dtype, int is_causal,
                       int has_weights, int is_bwd);

/* la_workspace_size and la_kernel_path for a value width Dv (la_fwd_v, la_bwd_v).  Dv != D
 * runs on the CUDA-core kernels. */
size_t la_workspace_size_v(int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dtype, int is_causal,
                           int has_weights, int is_bwd);
la_path la_kernel_path_v(int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dtype, int is_causal,
                         int has_weights, int is_bwd);

/* Forward, `linear_attn.fwd(q, k, v, is_causal, phi, eps, cos_weight, sin_weight)`:
 * writes out [B, Hq, N, D]. */
la_status la_fwd(const void *q, const void *k, const void *v, void *out, int B, int Hq,
                 int Hkv, int N, int D, la_dtype dtype, int is_causal, la_phi phi, float eps,
                 const float *cos_weight, const float *sin_weight, void *workspace,
                 size_t ws_bytes, void *stream);

/* la_fwd on inputs with strides: q_strides, k_strides, v_strides (NULL: contiguous) give
 * each input's element strides; out is contiguous.  The strides are used as given (the
 * caller guarantees every element they reach lies in the input's allocation); negative
 * strides: LA_ERR_ARG.  On the tensor-core path (la_kernel_path) every stride must be a
 * multiple of 8 elements (TMA: 16-byte row strides), else LA_ERR_ALIGN; the CUDA-core
 * path takes any.  The gqa page's wrapper passes strides to its kernel in the same way. */
la_status la_fwd_strided(const void *q, const void *k, const void *v, void *out, int B, int Hq,
                         int Hkv, int N, int D, la_dtype dtype, int is_causal, la_phi phi,
                         float eps, const float *cos_weight, const float *sin_weight,
                         const la_strides *q_strides, const la_strides *k_strides,
                         const la_strides *v_strides, void *workspace, size_t ws_bytes,
                         void *stream);

/* Backward, `linear_attn.bwd(q, k, v, grad_out, is_causal, phi, eps, cos_weight,
 * sin_weight) -> (dq, dk, dv)`: writes dq [B, Hq, N, D] and the group-summed dk, dv
 * [B, Hkv, N, D].  Recomputes what it needs of the forward from q, k, v. */
la_status la_bwd(const void *q, const void *k, const void *v, const void *grad_out, void *dq,
                 void *dk, void *dv, int B, int Hq, int Hkv, int N, int D, la_dtype dtype,
                 int is_causal, la_phi phi, float eps, const float *cos_weight,
                 const float *sin_weight, void *workspace, size_t ws_bytes, void *stream);

/* The same backward (same operation, same results) for a caller that has just run la_fwd
 * on these inputs: fwd_workspace / fwd_ws_bytes are that call's workspace, still holding
 * what la_fwd left there: its scanned per-segment states S, z and, on the tensor-core path,
 * every row's denominator den_i = sum_p a_i^p . z_i^p + eps, a record of the call and, with
 * cos/sin weights, the output rows in float32.  When
 * the forward and the backward cut the sequence the same way (the same kernel family, chunk
 * and segments; true whenever both run on the tensor-core path) the backward reads those
 * instead of recomputing them, which saves the forward's pass over q, k and v (la_bwd on the
 * tensor-core path runs that forward itself, with dq as its output scratch); otherwise it
 * recomputes them and fwd_workspace is not read.  The pages' `bwd` recomputes the forward
 * through autograd; keeping the forward's context is this library's design.
 *
 * The caller guarantees that la_fwd ran with the same q, k, v (same buffers and values),
 * sizes, mode, phi, eps and weights, that its workspace was not written since, and that
 * the forward is ordered before this call (same stream, or an event).  On the tensor-core
 * path the backward checks the forward's record (sizes, mode, phi, eps, segments and the
 * q, k, v addresses): a workspace that another call wrote makes la_get_status() return
 * LA_ERR_WORKSPACE (the gradients of that call are then not valid).  Values changed in the
 * same buffers cannot be detected.  fwd_workspace is read only.  Errors as la_bwd;
 * LA_ERR_ARG if fwd_workspace is NULL. */
la_status la_bwd_from_fwd(const void *q, const void *k, const void *v, const void *grad_out,
                          void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int D,
                          la_dtype dtype, int is_causal, la_phi phi, float eps,
                          const float *cos_weight, const float *sin_weight,
                          const void *fwd_workspace, size_t fwd_ws_bytes, void *workspace,
                          size_t ws_bytes, void *stream);

/* la_bwd (fwd_workspace NULL) or la_bwd_from_fwd (fwd_workspace given, from la_fwd_strided
 * with the same inputs and strides) on inputs with strides: q, k, v, grad_out strides as in
 * la_fwd_strided (NULL: contiguous); dq, dk, dv are contiguous.  Errors as la_fwd_strided
 * and la_bwd. */
la_status la_bwd_strided(const void *q, const void *k, const void *v, const void *grad_out,
                         void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int D,
                         la_dtype dtype, int is_causal, la_phi phi, float eps,
                         const float *cos_weight, const float *sin_weight,
                         const la_strides *q_strides, const la_strides *k_strides,
                         const la_strides *v_strides, const la_strides *g_strides,
                         const void *fwd_workspace, size_t fwd_ws_bytes, void *workspace,
                         size_t ws_bytes, void *stream);

/* la_fwd with a value width Dv in {32, 64, 128} of its own: q, k [.., N, D]; v [B, Hkv, N,
 * Dv]; writes out [B, Hq, N, Dv].  All contiguous.  The state S = sum_j b_j v_j^T is D x Dv;
 * Dv = D is la_fwd.  Workspace: la_workspace_size_v.  Errors as la_fwd. */
la_status la_fwd_v(const void *q, const void *k, const void *v, void *out, int B, int Hq, int Hkv, int N, int D,
                   int Dv, la_dtype dtype, int is_causal, la_phi phi, float eps, const float *cos_weight,
                   const float *sin_weight, void *workspace, size_t ws_bytes, void *stream);

/* la_bwd (fwd_workspace NULL) or la_bwd_from_fwd (fwd_workspace from la_fwd_v with the same
 * arguments) with a value width Dv: grad_out [B, Hq, N, Dv]; writes dq [B, Hq, N, D], dk
 * [B, Hkv, N, D] and dv [B, Hkv, N, Dv].  All contiguous.  Errors as la_bwd. */
la_status la_bwd_v(const void *q, const void *k, const void *v, const void *grad_out, void *dq, void *dk, void *dv,
                   int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dtype, int is_causal, la_phi phi, float eps,
                   const float *cos_weight, const float *sin_weight, const void *fwd_workspace, size_t fwd_ws_bytes,
                   void *workspace, size_t ws_bytes, void *stream);

/* Synchronises `stream`, then returns and clears the device-side error word of the
 * current device: LA_ERR_TIMEOUT if a kernel's bounded wait ran out since the last call,
 * LA_ERR_WORKSPACE if la_bwd_from_fwd was given a forward workspace that another call
 * wrote, LA_ERR_CUDA if the synchronisation failed, else LA_OK. */
la_status la_get_status(void *stream);

/* Static, NUL-terminated description of a status code (host). */
const char *la_status_str(la_status status);

/* Static description of the most recent CUDA error seen by this library on the calling
 * thread ("" if none). */
const char *la_last_cuda_error(void);

/* Kernel timing for reports.  Between la_trace_start() and la_trace_stop() the library
 * brackets each of its kernel launches with a pair of CUDA events recorded on the
 * launch's own stream (the kernels themselves are unchanged).  la_trace_collect()
 * waits for those events, folds them per kernel name, frees them and returns how many
 * distinct kernels ran; la_trace_kernel() then reads entry `index` (0-based): a static
 * name, the number of launches and their summed device time in milliseconds.  Host-side
 * state is process-wide and guarded by a mutex. */
la_status la_trace_start(void);
la_status la_trace_stop(void);
int la_trace_collect(void);
la_status la_trace_kernel(int index, const char **name, int *launches, double *total_ms);

/* Low-rank projection (module neuralops.core.triton_kernels.low_rank, `fwd`):
 *
 *   y = (x V^T) U^T + bias
 *
 * x [M, K_in], V [r, K_in], U [K_out, r], bias [K_out] (NULL: no bias), y [M, K_out]; every
 * tensor row-major and contiguous, bfloat16 (LA_BF16), on the device; the leading
 * dimensions of a caller's x (batch, sequence) are the M rows.  Arithmetic: float32
 * accumulation on the tensor cores; the bottleneck t = x V^T is rounded to bf16 once before
 * the second product (as a bf16 framework computes the two products).  One kernel does both
 * products per 128-row tile, so t never goes to memory.  No workspace.
 * Errors: LA_ERR_ARG for sizes <= 0, a null x, U, V or y or an unknown dtype;
 * LA_ERR_UNSUPPORTED for LA_F32, r > 256, or K_in, K_out or r not a multiple of 8 (rows
 * must start on 16-byte boundaries); LA_ERR_ALIGN for a pointer that is not 16-byte
 * aligned.  Asynchronous on `stream`, like la_fwd. */
la_status la_lowrank_fwd(const void *x, const void *U, const void *V, const void *bias, void *y, int M,
                         int K_in, int r, int K_out, la_dtype dtype, void *stream);

/* Bytes of workspace that la_lowrank_bwd (is_bwd = 1) needs; 0 for the forward or for
 * arguments the calls reject.  Host-only. */
size_t la_lowrank_workspace_size(int M, int K_in, int r, int K_out, la_dtype dtype, int is_bwd);

/* Backward of la_lowrank_fwd (the page's `bwd`: gradients for x, U, V and bias) for the
 * output gradient grad_out [M, K_out]:
 *   t = x V^T,  dt = grad_out U,  dx = dt V,  dU = grad_out^T t,  dV = dt^T x,
 *   dbias = sum over the M rows of grad_out.
 * Writes dx [M, K_in], dU [K_out, r], dV [r, K_in] and, when dbias is not NULL, dbias
 * [K_out] (bf16).  t and dt (bf16, rounded once like the forward's t) and the float32
 * partial sums of the row reductions live in the workspace (la_lowrank_workspace_size, 256-
 * byte aligned); the row reductions are summed in a fixed order, so results are
 * deterministic.  Errors as la_lowrank_fwd, plus LA_ERR_WORKSPACE. */
la_status la_lowrank_bwd(const void *x, const void *U, const void *V, const void *grad_out, void *dx, void *dU,
                         void *dV, void *dbias, int M, int K_in, int r, int K_out, la_dtype dtype,
                         void *workspace, size_t ws_bytes, void *stream);

/* la_lowrank_fwd that also writes the bottleneck t = x V^T (bf16, [M, r], rounded once: the
 * bits la_lowrank_bwd would recompute) to t_out, for la_lowrank_bwd_t.  LA_ERR_ARG if t_out
 * is NULL; otherwise as la_lowrank_fwd. */
la_status la_lowrank_fwd_t(const void *x, const void *U, const void *V, const void *bias, void *y,
                           void *t_out, int M, int K_in, int r, int K_out, la_dtype dtype,
                           void *stream);

/* la_lowrank_bwd given the t that la_lowrank_fwd_t wrote for these x and V (ordered before
 * this call): the same results, without the backward's own pass over x for t.  The caller
 * guarantees t matches x and V.  LA_ERR_ARG if t is NULL; otherwise as la_lowrank_bwd (the
 * workspace size is the same). */
la_status la_lowrank_bwd_t(const void *x, const void *U, const void *V, const void *t,
                           const void *grad_out, void *dx, void *dU, void *dV, void *dbias, int M,
                           int K_in, int r, int K_out, la_dtype dtype, void *workspace,
                           size_t ws_bytes, void *stream);

/* Forward for callers that cannot allocate device memory.
 *
 * Some callers have no way to obtain scratch memory on the GPU: a plugin host that hands
 * a kernel library only its input and output buffers, or a latency-critical loop that may
 * not call cudaMalloc/cudaFree because those can synchronise the whole device.  This entry
 * point computes exactly what la_fwd computes, with the same arguments minus the
 * workspace: its scratch lives in LA_STATIC_WS_BYTES bytes of static device memory inside
 * this library, which every GPU that loads the library holds until the process exits.
 * It calls no allocator (no cudaMalloc, cudaFree or allocating library routine).  The
 * pages have no counterpart of this entry point.
 *
 * - Sizes whose forward needs more scratch than LA_STATIC_WS_BYTES (see
 *   la_workspace_size(..., is_bwd = 0)) are rejected with LA_ERR_STATIC_WS_LIMIT before
 *   any CUDA call.
 * - The first call on each device looks up the device address of the static scratch
 *   (cudaGetSymbolAddress, with that device current); make that first call before any
 *   stream capture.
 * - All calls share the one scratch array, which keeps whatever the last call left in
 *   it; the forward writes every scratch word before reading it, so nothing needs
 *   clearing between calls.  Calls whose work can overlap on the GPU (different streams,
 *   or different host threads) race on the scratch and must be serialised by the caller.
 */
#define LA_STATIC_WS_BYTES (64u * 1024u * 1024u)
#define LA_ERR_STATIC_WS_LIMIT ((la_status)7)

la_status la_fwd_static_ws(const void *q, const void *k, const void *v, void *out, int B,
                           int Hq, int Hkv, int N, int D, la_dtype dtype, int is_causal,
                           la_phi phi, float eps, const float *cos_weight,
                           const float *sin_weight, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_H */
