// la_internal.cuh -- shared definitions of the linear-attention library (not part of the
// public ABI): launch parameters, the work plan, and small device helpers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "la.h"

namespace la {

// Segments per sequence up to which the tensor-core kernels join segment states themselves
// (summing at most this many states when they load a segment's starting state) instead of
// launching the scan kernel.
constexpr int kScanInKernelMaxSeg = 8;

// Number of SMs the work split is planned for (GB300: 152).  The split only sets how a
// head's sequence is cut into segments; results are correct on any device, and for a
// given set of arguments the split (and so the float summation order) never depends on
// the device.
constexpr int kPlanSms = 152;

// Device error word values (latched by kernels, read by la_get_status).
constexpr int kErrNone = 0;
constexpr int kErrTimeout = 1;
constexpr int kErrStaleWorkspace = 2;   // la_bwd_from_fwd got a workspace another call wrote

// Words of the record that the tensor-core forward leaves in its workspace (what it was run
// on), checked by the backward kernels when they take the forward's states and dens.
constexpr int kHdrWords = 16;
constexpr int kHdrMagic = 0x4c414631;

// Element strides of a [B, H, N, D] tensor along B, H and N (D is contiguous).
struct Strides {
    long long b, h, n;
};
inline Strides contiguous_strides(int H, int N, int D) {
    return Strides{(long long)H * N * D, (long long)N * D, (long long)D};
}

// Everything a kernel needs.  Tensor pointers are typed void: the element type is a
// template parameter of each kernel.
struct Params {
    const void *q, *k, *v, *g;   // inputs ([B,Hq,N,D] for q, g; [B,Hkv,N,D] for k, v)
    Strides st_q, st_k, st_v, st_g;   // their strides (outputs and workspace rows are contiguous)
    void *out, *dq, *dk, *dv;    // outputs
    const float *cw, *sw;        // position weights or null
    int B, Hq, Hkv, N, D, n_rep, P, phi, causal;
    int Dv;                      // value width (v, out, grad_out, dv rows); D on the tensor-core path
    float eps;
    int chunk, seg_len, nseg;    // work split along the sequence
    int scan_in_kernel;          // tensor-core path with few segments: the kernels that read a
                                 // segment's starting state sum the per-segment states themselves
                                 // (in the scan's order) and no scan kernel runs
    float *state;                // per (b, kv head, segment) forward state partials
    int state_given;             // backward: `state` already holds the scanned forward states
    float *rstate;               // per (b, kv head, segment) backward state partials
    float *den;                  // [B, Hq, N] row denominators incl. eps: written by the tensor-core
                                 // forward and read by the tensor-core dq kernel; written and read by
                                 // the CUDA-core backward kernels
    int den_stride;              // floats between the den rows of consecutive heads (N, or N rounded
                                 // up to 32 on the tensor-core path, for 16-byte TMA strides)
    int *hdr;                    // tensor-core forward: its record (kHdrWords); backward: the record
                                 // to check (null: nothing to check)
    float *gd;                   // [B, Hq, N] per-row denominator terms (backward; see each kernel)
    void *phis;                  // [B, Hq, N, D] bf16 phi(q) / den, written by the tensor-core dq
                                 // kernel for the dk/dv kernel (causal tensor-core backward; else null)
    // tensor-core forward with cos/sin weights, run as two passes (cos, then sin)
    int pass;                    // 0: one pass; 1: the cos pass; 2: the sin pass
    const float *wrow;           // this pass's position weights (cw or sw), on phi(q) and phi(k) rows
    float *part_num;             // fp32, chunk-blocked (blocked_index, the forward's chunk): the cos
                                 // pass's numerator rows (unnormalised), then the float32 output rows
    float *part_den;             // [B, Hq, N] fp32: the cos pass's denominators (without eps)
    // ... and its backward: the cos pass's gradients (fp32), added in by the sin pass; the
    // forward's float32 output rows (part_num after the sin pass) give h = -g . out, written
    // to `gd`
    float *part_dq;              // fp32, chunk-blocked (blocked_index, the dq kernel's chunk)
    float *part_dk, *part_dv;    // [B, Hkv, N, D]
    int *err;                    // device error word
};

// How one call is carried out.  Filled by make_plan() from the arguments alone.
struct Plan {
    la_path path;
    int P;            // 1, or 2 with cos/sin weights
    int chunk;        // tokens per chunk
    int seg_len;      // tokens per segment (a multiple of chunk)
    int nseg;         // segments per (batch, kv head)
    int scan_in_kernel;   // see Params
    size_t state_elems;   // floats of one segment state (all terms)
    size_t off_state, off_rstate, off_den, off_gd, off_phis, off_hdr;   // workspace byte offsets
    size_t off_pnum, off_pden;    // tensor-core forward with cos/sin weights: the cos pass's partials
    size_t off_pdq, off_pdk, off_pdv;   // ... and backward
    size_t ws_bytes;
};

// Element (row t of head bh, column e) of a chunk-blocked float32 array over C-token chunks,
// [heads][ceil(N / C)][D][C]: for each column the C rows of a chunk are contiguous, so a warp
// of consecutive rows stores or loads one run (the cos/sin passes' partials, which a thread
// per row writes and reads).  At most heads (N + C - 1) D floats.
__host__ __device__ inline size_t blocked_index(int bh, int t, int e, int N, int D, int C) {
    const int nck = (N + C - 1) / C;
    return (((size_t)bh * nck + t / C) * D + e) * C + (t % C);
}
// Floats of such an array for any chunk length up to 128.
inline size_t blocked_floats(int heads, int N, int D) { return (size_t)heads * (N + 128) * D; }

// Row stride of the per-row den array on the tensor-core path (16-byte aligned rows).
inline int tc_den_stride(int N) { return (N + 31) / 32 * 32; }

// --- device helpers --------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// phi and its derivative (phi = 0: elu(x) + 1, alpha = 1; phi = 1: relu; phi = 2: x).
__device__ __forceinline__ float feature(float x, int phi) {
    if (phi == LA_PHI_ELU1) return x > 0.f ? x + 1.f : expf(x);
    if (phi == LA_PHI_IDENTITY) return x;
    return x > 0.f ? x : 0.f;
}
__device__ __forceinline__ float feature_grad(float x, int phi) {
    if (phi == LA_PHI_ELU1) return x > 0.f ? 1.f : expf(x);
    if (phi == LA_PHI_IDENTITY) return 1.f;
    return x > 0.f ? 1.f : 0.f;
}

// Position weight of term p at token t (1 when there are no weights).
__device__ __forceinline__ float pos_weight(const Params &p, int term, int t) {
    if (!p.cw) return 1.f;
    return term == 0 ? p.cw[t] : p.sw[t];
}

// --- programmatic dependent launch ---------------------------------------------------------
// The hot-path kernels are launched so that the next one in the stream is scheduled as the
// previous one's blocks leave their SMs, instead of after the whole grid has been retired
// (launch_pdl).  Each of them calls pdl_wait() as its first statement, before any global-memory
// access and before it allocates tensor memory: the wait returns once every grid it depends on
// has completed and its writes are visible (at once when the launch had no programmatic
// dependency).  No kernel triggers its dependents early: with the trigger at kernel start, the
// next grid's blocks waited beside the running ones and the long-context step took 0.7 % longer
// instead of 1.2 % less.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// --- trace facility (la_trace_*) ---------------------------------------------------------

// Brackets one kernel launch with CUDA events while tracing is on; a no-op otherwise.
class TraceScope {
  public:
    TraceScope(const char *name, cudaStream_t s);
    ~TraceScope();
    TraceScope(const TraceScope &) = delete;
    TraceScope &operator=(const TraceScope &) = delete;

  private:
    const char *name_;
    cudaStream_t stream_;
    cudaEvent_t start_ = nullptr;
};

// --- launchers (defined in the kernel translation units) --------------------------------

// Scan of per-segment states along the sequence (fixed order, per (batch, kv head)).
enum ScanMode { kScanPrefix = 0, kScanSuffix = 1, kScanTotal = 2 };
cudaError_t scan_segments(float *X, const Params &p, int mode, size_t elems, cudaStream_t s);

cudaError_t simt_forward(const Params &p, la_dtype dt, cudaStream_t s);
cudaError_t simt_backward(const Params &p, la_dtype dt, cudaStream_t s);
cudaError_t tc_forward(const Params &p, cudaStream_t s);
cudaError_t tc_backward(const Params &p, cudaStream_t s);
bool tc_supported(int Hq, int Hkv, int N, int D, la_dtype dt, int P, int causal, int is_bwd);
int tc_chunk(int n_rep, int D);   // tokens per chunk of the tensor-core forward (the plan's chunk)
bool tc_bwd_supported(int n_rep, int D);

// Low-rank projection y = (x V^T) U^T + bias (bf16, tensor cores).
cudaError_t lowrank_forward(const void *x, const void *U, const void *V, const void *bias, void *y, void *t_out, int M,
                            int K_in, int r, int K_out, int *err, cudaStream_t s);
size_t lowrank_bwd_workspace(int M, int K_in, int r, int K_out);
cudaError_t lowrank_backward(const void *x, const void *U, const void *V, const void *t_given, const void *g, void *dx,
                             void *dU, void *dV, void *dbias, int M, int K_in, int r, int K_out, void *ws, int *err,
                             cudaStream_t s);

}  // namespace la
