// la_api.cu -- the C ABI of libla.so: argument checks, the work plan, dispatch to the
// kernel families, and the device error word.
//
// Entry points follow linear_attn.fwd(q, k, v, is_causal, phi, eps, cos_weight,
// sin_weight) and linear_attn.bwd(..., grad_out) -> (dq, dk, dv) (module
// neuralops.core.triton_kernels.linear_attn), with the key/value head count taken from
// the caller as in gqa.fwd(k, v, num_kv_heads, num_heads) (module
// neuralops.core.triton_kernels.gqa; its rule: both counts positive and the query count a
// multiple of the key/value count).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "la_internal.cuh"

namespace la {

// Latched by kernels whose bounded waits run out; read and cleared by la_get_status().
__device__ int g_error_word;

namespace {

thread_local char t_last_cuda[256] = "";

la_status cuda_fail(cudaError_t e) {
    std::snprintf(t_last_cuda, sizeof t_last_cuda, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return LA_ERR_CUDA;
}

// Device address of g_error_word on the current device (looked up once per device).
cudaError_t error_word(int **out) {
    static std::mutex mu;
    static int *cache[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_error_word);
        if (e != cudaSuccess) return e;
        cache[dev] = static_cast<int *>(ptr);
    }
    *out = cache[dev];
    return cudaSuccess;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Host-only argument checks shared by every entry point.
la_status check_shape(int B, int Hq, int Hkv, int N, int D, int Dv, int dtype, int phi, float eps,
                      const float *cw, const float *sw) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || D <= 0 || Dv <= 0) return LA_ERR_ARG;
    if (Hq % Hkv != 0) return LA_ERR_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_ARG;
    if (phi != LA_PHI_ELU1 && phi != LA_PHI_RELU && phi != LA_PHI_IDENTITY) return LA_ERR_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return LA_ERR_ARG;
    if ((cw == nullptr) != (sw == nullptr)) return LA_ERR_ARG;
    // element counts must fit comfortably in 64 bits
    const unsigned long long elems = (unsigned long long)B * (unsigned long long)Hq *
                                     (unsigned long long)N * (unsigned long long)(D > Dv ? D : Dv);
    if (elems >> 60) return LA_ERR_ARG;
    if (D != 32 && D != 64 && D != 128) return LA_ERR_UNSUPPORTED;
    if (Dv != 32 && Dv != 64 && Dv != 128) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

// The work plan, a pure function of the arguments.
Plan make_plan(int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dt, int causal, int has_w, int is_bwd) {
    Plan pl{};
    pl.P = has_w ? 2 : 1;
    // the tensor-core kernels are written for Dv = D; other value widths run on the CUDA cores
    pl.path = Dv == D && tc_supported(Hq, Hkv, N, D, dt, pl.P, causal, is_bwd) ? LA_PATH_TCGEN05 : LA_PATH_SIMT;
    const int bg = B * Hkv;
    int slots;   // CTAs that run at once on kPlanSms SMs
    if (pl.path == LA_PATH_TCGEN05) {
        pl.chunk = tc_chunk(Hq / Hkv, D);
        slots = kPlanSms;                            // one CTA per SM (shared memory bound)
    } else {
        pl.chunk = 16;
        slots = 2 * kPlanSms;                        // about two CTAs per SM
    }
    const int nchunks = (N + pl.chunk - 1) / pl.chunk;
    // segments per (batch, kv head): the count whose schedule ends first, counting waves of
    // `slots` CTAs that each run their segment's chunks in turn plus about two chunks' worth of
    // pipeline fill and drain (the fewest segments on a tie)
    int chunks_per_seg = nchunks;
    long long best = -1;
    const int max_want = nchunks < 4 * slots ? nchunks : 4 * slots;
    for (int want = 1; want <= max_want; ++want) {
        const int cps = (nchunks + want - 1) / want;
        const int nseg = (nchunks + cps - 1) / cps;
        const long long waves = ((long long)bg * nseg + slots - 1) / slots;
        const long long cost = waves * (cps + 2);
        if (best < 0 || cost < best) {
            best = cost;
            chunks_per_seg = cps;
        }
    }
    pl.seg_len = chunks_per_seg * pl.chunk;
    pl.nseg = (N + pl.seg_len - 1) / pl.seg_len;
    pl.scan_in_kernel = pl.path == LA_PATH_TCGEN05 && pl.nseg <= kScanInKernelMaxSeg;
    pl.state_elems = (size_t)pl.P * D * (Dv + 1);
    const size_t state_bytes = align_up((size_t)bg * pl.nseg * pl.state_elems * sizeof(float), 256);
    pl.off_state = 0;
    size_t off = state_bytes;
    const bool tc = pl.path == LA_PATH_TCGEN05;
    const size_t row_bytes = align_up((size_t)B * Hq * N * sizeof(float), 256);
    // tensor-core path: den rows padded to a 16-byte multiple (TMA row stride)
    const size_t den_bytes = tc ? align_up((size_t)B * Hq * tc_den_stride(N) * sizeof(float), 256) : row_bytes;
    if (is_bwd) {
        pl.off_rstate = off;
        off += state_bytes;
        pl.off_den = off;
        off += den_bytes;
        pl.off_gd = off;
        off += row_bytes;
        if (tc && causal) {   // phi(q) / den rows, bf16
            pl.off_phis = off;
            off += align_up((size_t)B * Hq * N * D * 2, 256);
        }
        if (tc && pl.P == 2) {   // cos/sin passes: the forward's partials (when the backward runs
                                 // it) and the cos pass's dq, dk, dv (fp32)
            pl.off_pnum = off;
            off += align_up(blocked_floats(B * Hq, N, D) * sizeof(float), 256);
            pl.off_pden = off;
            off += row_bytes;
            pl.off_pdq = off;
            off += align_up(blocked_floats(B * Hq, N, D) * sizeof(float), 256);
            pl.off_pdk = off;
            off += align_up((size_t)B * Hkv * N * D * sizeof(float), 256);
            pl.off_pdv = off;
            off += align_up((size_t)B * Hkv * N * D * sizeof(float), 256);
        }
    } else if (tc) {   // the forward leaves its per-row dens for the backward
        pl.off_den = off;
        off += den_bytes;
        if (pl.P == 2) {   // cos pass -> sin pass: numerator rows and dens of the cos terms
            pl.off_pnum = off;
            off += align_up(blocked_floats(B * Hq, N, D) * sizeof(float), 256);
            pl.off_pden = off;
            off += row_bytes;
        }
    }
    if (tc) {   // and a record of what it was run on
        pl.off_hdr = off;
        off += 256;
    }
    pl.ws_bytes = off;
    return pl;
}

la_status run(bool bwd, const void *q, const void *k, const void *v, const void *g, void *out,
              void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dt,
              int causal, la_phi phi, float eps, const float *cw, const float *sw, void *ws,
              size_t ws_bytes, void *stream, const void *fwd_ws = nullptr, size_t fwd_ws_bytes = 0,
              const la_strides *const *strides = nullptr) {
    la_status st = check_shape(B, Hq, Hkv, N, D, Dv, dt, phi, eps, cw, sw);
    if (st != LA_OK) return st;
    if (!q || !k || !v) return LA_ERR_ARG;
    if (bwd ? (!g || !dq || !dk || !dv) : !out) return LA_ERR_ARG;
    const void *ptrs[] = {q, k, v, g, out, dq, dk, dv, cw, sw};
    for (const void *ptr : ptrs)
        if (ptr && !aligned(ptr, 16)) return LA_ERR_ALIGN;
    // input strides (q, k, v, grad_out): contiguous unless given
    Strides ist[4] = {contiguous_strides(Hq, N, D), contiguous_strides(Hkv, N, D), contiguous_strides(Hkv, N, Dv),
                     contiguous_strides(Hq, N, Dv)};
    for (int i = 0; strides && i < 4; ++i)
        if (strides[i]) {
            if (strides[i]->b < 0 || strides[i]->h < 0 || strides[i]->n < 0) return LA_ERR_ARG;
            ist[i] = Strides{strides[i]->b, strides[i]->h, strides[i]->n};
        }
    const Plan pl = make_plan(B, Hq, Hkv, N, D, Dv, dt, causal, cw != nullptr, bwd);
    if (pl.ws_bytes > 0) {
        if (!ws || ws_bytes < pl.ws_bytes) return LA_ERR_WORKSPACE;
        if (!aligned(ws, 256)) return LA_ERR_ALIGN;
    }
    if (pl.path == LA_PATH_TCGEN05)   // TMA: every stride a multiple of 16 bytes (8 bf16)
        for (const Strides &x : ist)
            if (x.b % 8 || x.h % 8 || x.n % 8) return LA_ERR_ALIGN;

    Params p{};
    p.q = q; p.k = k; p.v = v; p.g = g;
    p.st_q = ist[0]; p.st_k = ist[1]; p.st_v = ist[2]; p.st_g = ist[3];
    p.out = out; p.dq = dq; p.dk = dk; p.dv = dv;
    p.cw = cw; p.sw = sw;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.D = D; p.Dv = Dv; p.n_rep = Hq / Hkv;
    p.P = pl.P; p.phi = phi; p.causal = causal ? 1 : 0; p.eps = eps;
    p.chunk = pl.chunk; p.seg_len = pl.seg_len; p.nseg = pl.nseg; p.scan_in_kernel = pl.scan_in_kernel;
    char *base = static_cast<char *>(ws);
    const bool tc = pl.path == LA_PATH_TCGEN05;
    p.state = reinterpret_cast<float *>(base + pl.off_state);
    p.rstate = bwd ? reinterpret_cast<float *>(base + pl.off_rstate) : nullptr;
    p.den = (bwd || tc) ? reinterpret_cast<float *>(base + pl.off_den) : nullptr;
    p.den_stride = tc ? tc_den_stride(N) : N;
    p.hdr = tc ? reinterpret_cast<int *>(base + pl.off_hdr) : nullptr;
    p.gd = bwd ? reinterpret_cast<float *>(base + pl.off_gd) : nullptr;
    p.phis = bwd && pl.off_phis ? static_cast<void *>(base + pl.off_phis) : nullptr;
    p.part_num = pl.off_pnum ? reinterpret_cast<float *>(base + pl.off_pnum) : nullptr;
    p.part_den = pl.off_pden ? reinterpret_cast<float *>(base + pl.off_pden) : nullptr;
    p.part_dq = pl.off_pdq ? reinterpret_cast<float *>(base + pl.off_pdq) : nullptr;
    p.part_dk = pl.off_pdk ? reinterpret_cast<float *>(base + pl.off_pdk) : nullptr;
    p.part_dv = pl.off_pdv ? reinterpret_cast<float *>(base + pl.off_pdv) : nullptr;
    if (bwd && fwd_ws) {
        // the forward's workspace holds its scanned segment states (and, on the tensor-core
        // path, its per-row dens and its record); they are the backward's when both plans cut
        // the sequence the same way
        const Plan pf = make_plan(B, Hq, Hkv, N, D, Dv, dt, causal, cw != nullptr, 0);
        if (pf.path == pl.path && pf.chunk == pl.chunk && pf.seg_len == pl.seg_len && pf.nseg == pl.nseg &&
            pf.scan_in_kernel == pl.scan_in_kernel &&
            pf.P == pl.P && pf.state_elems == pl.state_elems && fwd_ws_bytes >= pf.ws_bytes && aligned(fwd_ws, 256)) {
            char *f = const_cast<char *>(static_cast<const char *>(fwd_ws));
            p.state = reinterpret_cast<float *>(f + pf.off_state);
            if (tc) {
                p.den = reinterpret_cast<float *>(f + pf.off_den);
                p.hdr = reinterpret_cast<int *>(f + pf.off_hdr);
                if (pl.P == 2) {   // the forward's float32 output rows (for h) and its partials
                    p.part_num = reinterpret_cast<float *>(f + pf.off_pnum);
                    p.part_den = reinterpret_cast<float *>(f + pf.off_pden);
                }
            }
            p.state_given = 1;
        }
    }
    cudaError_t e = error_word(&p.err);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.path == LA_PATH_TCGEN05)
        e = bwd ? tc_backward(p, s) : tc_forward(p, s);
    else
        e = bwd ? simt_backward(p, dt, s) : simt_forward(p, dt, s);
    return e == cudaSuccess ? LA_OK : cuda_fail(e);
}

}  // namespace

// ---- trace facility --------------------------------------------------------------------

namespace {
struct TraceRecord {
    const char *name;
    cudaEvent_t start, stop;
};
struct TraceTotal {
    const char *name;
    int launches;
    double ms;
};
std::mutex g_trace_mu;
std::atomic<bool> g_trace_on{false};
std::vector<TraceRecord> g_trace_records;
std::vector<TraceTotal> g_trace_totals;
}  // namespace

TraceScope::TraceScope(const char *name, cudaStream_t s) : name_(name), stream_(s) {
    if (!g_trace_on.load(std::memory_order_relaxed)) return;
    if (cudaEventCreate(&start_) != cudaSuccess || cudaEventRecord(start_, s) != cudaSuccess) {
        if (start_) cudaEventDestroy(start_);
        start_ = nullptr;
    }
}

TraceScope::~TraceScope() {
    if (!start_) return;
    cudaEvent_t stop = nullptr;
    if (cudaEventCreate(&stop) != cudaSuccess || cudaEventRecord(stop, stream_) != cudaSuccess) {
        cudaEventDestroy(start_);
        if (stop) cudaEventDestroy(stop);
        return;
    }
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace_records.push_back({name_, start_, stop});
}

}  // namespace la

using namespace la;

extern "C" {

size_t la_workspace_size(int B, int Hq, int Hkv, int N, int D, la_dtype dtype, int is_causal,
                         int has_weights, int is_bwd) {
    return la_workspace_size_v(B, Hq, Hkv, N, D, D, dtype, is_causal, has_weights, is_bwd);
}

la_path la_kernel_path(int B, int Hq, int Hkv, int N, int D, la_dtype dtype, int is_causal,
                       int has_weights, int is_bwd) {
    return la_kernel_path_v(B, Hq, Hkv, N, D, D, dtype, is_causal, has_weights, is_bwd);
}

size_t la_workspace_size_v(int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dtype, int is_causal,
                           int has_weights, int is_bwd) {
    const float *w = has_weights ? reinterpret_cast<const float *>(16) : nullptr;
    if (check_shape(B, Hq, Hkv, N, D, Dv, dtype, LA_PHI_ELU1, 0.f, w, w) != LA_OK) return 0;
    return make_plan(B, Hq, Hkv, N, D, Dv, dtype, is_causal, has_weights, is_bwd).ws_bytes;
}

la_path la_kernel_path_v(int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dtype, int is_causal,
                         int has_weights, int is_bwd) {
    const float *w = has_weights ? reinterpret_cast<const float *>(16) : nullptr;
    if (check_shape(B, Hq, Hkv, N, D, Dv, dtype, LA_PHI_ELU1, 0.f, w, w) != LA_OK) return LA_PATH_SIMT;
    return make_plan(B, Hq, Hkv, N, D, Dv, dtype, is_causal, has_weights, is_bwd).path;
}

la_status la_fwd_v(const void *q, const void *k, const void *v, void *out, int B, int Hq, int Hkv, int N, int D,
                   int Dv, la_dtype dtype, int is_causal, la_phi phi, float eps, const float *cos_weight,
                   const float *sin_weight, void *workspace, size_t ws_bytes, void *stream) {
    return run(false, q, k, v, nullptr, out, nullptr, nullptr, nullptr, B, Hq, Hkv, N, D, Dv, dtype, is_causal, phi,
               eps, cos_weight, sin_weight, workspace, ws_bytes, stream);
}

la_status la_bwd_v(const void *q, const void *k, const void *v, const void *grad_out, void *dq, void *dk, void *dv,
                   int B, int Hq, int Hkv, int N, int D, int Dv, la_dtype dtype, int is_causal, la_phi phi, float eps,
                   const float *cos_weight, const float *sin_weight, const void *fwd_workspace, size_t fwd_ws_bytes,
                   void *workspace, size_t ws_bytes, void *stream) {
    return run(true, q, k, v, grad_out, nullptr, dq, dk, dv, B, Hq, Hkv, N, D, Dv, dtype, is_causal, phi, eps,
               cos_weight, sin_weight, workspace, ws_bytes, stream, fwd_workspace, fwd_ws_bytes);
}

la_status la_fwd(const void *q, const void *k, const void *v, void *out, int B, int Hq, int Hkv,
                 int N, int D, la_dtype dtype, int is_causal, la_phi phi, float eps,
                 const float *cos_weight, const float *sin_weight, void *workspace,
                 size_t ws_bytes, void *stream) {
    return run(false, q, k, v, nullptr, out, nullptr, nullptr, nullptr, B, Hq, Hkv, N, D, D, dtype,
               is_causal, phi, eps, cos_weight, sin_weight, workspace, ws_bytes, stream);
}

la_status la_bwd(const void *q, const void *k, const void *v, const void *grad_out, void *dq,
                 void *dk, void *dv, int B, int Hq, int Hkv, int N, int D, la_dtype dtype,
                 int is_causal, la_phi phi, float eps, const float *cos_weight,
                 const float *sin_weight, void *workspace, size_t ws_bytes, void *stream) {
    return run(true, q, k, v, grad_out, nullptr, dq, dk, dv, B, Hq, Hkv, N, D, D, dtype, is_causal,
               phi, eps, cos_weight, sin_weight, workspace, ws_bytes, stream);
}

la_status la_bwd_from_fwd(const void *q, const void *k, const void *v, const void *grad_out, void *dq, void *dk,
                          void *dv, int B, int Hq, int Hkv, int N, int D, la_dtype dtype, int is_causal, la_phi phi,
                          float eps, const float *cos_weight, const float *sin_weight, const void *fwd_workspace,
                          size_t fwd_ws_bytes, void *workspace, size_t ws_bytes, void *stream) {
    if (!fwd_workspace) return LA_ERR_ARG;
    return run(true, q, k, v, grad_out, nullptr, dq, dk, dv, B, Hq, Hkv, N, D, D, dtype, is_causal, phi, eps,
               cos_weight, sin_weight, workspace, ws_bytes, stream, fwd_workspace, fwd_ws_bytes);
}

la_status la_fwd_strided(const void *q, const void *k, const void *v, void *out, int B, int Hq, int Hkv, int N, int D,
                         la_dtype dtype, int is_causal, la_phi phi, float eps, const float *cos_weight,
                         const float *sin_weight, const la_strides *q_strides, const la_strides *k_strides,
                         const la_strides *v_strides, void *workspace, size_t ws_bytes, void *stream) {
    const la_strides *st[4] = {q_strides, k_strides, v_strides, nullptr};
    return run(false, q, k, v, nullptr, out, nullptr, nullptr, nullptr, B, Hq, Hkv, N, D, D, dtype, is_causal, phi, eps,
               cos_weight, sin_weight, workspace, ws_bytes, stream, nullptr, 0, st);
}
la_status la_bwd_strided(const void *q, const void *k, const void *v, const void *grad_out, void *dq, void *dk, void *dv,
                         int B, int Hq, int Hkv, int N, int D, la_dtype dtype, int is_causal, la_phi phi, float eps,
                         const float *cos_weight, const float *sin_weight, const la_strides *q_strides,
                         const la_strides *k_strides, const la_strides *v_strides, const la_strides *g_strides,
                         const void *fwd_workspace, size_t fwd_ws_bytes, void *workspace, size_t ws_bytes,
                         void *stream) {
    const la_strides *st[4] = {q_strides, k_strides, v_strides, g_strides};
    return run(true, q, k, v, grad_out, nullptr, dq, dk, dv, B, Hq, Hkv, N, D, D, dtype, is_causal, phi, eps, cos_weight,
               sin_weight, workspace, ws_bytes, stream, fwd_workspace, fwd_ws_bytes, st);
}

la_status la_get_status(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    if (word != kErrNone) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e);
        return word == kErrStaleWorkspace ? LA_ERR_WORKSPACE : LA_ERR_TIMEOUT;
    }
    return LA_OK;
}

const char *la_status_str(la_status status) {
    switch (status) {
        case LA_OK: return "ok";
        case LA_ERR_ARG: return "invalid argument";
        case LA_ERR_UNSUPPORTED: return "unsupported head dimension (D and Dv must be 32, 64 or 128)";
        case LA_ERR_ALIGN: return "misaligned pointer (16 bytes; workspace 256 bytes)";
        case LA_ERR_CUDA: return "CUDA error";
        case LA_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
        case LA_ERR_WORKSPACE: return "workspace missing or too small";
        case LA_ERR_STATIC_WS_LIMIT:
            return "problem needs more scratch than the static workspace holds (LA_STATIC_WS_BYTES)";
    }
    return "unknown status";
}

const char *la_last_cuda_error(void) { return t_last_cuda; }

la_status la_trace_start(void) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    for (auto &r : g_trace_records) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_trace_records.clear();
    g_trace_totals.clear();
    g_trace_on.store(true);
    return LA_OK;
}

la_status la_trace_stop(void) {
    g_trace_on.store(false);
    return LA_OK;
}

int la_trace_collect(void) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    for (auto &r : g_trace_records) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) == cudaSuccess &&
            cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
            bool found = false;
            for (auto &t : g_trace_totals)
                if (std::strcmp(t.name, r.name) == 0) {
                    t.launches += 1;
                    t.ms += ms;
                    found = true;
                    break;
                }
            if (!found) g_trace_totals.push_back({r.name, 1, (double)ms});
        }
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_trace_records.clear();
    return (int)g_trace_totals.size();
}

la_status la_trace_kernel(int index, const char **name, int *launches, double *total_ms) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (index < 0 || index >= (int)g_trace_totals.size() || !name || !launches || !total_ms)
        return LA_ERR_ARG;
    *name = g_trace_totals[index].name;
    *launches = g_trace_totals[index].launches;
    *total_ms = g_trace_totals[index].ms;
    return LA_OK;
}

}  // extern "C"

// ---- low-rank projection ------------------------------------------------------------------

namespace {

// Host-only checks of the low-rank projection's arguments.
la_status lowrank_check(int M, int K_in, int r, int K_out, int dtype) {
    if (M <= 0 || K_in <= 0 || r <= 0 || K_out <= 0) return LA_ERR_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_ARG;
    const unsigned long long big = (unsigned long long)M * (unsigned long long)(K_in > K_out ? K_in : K_out);
    if (big >> 60) return LA_ERR_ARG;
    if (dtype != LA_BF16 || r > 256) return LA_ERR_UNSUPPORTED;
    // rows of x, y, U and V must start on 16-byte boundaries (TMA row strides)
    if (K_in % 8 || K_out % 8 || r % 8) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

}  // namespace

namespace {
la_status lowrank_fwd_run(const void *x, const void *U, const void *V, const void *bias, void *y, void *t_out, int M,
                          int K_in, int r, int K_out, la_dtype dtype, void *stream) {
    la_status st = lowrank_check(M, K_in, r, K_out, dtype);
    if (st != LA_OK) return st;
    if (!x || !U || !V || !y) return LA_ERR_ARG;
    const void *ptrs[] = {x, U, V, bias, y, t_out};
    for (const void *ptr : ptrs)
        if (ptr && !aligned(ptr, 16)) return LA_ERR_ALIGN;
    int *err = nullptr;
    cudaError_t e = error_word(&err);
    if (e == cudaSuccess)
        e = lowrank_forward(x, U, V, bias, y, t_out, M, K_in, r, K_out, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LA_OK : cuda_fail(e);
}

la_status lowrank_bwd_run(const void *x, const void *U, const void *V, const void *t, const void *grad_out, void *dx,
                          void *dU, void *dV, void *dbias, int M, int K_in, int r, int K_out, la_dtype dtype,
                          void *workspace, size_t ws_bytes, void *stream) {
    la_status st = lowrank_check(M, K_in, r, K_out, dtype);
    if (st != LA_OK) return st;
    if (!x || !U || !V || !grad_out || !dx || !dU || !dV) return LA_ERR_ARG;
    const void *ptrs[] = {x, U, V, t, grad_out, dx, dU, dV, dbias};
    for (const void *ptr : ptrs)
        if (ptr && !aligned(ptr, 16)) return LA_ERR_ALIGN;
    const size_t need = lowrank_bwd_workspace(M, K_in, r, K_out);
    if (!workspace || ws_bytes < need) return LA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return LA_ERR_ALIGN;
    int *err = nullptr;
    cudaError_t e = error_word(&err);
    if (e == cudaSuccess)
        e = lowrank_backward(x, U, V, t, grad_out, dx, dU, dV, dbias, M, K_in, r, K_out, workspace, err,
                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LA_OK : cuda_fail(e);
}
}  // namespace

extern "C" la_status la_lowrank_fwd(const void *x, const void *U, const void *V, const void *bias, void *y, int M,
                                    int K_in, int r, int K_out, la_dtype dtype, void *stream) {
    return lowrank_fwd_run(x, U, V, bias, y, nullptr, M, K_in, r, K_out, dtype, stream);
}
extern "C" la_status la_lowrank_fwd_t(const void *x, const void *U, const void *V, const void *bias, void *y,
                                      void *t_out, int M, int K_in, int r, int K_out, la_dtype dtype, void *stream) {
    if (!t_out) return LA_ERR_ARG;
    return lowrank_fwd_run(x, U, V, bias, y, t_out, M, K_in, r, K_out, dtype, stream);
}

extern "C" size_t la_lowrank_workspace_size(int M, int K_in, int r, int K_out, la_dtype dtype, int is_bwd) {
    if (lowrank_check(M, K_in, r, K_out, dtype) != LA_OK || !is_bwd) return 0;
    return lowrank_bwd_workspace(M, K_in, r, K_out);
}

extern "C" la_status la_lowrank_bwd(const void *x, const void *U, const void *V, const void *grad_out, void *dx,
                                    void *dU, void *dV, void *dbias, int M, int K_in, int r, int K_out,
                                    la_dtype dtype, void *workspace, size_t ws_bytes, void *stream) {
    return lowrank_bwd_run(x, U, V, nullptr, grad_out, dx, dU, dV, dbias, M, K_in, r, K_out, dtype, workspace,
                           ws_bytes, stream);
}
extern "C" la_status la_lowrank_bwd_t(const void *x, const void *U, const void *V, const void *t, const void *grad_out,
                                      void *dx, void *dU, void *dV, void *dbias, int M, int K_in, int r, int K_out,
                                      la_dtype dtype, void *workspace, size_t ws_bytes, void *stream) {
    if (!t) return LA_ERR_ARG;
    return lowrank_bwd_run(x, U, V, t, grad_out, dx, dU, dV, dbias, M, K_in, r, K_out, dtype, workspace, ws_bytes,
                           stream);
}

// ---- forward without a caller workspace ------------------------------------------------
//
// For callers that cannot allocate device memory (plugin hosts that only pass input and
// output buffers; loops that must not call cudaMalloc/cudaFree, which can synchronise the
// device).  The scratch is this file-scope static device array.  In host code its name is
// only a host-side stand-in, so the device address is looked up with
// cudaGetSymbolAddress, once per device with that device current, and passed on.

static __device__ __align__(256) unsigned char g_static_ws[LA_STATIC_WS_BYTES];

namespace {

cudaError_t static_ws_address(void **out) {
    static std::mutex mu;
    static void *cache[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_ws);
        if (e != cudaSuccess) return e;
        cache[dev] = ptr;
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" la_status la_fwd_static_ws(const void *q, const void *k, const void *v, void *out,
                                      int B, int Hq, int Hkv, int N, int D, la_dtype dtype,
                                      int is_causal, la_phi phi, float eps,
                                      const float *cos_weight, const float *sin_weight,
                                      void *stream) {
    la_status st = check_shape(B, Hq, Hkv, N, D, D, dtype, phi, eps, cos_weight, sin_weight);
    if (st != LA_OK) return st;
    const size_t need =
        make_plan(B, Hq, Hkv, N, D, D, dtype, is_causal, cos_weight != nullptr, 0).ws_bytes;
    if (need > LA_STATIC_WS_BYTES) return LA_ERR_STATIC_WS_LIMIT;
    void *ws = nullptr;
    cudaError_t e = static_ws_address(&ws);
    if (e != cudaSuccess) return cuda_fail(e);
    return run(false, q, k, v, nullptr, out, nullptr, nullptr, nullptr, B, Hq, Hkv, N, D, D, dtype,
               is_causal, phi, eps, cos_weight, sin_weight, ws, LA_STATIC_WS_BYTES, stream);
}
