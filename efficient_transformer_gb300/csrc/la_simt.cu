// la_simt.cu -- general linear-attention kernels on the CUDA cores (float32 FMA).
//
// These kernels carry every mode of the operation (causal and bidirectional, elu+1 and
// relu, with or without cos/sin position weights, grouped key/value heads, float32 or
// bfloat16 inputs, D in {32, 64, 128}) with float32 arithmetic throughout.  They are the
// path for float32 inputs, whose tolerance rules out bfloat16 tensor-core operands, and
// for the shapes the tensor-core path does not take.
//
// Work split (the "chunked causal streaming" and "bidirectional parallel reduction" of the
// linear_attn module docstring): each (batch, kv head) sequence is cut into segments; one
// CTA owns one segment and walks it in chunks of kC tokens, serving all n_rep query heads
// of the group from the same key/value chunk.  Segment states are joined by a scan:
//
//   forward   k_seg_state -> k_scan (exclusive prefix, or total when bidirectional)
//             -> k_fwd
//   backward  k_seg_state -> k_scan -> k_bwd_dq (dq, and per-row den, gd)
//             -> k_seg_rstate -> k_scan (exclusive suffix, or total) -> k_bwd_dkdv
//
// State layout in the workspace: [B*Hkv][nseg][P][D][Dv+1] float32, where column Dv holds
// z (the value vector is augmented with a constant 1, so S and z update together).  The
// value width Dv (v, out, grad_out and dv rows) may differ from the head dimension D (q, k,
// dq and dk rows); the kernels take both as template parameters D and DV.
#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kC = 16;          // tokens per chunk
constexpr int kThreads = 256;   // 16 x 16 threads

// Segment of this CTA.
struct Seg {
    int bg, b, g, s, t0, t1;
};
__device__ __forceinline__ Seg my_segment(const Params &p) {
    Seg r;
    r.bg = blockIdx.x / p.nseg;
    r.s = blockIdx.x % p.nseg;
    r.b = r.bg / p.Hkv;
    r.g = r.bg % p.Hkv;
    r.t0 = r.s * p.seg_len;
    r.t1 = min(p.N, r.t0 + p.seg_len);
    return r;
}

// Head bh = b H + h of an input with element strides st (rows t at t st.n).
template <typename T>
__device__ __forceinline__ const T *head_ptr(const void *base, const Strides &st, int bh, int H) {
    return static_cast<const T *>(base) + (long long)(bh / H) * st.b + (long long)(bh % H) * st.h;
}

// Key/value chunk [c0, c0 + kC) clipped to t1: bsm[term][j][d] = w_j^term phi(k_jd) (row
// pitch D + 1), vsm[j][e] = v_je with vsm[j][DV] = 1 (row pitch DV + 1); rows past t1 are
// all zero (phi(0) is not 0 for elu+1, so padding must be explicit).  kraw (optional) gets k
// itself.
template <typename T, int D, int DV, int P>
__device__ void load_kv(const Params &p, const T *kb, const T *vb, int c0, int t1, float *bsm,
                        float *vsm, float *kraw) {
    constexpr int DP = D + 1, DVP = DV + 1;
    for (int idx = threadIdx.x; idx < kC * D; idx += kThreads) {
        const int j = idx / D, d = idx - j * D, t = c0 + j;
        const bool ok = t < t1;
        const float kv = ok ? to_f32(kb[(long long)t * p.st_k.n + d]) : 0.f;
        const float f = ok ? feature(kv, p.phi) : 0.f;
#pragma unroll
        for (int term = 0; term < P; ++term)
            bsm[(term * kC + j) * DP + d] = ok ? pos_weight(p, term, t) * f : 0.f;
        if (kraw) kraw[j * DP + d] = kv;
    }
    for (int idx = threadIdx.x; idx < kC * DVP; idx += kThreads) {
        const int j = idx / DVP, e = idx - j * DVP, t = c0 + j;
        vsm[idx] = t < t1 ? (e < DV ? to_f32(vb[(long long)t * p.st_v.n + e]) : 1.f) : 0.f;
    }
}

// Query chunk: asm_[term][i][d] = w_i^term phi(q_id) (0 past t1); qraw gets q.
template <typename T, int D, int P>
__device__ void load_q(const Params &p, const T *qb, int c0, int t1, float *asm_, float *qraw) {
    constexpr int DP = D + 1;
    for (int idx = threadIdx.x; idx < kC * D; idx += kThreads) {
        const int i = idx / D, d = idx - i * D, t = c0 + i;
        const bool ok = t < t1;
        const float qv = ok ? to_f32(qb[(long long)t * p.st_q.n + d]) : 0.f;
        const float f = ok ? feature(qv, p.phi) : 0.f;
#pragma unroll
        for (int term = 0; term < P; ++term)
            asm_[(term * kC + i) * DP + d] = ok ? pos_weight(p, term, t) * f : 0.f;
        if (qraw) qraw[i * DP + d] = qv;
    }
}

// gx[i][e] = g_ie / den_i and gx[i][DV] = gd_i from the saved per-row den and gd.
template <typename T, int DV>
__device__ void load_gx(const Params &p, const T *gb, const float *denb, const float *gdb, int c0,
                        int t1, float *gx) {
    constexpr int DVP = DV + 1;
    for (int idx = threadIdx.x; idx < kC * DVP; idx += kThreads) {
        const int i = idx / DVP, e = idx - i * DVP, t = c0 + i;
        float x = 0.f;
        if (t < t1) x = (e < DV) ? to_f32(gb[(long long)t * p.st_g.n + e]) / denb[t] : gdb[t];
        gx[idx] = x;
    }
}

// Masked intra-chunk scores A[i][j] = sum_term a_i^term . b_j^term for j <= i (else 0).
template <int D, int P>
__device__ void intra_scores(const float *asm_, const float *bsm, float *Asm) {
    constexpr int DP = D + 1;
    const int i = threadIdx.x / kC, j = threadIdx.x % kC;
    float acc = 0.f;
    if (j <= i) {
#pragma unroll
        for (int term = 0; term < P; ++term) {
            const float *ar = asm_ + (term * kC + i) * DP, *br = bsm + (term * kC + j) * DP;
#pragma unroll 8
            for (int d = 0; d < D; ++d) acc += ar[d] * br[d];
        }
    }
    Asm[i * kC + j] = acc;
}

// S[term][d][e] += sum_j rows[term][j][d] * cols[j][e] over the whole state (rows: feature
// rows of pitch D + 1; cols: augmented value rows of pitch DV + 1).
template <int D, int DV, int P>
__device__ void state_update(float *S, const float *rows, const float *cols) {
    constexpr int DP = D + 1, DVP = DV + 1;
    for (int idx = threadIdx.x; idx < P * D * DVP; idx += kThreads) {
        const int pd = idx / DVP, e = idx - pd * DVP, term = pd / D, d = pd - term * D;
        const float *rc = rows + term * kC * DP + d;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kC; ++j) acc += rc[j * DP] * cols[j * DVP + e];
        S[idx] += acc;
    }
}

template <int D, int DV, int P>
__device__ void load_state(float *S, const float *src) {
    for (int i = threadIdx.x; i < P * D * (DV + 1); i += kThreads) S[i] = src[i];
}

// Sum over the 16 lanes that share a row (lanes 0-15 or 16-31 of a warp).
__device__ __forceinline__ float row_sum16(float x) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---------------------------------------------------------------------------------------
// Per-segment state S = sum_j b_j [v_j, 1]^T over the segment's tokens.
template <typename T, int D, int DV, int P>
__global__ void __launch_bounds__(kThreads) k_seg_state(Params p) {
    pdl_wait();
    constexpr int DP = D + 1, DVP = DV + 1;
    extern __shared__ float sm[];
    float *S = sm, *bsm = S + P * D * DVP, *vsm = bsm + P * kC * DP;
    const Seg sg = my_segment(p);
    for (int i = threadIdx.x; i < P * D * DVP; i += kThreads) S[i] = 0.f;
    const T *kb = head_ptr<T>(p.k, p.st_k, sg.bg, p.Hkv), *vb = head_ptr<T>(p.v, p.st_v, sg.bg, p.Hkv);
    for (int c0 = sg.t0; c0 < sg.t1; c0 += kC) {
        __syncthreads();
        load_kv<T, D, DV, P>(p, kb, vb, c0, sg.t1, bsm, vsm, nullptr);
        __syncthreads();
        state_update<D, DV, P>(S, bsm, vsm);
    }
    __syncthreads();
    float *dst = p.state + ((size_t)sg.bg * p.nseg + sg.s) * (P * D * DVP);
    for (int i = threadIdx.x; i < P * D * DVP; i += kThreads) dst[i] = S[i];
}

// Scan of segment states along the sequence, per (batch, kv head), in a fixed order.
__global__ void k_scan(float *X, int nseg, size_t elems, int mode) {
    pdl_wait();
    const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= elems) return;
    float *base = X + (size_t)blockIdx.y * nseg * elems + e;
    if (mode == kScanTotal) {
        float acc = 0.f;
#pragma unroll 32
        for (int s = 0; s < nseg; ++s) acc += base[(size_t)s * elems];
        for (int s = 0; s < nseg; ++s) base[(size_t)s * elems] = acc;
        return;
    }
    // batches of 32 segments (one batch for up to 32 segments per sequence): all loads of a
    // batch are issued before its stores
    float acc = 0.f;
    for (int k0 = 0; k0 < nseg; k0 += 32) {
        float t[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int k = k0 + u, s = (mode == kScanPrefix) ? k : nseg - 1 - k;
            t[u] = k < nseg ? base[(size_t)s * elems] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int k = k0 + u, s = (mode == kScanPrefix) ? k : nseg - 1 - k;
            if (k < nseg) base[(size_t)s * elems] = acc;
            acc += t[u];
        }
    }
}

// ---------------------------------------------------------------------------------------
// Forward: out_i = (A V + a S)_i / (rowsum A + a . z + eps)_i per query head.  Thread
// (i, l): query row i of the chunk, output columns l + 16 m.
template <typename T, int D, int DV, int P>
__global__ void __launch_bounds__(kThreads) k_fwd(Params p) {
    pdl_wait();
    constexpr int DP = D + 1, DVP = DV + 1, M = D / 16, MV = DV / 16;
    extern __shared__ float sm[];
    float *S = sm, *asm_ = S + P * D * DVP, *bsm = asm_ + P * kC * DP, *vsm = bsm + P * kC * DP,
          *Asm = vsm + kC * DVP;
    const Seg sg = my_segment(p);
    load_state<D, DV, P>(S, p.state + ((size_t)sg.bg * p.nseg + sg.s) * (P * D * DVP));
    const T *kb = head_ptr<T>(p.k, p.st_k, sg.bg, p.Hkv), *vb = head_ptr<T>(p.v, p.st_v, sg.bg, p.Hkv);
    const int i = threadIdx.x / 16, l = threadIdx.x % 16;
    for (int c0 = sg.t0; c0 < sg.t1; c0 += kC) {
        __syncthreads();
        load_kv<T, D, DV, P>(p, kb, vb, c0, sg.t1, bsm, vsm, nullptr);
        for (int r = 0; r < p.n_rep; ++r) {
            const int bh = sg.b * p.Hq + sg.g * p.n_rep + r;
            __syncthreads();
            load_q<T, D, P>(p, head_ptr<T>(p.q, p.st_q, bh, p.Hq), c0, sg.t1, asm_, nullptr);
            __syncthreads();
            if (p.causal) intra_scores<D, P>(asm_, bsm, Asm);
            __syncthreads();
            float acc[MV];
#pragma unroll
            for (int m = 0; m < MV; ++m) acc[m] = 0.f;
            float dpart = 0.f;
            if (p.causal) {
                for (int j = 0; j < kC; ++j) {
                    const float a = Asm[i * kC + j];
#pragma unroll
                    for (int m = 0; m < MV; ++m) acc[m] += a * vsm[j * DVP + l + 16 * m];
                }
                dpart += Asm[i * kC + l];
            }
#pragma unroll
            for (int term = 0; term < P; ++term) {
                const float *ar = asm_ + (term * kC + i) * DP, *St = S + term * D * DVP;
                for (int d = 0; d < D; ++d) {
                    const float a = ar[d];
#pragma unroll
                    for (int m = 0; m < MV; ++m) acc[m] += a * St[d * DVP + l + 16 * m];
                }
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const int d = l + 16 * m;
                    dpart += ar[d] * St[d * DVP + DV];
                }
            }
            const float den = row_sum16(dpart) + p.eps;
            const int t = c0 + i;
            if (t < sg.t1) {
                T *ob = static_cast<T *>(p.out) + ((size_t)bh * p.N + t) * DV;
#pragma unroll
                for (int m = 0; m < MV; ++m) ob[l + 16 * m] = from_f32<T>(acc[m] / den);
            }
        }
        if (p.causal) {
            __syncthreads();
            state_update<D, DV, P>(S, bsm, vsm);
        }
    }
}

// ---------------------------------------------------------------------------------------
// Backward, pass 1: dq, and the per-row den_i and gd_i = -(g_i . num_i) / den_i^2.
template <typename T, int D, int DV, int P>
__global__ void __launch_bounds__(kThreads) k_bwd_dq(Params p) {
    pdl_wait();
    constexpr int DP = D + 1, DVP = DV + 1, M = D / 16, MV = DV / 16;
    extern __shared__ float sm[];
    float *S = sm, *asm_ = S + P * D * DVP, *bsm = asm_ + P * kC * DP, *vsm = bsm + P * kC * DP,
          *qraw = vsm + kC * DVP, *gx = qraw + kC * DP, *Asm = gx + kC * DVP, *dAsm = Asm + kC * kC;
    const Seg sg = my_segment(p);
    load_state<D, DV, P>(S, p.state + ((size_t)sg.bg * p.nseg + sg.s) * (P * D * DVP));
    const T *kb = head_ptr<T>(p.k, p.st_k, sg.bg, p.Hkv), *vb = head_ptr<T>(p.v, p.st_v, sg.bg, p.Hkv);
    const int i = threadIdx.x / 16, l = threadIdx.x % 16;
    for (int c0 = sg.t0; c0 < sg.t1; c0 += kC) {
        __syncthreads();
        load_kv<T, D, DV, P>(p, kb, vb, c0, sg.t1, bsm, vsm, nullptr);
        for (int r = 0; r < p.n_rep; ++r) {
            const int bh = sg.b * p.Hq + sg.g * p.n_rep + r;
            const T *gb = head_ptr<T>(p.g, p.st_g, bh, p.Hq);
            __syncthreads();
            load_q<T, D, P>(p, head_ptr<T>(p.q, p.st_q, bh, p.Hq), c0, sg.t1, asm_, qraw);
            __syncthreads();
            if (p.causal) intra_scores<D, P>(asm_, bsm, Asm);
            __syncthreads();
            // num, den for row i (lane l holds value columns l + 16 m)
            float acc[MV];
#pragma unroll
            for (int m = 0; m < MV; ++m) acc[m] = 0.f;
            float dpart = 0.f;
            if (p.causal) {
                for (int j = 0; j < kC; ++j) {
                    const float a = Asm[i * kC + j];
#pragma unroll
                    for (int m = 0; m < MV; ++m) acc[m] += a * vsm[j * DVP + l + 16 * m];
                }
                dpart += Asm[i * kC + l];
            }
#pragma unroll
            for (int term = 0; term < P; ++term) {
                const float *ar = asm_ + (term * kC + i) * DP, *St = S + term * D * DVP;
                for (int d = 0; d < D; ++d) {
                    const float a = ar[d];
#pragma unroll
                    for (int m = 0; m < MV; ++m) acc[m] += a * St[d * DVP + l + 16 * m];
                }
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const int d = l + 16 * m;
                    dpart += ar[d] * St[d * DVP + DV];
                }
            }
            const float den = row_sum16(dpart) + p.eps;
            const int t = c0 + i;
            const bool ok = t < sg.t1;
            float gv[MV], gdot = 0.f;
#pragma unroll
            for (int m = 0; m < MV; ++m) {
                gv[m] = ok ? to_f32(gb[(long long)t * p.st_g.n + l + 16 * m]) : 0.f;
                gdot += gv[m] * acc[m];
            }
            gdot = row_sum16(gdot);
            const float gdi = ok ? -gdot / (den * den) : 0.f;
#pragma unroll
            for (int m = 0; m < MV; ++m) gx[i * DVP + l + 16 * m] = gv[m] / den;
            if (l == 0) {
                gx[i * DVP + DV] = gdi;
                if (ok) {
                    p.den[(size_t)bh * p.N + t] = den;
                    p.gd[(size_t)bh * p.N + t] = gdi;
                }
            }
            __syncthreads();
            if (p.causal) {  // dA[i][j] = gn_i . v_j + gd_i for j <= i
                const int ii = threadIdx.x / kC, j = threadIdx.x % kC;
                float x = 0.f;
                if (j <= ii)
                    for (int e = 0; e < DVP; ++e) x += gx[ii * DVP + e] * vsm[j * DVP + e];
                dAsm[ii * kC + j] = x;
            }
            __syncthreads();
            // da^term_i = sum_j dA_ij b_j^term + S^term gn_i + gd_i z^term (lane l: features l + 16 m)
            float wt[P];
#pragma unroll
            for (int term = 0; term < P; ++term) wt[term] = ok ? pos_weight(p, term, t) : 0.f;
            float dqv[M];
#pragma unroll
            for (int m = 0; m < M; ++m) dqv[m] = 0.f;
#pragma unroll
            for (int term = 0; term < P; ++term) {
                float da[M];
#pragma unroll
                for (int m = 0; m < M; ++m) da[m] = 0.f;
                if (p.causal)
                    for (int j = 0; j < kC; ++j) {
                        const float x = dAsm[i * kC + j];
#pragma unroll
                        for (int m = 0; m < M; ++m) da[m] += x * bsm[(term * kC + j) * DP + l + 16 * m];
                    }
                const float *St = S + term * D * DVP;
                for (int e = 0; e < DVP; ++e) {
                    const float x = gx[i * DVP + e];
#pragma unroll
                    for (int m = 0; m < M; ++m) da[m] += St[(l + 16 * m) * DVP + e] * x;
                }
#pragma unroll
                for (int m = 0; m < M; ++m) dqv[m] += wt[term] * da[m];
            }
            if (ok) {
                T *db = static_cast<T *>(p.dq) + ((size_t)bh * p.N + t) * D;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const int d = l + 16 * m;
                    db[d] = from_f32<T>(feature_grad(qraw[i * DP + d], p.phi) * dqv[m]);
                }
            }
        }
        if (p.causal) {
            __syncthreads();
            state_update<D, DV, P>(S, bsm, vsm);
        }
    }
}

// Backward, per-segment R = sum over the group's query heads and the segment's rows of
// a_i [gn_i, gd_i]^T (column DV holds r).
template <typename T, int D, int DV, int P>
__global__ void __launch_bounds__(kThreads) k_seg_rstate(Params p) {
    pdl_wait();
    constexpr int DP = D + 1, DVP = DV + 1;
    extern __shared__ float sm[];
    float *R = sm, *asm_ = R + P * D * DVP, *gx = asm_ + P * kC * DP;
    const Seg sg = my_segment(p);
    for (int i = threadIdx.x; i < P * D * DVP; i += kThreads) R[i] = 0.f;
    for (int c0 = sg.t0; c0 < sg.t1; c0 += kC) {
        for (int r = 0; r < p.n_rep; ++r) {
            const int bh = sg.b * p.Hq + sg.g * p.n_rep + r;
            __syncthreads();
            load_q<T, D, P>(p, head_ptr<T>(p.q, p.st_q, bh, p.Hq), c0, sg.t1, asm_, nullptr);
            load_gx<T, DV>(p, head_ptr<T>(p.g, p.st_g, bh, p.Hq), p.den + (size_t)bh * p.N,
                           p.gd + (size_t)bh * p.N, c0, sg.t1, gx);
            __syncthreads();
            state_update<D, DV, P>(R, asm_, gx);
        }
    }
    __syncthreads();
    float *dst = p.rstate + ((size_t)sg.bg * p.nseg + sg.s) * (P * D * DVP);
    for (int i = threadIdx.x; i < P * D * DVP; i += kThreads) dst[i] = R[i];
}

// Backward, pass 2 (reverse over chunks): dk, dv for the kv head, summed over the group.
// Thread (j, l): key row j of the chunk; features l + 16 m (dk) and value columns l + 16 m (dv).
template <typename T, int D, int DV, int P>
__global__ void __launch_bounds__(kThreads) k_bwd_dkdv(Params p) {
    pdl_wait();
    constexpr int DP = D + 1, DVP = DV + 1, M = D / 16, MV = DV / 16;
    extern __shared__ float sm[];
    float *R = sm, *asm_ = R + P * D * DVP, *bsm = asm_ + P * kC * DP, *vsm = bsm + P * kC * DP,
          *kraw = vsm + kC * DVP, *gx = kraw + kC * DP, *Asm = gx + kC * DVP, *dAsm = Asm + kC * kC;
    const Seg sg = my_segment(p);
    load_state<D, DV, P>(R, p.rstate + ((size_t)sg.bg * p.nseg + sg.s) * (P * D * DVP));
    const T *kb = head_ptr<T>(p.k, p.st_k, sg.bg, p.Hkv), *vb = head_ptr<T>(p.v, p.st_v, sg.bg, p.Hkv);
    const int j = threadIdx.x / 16, l = threadIdx.x % 16;
    const int nchunks = (sg.t1 - sg.t0 + kC - 1) / kC;
    for (int c = nchunks - 1; c >= 0; --c) {
        const int c0 = sg.t0 + c * kC;
        __syncthreads();
        load_kv<T, D, DV, P>(p, kb, vb, c0, sg.t1, bsm, vsm, kraw);
        __syncthreads();
        // Inter-chunk part from the rows after this chunk: db^term_j = R^term [v_j, 1],
        // dv_j = sum_term (R^term)^T b_j^term.
        float db[P][M], dvv[MV];
#pragma unroll
        for (int term = 0; term < P; ++term) {
            const float *Rt = R + term * D * DVP;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int d = l + 16 * m;
                float x = 0.f;
                for (int e = 0; e < DVP; ++e) x += Rt[d * DVP + e] * vsm[j * DVP + e];
                db[term][m] = x;
            }
        }
#pragma unroll
        for (int m = 0; m < MV; ++m) dvv[m] = 0.f;
#pragma unroll
        for (int term = 0; term < P; ++term) {
            const float *Rt = R + term * D * DVP;
            for (int d = 0; d < D; ++d) {
                const float bv = bsm[(term * kC + j) * DP + d];
#pragma unroll
                for (int m = 0; m < MV; ++m) dvv[m] += Rt[d * DVP + l + 16 * m] * bv;
            }
        }
        // Intra-chunk part (causal only; bidirectional rows see every key through R).
        for (int r = 0; p.causal && r < p.n_rep; ++r) {
            const int bh = sg.b * p.Hq + sg.g * p.n_rep + r;
            __syncthreads();
            load_q<T, D, P>(p, head_ptr<T>(p.q, p.st_q, bh, p.Hq), c0, sg.t1, asm_, nullptr);
            load_gx<T, DV>(p, head_ptr<T>(p.g, p.st_g, bh, p.Hq), p.den + (size_t)bh * p.N,
                           p.gd + (size_t)bh * p.N, c0, sg.t1, gx);
            __syncthreads();
            {
                intra_scores<D, P>(asm_, bsm, Asm);
                const int ii = threadIdx.x / kC, jj = threadIdx.x % kC;
                float x = 0.f;
                if (jj <= ii)
                    for (int e = 0; e < DVP; ++e) x += gx[ii * DVP + e] * vsm[jj * DVP + e];
                dAsm[ii * kC + jj] = x;
                __syncthreads();
                // intra: db^term_j += sum_{i >= j} dA_ij a_i^term; dv_j += sum_{i >= j} A_ij gn_i
                for (int i = 0; i < kC; ++i) {
                    const float x1 = dAsm[i * kC + j], x2 = Asm[i * kC + j];
#pragma unroll
                    for (int term = 0; term < P; ++term)
#pragma unroll
                        for (int m = 0; m < M; ++m) db[term][m] += x1 * asm_[(term * kC + i) * DP + l + 16 * m];
#pragma unroll
                    for (int m = 0; m < MV; ++m) dvv[m] += x2 * gx[i * DVP + l + 16 * m];
                }
                // rows of this chunk join the suffix state for earlier chunks
                state_update<D, DV, P>(R, asm_, gx);
            }
        }
        const int t = c0 + j;
        if (t < sg.t1) {
            T *dkb = static_cast<T *>(p.dk) + ((size_t)sg.bg * p.N + t) * D;
            T *dvb = static_cast<T *>(p.dv) + ((size_t)sg.bg * p.N + t) * DV;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int d = l + 16 * m;
                float x = 0.f;
#pragma unroll
                for (int term = 0; term < P; ++term) x += pos_weight(p, term, t) * db[term][m];
                dkb[d] = from_f32<T>(feature_grad(kraw[j * DP + d], p.phi) * x);
            }
#pragma unroll
            for (int m = 0; m < MV; ++m) dvb[l + 16 * m] = from_f32<T>(dvv[m]);
        }
    }
}

// ---------------------------------------------------------------------------------------
template <int D, int DV, int P> constexpr size_t smem_state() { return sizeof(float) * P * D * (DV + 1); }
template <int W> constexpr size_t smem_row() { return sizeof(float) * kC * (W + 1); }   // kC rows of W + 1
constexpr size_t smem_tile() { return sizeof(float) * kC * kC; }

template <typename K>
cudaError_t launch(const char *name, K kernel, size_t smem, int grid, const Params &p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    TraceScope ts(name, s);
    return launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, s, p);
}

// Dynamic shared memory of each kernel: its state, then its feature rows (pitch D + 1), value
// rows (pitch DV + 1) and score tiles, in the order the kernel lays them out.
template <int D, int DV, int P> constexpr size_t smem_seg_state() {
    return smem_state<D, DV, P>() + P * smem_row<D>() + smem_row<DV>();
}
template <int D, int DV, int P> constexpr size_t smem_fwd() {
    return smem_state<D, DV, P>() + 2 * P * smem_row<D>() + smem_row<DV>() + smem_tile();
}
template <int D, int DV, int P> constexpr size_t smem_bwd() {   // k_bwd_dq and k_bwd_dkdv
    return smem_state<D, DV, P>() + (2 * P + 1) * smem_row<D>() + 2 * smem_row<DV>() + 2 * smem_tile();
}
template <int D, int DV, int P> constexpr size_t smem_seg_rstate() {
    return smem_state<D, DV, P>() + P * smem_row<D>() + smem_row<DV>();
}

// Every kernel's shared memory fits one block (227 KB) at the largest state, D = Dv = 128 with
// cos/sin weights; the other (D, Dv, P) need less.
static_assert(smem_bwd<128, 128, 2>() <= 227 * 1024 && smem_fwd<128, 128, 2>() <= 227 * 1024 &&
                  smem_seg_state<128, 128, 2>() <= 227 * 1024 && smem_seg_rstate<128, 128, 2>() <= 227 * 1024,
              "CUDA-core kernels' shared memory");

template <typename T, int D, int DV, int P>
cudaError_t forward_impl(const Params &p, cudaStream_t s) {
    const int grid = p.B * p.Hkv * p.nseg;
    const size_t elems = (size_t)P * D * (DV + 1);
    cudaError_t e = launch("simt_seg_state", k_seg_state<T, D, DV, P>, smem_seg_state<D, DV, P>(), grid, p, s);
    if (e == cudaSuccess) e = scan_segments(p.state, p, p.causal ? kScanPrefix : kScanTotal, elems, s);
    if (e == cudaSuccess) e = launch("simt_fwd", k_fwd<T, D, DV, P>, smem_fwd<D, DV, P>(), grid, p, s);
    return e;
}

template <typename T, int D, int DV, int P>
cudaError_t backward_impl(const Params &p, cudaStream_t s) {
    const int grid = p.B * p.Hkv * p.nseg;
    const size_t elems = (size_t)P * D * (DV + 1);
    cudaError_t e = cudaSuccess;
    if (!p.state_given) {
        e = launch("simt_seg_state", k_seg_state<T, D, DV, P>, smem_seg_state<D, DV, P>(), grid, p, s);
        if (e == cudaSuccess) e = scan_segments(p.state, p, p.causal ? kScanPrefix : kScanTotal, elems, s);
    }
    if (e == cudaSuccess) e = launch("simt_bwd_dq", k_bwd_dq<T, D, DV, P>, smem_bwd<D, DV, P>(), grid, p, s);
    if (e == cudaSuccess)
        e = launch("simt_seg_rstate", k_seg_rstate<T, D, DV, P>, smem_seg_rstate<D, DV, P>(), grid, p, s);
    if (e == cudaSuccess) e = scan_segments(p.rstate, p, p.causal ? kScanSuffix : kScanTotal, elems, s);
    if (e == cudaSuccess) e = launch("simt_bwd_dkdv", k_bwd_dkdv<T, D, DV, P>, smem_bwd<D, DV, P>(), grid, p, s);
    return e;
}

template <typename T, int D, int P>
cudaError_t dispatch_dv(const Params &p, cudaStream_t s, bool bwd) {
    switch (p.Dv) {
        case 32: return bwd ? backward_impl<T, D, 32, P>(p, s) : forward_impl<T, D, 32, P>(p, s);
        case 64: return bwd ? backward_impl<T, D, 64, P>(p, s) : forward_impl<T, D, 64, P>(p, s);
        case 128: return bwd ? backward_impl<T, D, 128, P>(p, s) : forward_impl<T, D, 128, P>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int P>
cudaError_t dispatch_d(const Params &p, cudaStream_t s, bool bwd) {
    switch (p.D) {
        case 32: return dispatch_dv<T, 32, P>(p, s, bwd);
        case 64: return dispatch_dv<T, 64, P>(p, s, bwd);
        case 128: return dispatch_dv<T, 128, P>(p, s, bwd);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t dispatch_p(const Params &p, cudaStream_t s, bool bwd) {
    return p.P == 2 ? dispatch_d<T, 2>(p, s, bwd) : dispatch_d<T, 1>(p, s, bwd);
}

}  // namespace

cudaError_t scan_segments(float *X, const Params &p, int mode, size_t elems, cudaStream_t s) {
    dim3 grid((unsigned)((elems + 255) / 256), (unsigned)(p.B * p.Hkv));
    TraceScope ts("scan", s);
    return launch_pdl(k_scan, grid, dim3(256), 0, s, X, p.nseg, elems, mode);
}

cudaError_t simt_forward(const Params &p, la_dtype dt, cudaStream_t s) {
    return dt == LA_F32 ? dispatch_p<float>(p, s, false) : dispatch_p<__nv_bfloat16>(p, s, false);
}

cudaError_t simt_backward(const Params &p, la_dtype dt, cudaStream_t s) {
    return dt == LA_F32 ? dispatch_p<float>(p, s, true) : dispatch_p<__nv_bfloat16>(p, s, true);
}

}  // namespace la
