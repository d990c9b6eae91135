// la_tc_bwd.cu -- tensor-core backward (tcgen05 / TMEM / TMA) for bfloat16 inputs.
//
// The gradient of the linear_attn page's `fwd` (its `bwd` differentiates `fwd`), without
// re-running the forward through autograd.  With gn_i = g_i / den_i and
// gd_i = -(g_i . num_i) / den_i^2, the forward's chunked structure carries over to the
// backward: dA_ij = gn_i . v_j + gd_i (j <= i) plays the role of the scores, and the
// suffix state R = sum_{i after} phi(q_i) gn_i^T, r = sum gd_i phi(q_i) carries the rows
// that come later.  Launch order:
//
//   k_tc_state -> scan (prefix S)
//   k_tc_bwd_dq   forward over chunks: dq, per-row den and gd, and each segment's
//                 R (tensor cores) and r (fp32)
//   scan (suffix R)
//   k_tc_bwd_dkdv reverse over chunks: dk, dv (summed over the n_rep heads of the group)
//
// Per chunk of k_tc_bwd_dq (128 stacked query rows, C keys):
//   A = phi(Q) phi(K)^T -> P;  O = P V + phi(Q) S_bf -> num; den = rowsum P + phi(q).z + eps
//   gn = g / den (bf16, written over the grad_out tile), gd = -(g . num) / den^2
//   dA = gn V^T -> dP = mask(dA + gd);  da = dP phi(K) + gn S_bf^T
//   dq = phi'(q) * (da + gd z);  R += phi(Q)^T gn;  S += phi(K)^T V
// Per chunk of k_tc_bwd_dkdv, computed transposed so the 128 query rows stay on the MMA's
// K dimension (and the sum over the group's heads comes for free):
//   dk^T = phi(Q)^T dP + R_bf V^T (+ r),  dv^T = gn^T P + R_bf^T phi(K)^T,  R += phi(Q)^T gn
// Warp roles as in the forward: warp 0 TMA, warp 1 MMA, warps 4-7 prologue, warps 8-11
// row work and epilogues, warps 12-15 state conversion.
#include "la_tc_common.cuh"

namespace la {
namespace {

template <int D, int G>
struct BwdCfg {
    static constexpr int C = 128 / G;
    static constexpr int DB = D / 64;
    static constexpr int Q_BYTES = 128 * D * 2;
    static constexpr int K_BYTES = C * D * 2;
    static constexpr int V_BYTES = C * D * 2;
    static constexpr int G_BYTES = 128 * D * 2;
    static constexpr int STAGE = Q_BYTES + K_BYTES + V_BYTES + G_BYTES;   // [phi(Q) | phi(K) | V | g]
    static constexpr int NS = 2;
    static constexpr int P_BYTES = ((C + 63) / 64) * 128 * 128;
    static constexpr int S_BYTES = DB * D * 128;            // S_bf: D rows (d) x D columns (e)
    static constexpr int R_BYTES = 2 * 128 * 128;           // R_bf: 128 rows x 128 columns (padded)
    static constexpr int DQ_SMEM = NS * STAGE + P_BYTES + S_BYTES + 2 * D * 4 + 128 * 4 + 1024;
    static constexpr int DKDV_SMEM = NS * STAGE + 2 * P_BYTES + R_BYTES + NS * 128 * 4 + 1024;
    static constexpr bool FITS = DQ_SMEM <= kSmemLimit - 1024 && DKDV_SMEM <= kSmemLimit - 1024;
};

__device__ __forceinline__ float feat_grad_from_feat(float f, int phi) {
    // elu+1: phi = x + 1 > 1 for x > 0 (derivative 1), phi = exp(x) <= 1 otherwise
    // (derivative exp(x) = phi); relu: derivative 1 where phi > 0.
    return phi == LA_PHI_ELU1 ? (f > 1.f ? 1.f : f) : (f > 0.f ? 1.f : 0.f);
}

// ---------------------------------------------------------------------------------------
template <int D, int G, bool CAUSAL>
__global__ void __launch_bounds__(512, 1) k_tc_bwd_dq(const __grid_constant__ CUtensorMap map_q,
                                                      const __grid_constant__ CUtensorMap map_k,
                                                      const __grid_constant__ CUtensorMap map_v,
                                                      const __grid_constant__ CUtensorMap map_g, Params p) {
    using K = BwdCfg<D, G>;
    constexpr int C = K::C, NS = K::NS;
    constexpr int OFF_K = K::Q_BYTES, OFF_V = OFF_K + K::K_BYTES, OFF_G = OFF_V + K::V_BYTES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full[NS], bar_ready[NS], bar_empty[NS];
    __shared__ uint64_t bar_afull, bar_pready, bar_ofull, bar_gnready, bar_dafull, bar_dpready, bar_dqfull,
        bar_dofree, bar_sfull, bar_sbf, bar_fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::DQ_SMEM;
    (void)sm_lo;
    (void)sm_hi;
    uint8_t *pbuf = stage0 + NS * K::STAGE;
    uint8_t *sbf = pbuf + K::P_BYTES;
    float *zf = reinterpret_cast<float *>(sbf + K::S_BYTES);   // [2][D]
    float *gds = zf + 2 * D;                                    // [128]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;
    const int bh0 = b * p.Hq + g * G;
    const size_t seg_state = ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1));
    const float *state = p.state + seg_state;
    float *rstate = p.rstate + seg_state;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_ready[s], 128);
            mbar_init(&bar_empty[s], 1 + 128);
        }
        mbar_init(&bar_afull, 1);
        mbar_init(&bar_pready, 128);
        mbar_init(&bar_ofull, 1);
        mbar_init(&bar_gnready, 128);
        mbar_init(&bar_dafull, 1);
        mbar_init(&bar_dpready, 128);
        mbar_init(&bar_dqfull, 1);
        mbar_init(&bar_dofree, 128);
        mbar_init(&bar_sfull, 1);
        mbar_init(&bar_sbf, 128);
        mbar_init(&bar_fin, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base, tO = tmem_base + 128, tA = tmem_base + 256, tR = tmem_base + 384;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            constexpr uint32_t bytes = CAUSAL ? K::STAGE : K::Q_BYTES + K::G_BYTES;
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (k >= NS && !mbar_wait(&bar_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C;
                if (!LA_CHECK(in_smem(st, K::STAGE, sm_lo, sm_hi) && c0 < p.N, 301, smem_u32(st) - sm_lo, c0)) break;
                mbar_arrive_expect_tx(&bar_full[s], bytes);
                for (int r = 0; r < G; ++r)
                    for (int blk = 0; blk < K::DB; ++blk) {
                        tma_load_3d(st + blk * 128 * 128 + r * C * 128, &map_q, &bar_full[s], blk * 64, c0, bh0 + r);
                        tma_load_3d(st + OFF_G + blk * 128 * 128 + r * C * 128, &map_g, &bar_full[s], blk * 64, c0,
                                    bh0 + r);
                    }
                if (CAUSAL)
                    for (int blk = 0; blk < K::DB; ++blk) {
                        tma_load_3d(st + OFF_K + blk * C * 128, &map_k, &bar_full[s], blk * 64, c0, bg);
                        tma_load_3d(st + OFF_V + blk * C * 128, &map_v, &bar_full[s], blk * 64, c0, bg);
                    }
                issued = k + 1;
            }
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k) mbar_drain(&bar_full[k % NS], (k / NS) & 1);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idA = idesc_bf16(128, C, false, false);
            constexpr uint32_t idO = idesc_bf16(128, D, false, true);
            constexpr uint32_t idOK = idesc_bf16(128, D, false, false);
            constexpr uint32_t idR = idesc_bf16(128, D, true, true);
            const uint32_t sbf_u = smem_u32(sbf), pb = smem_u32(pbuf);
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (!mbar_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), ks_ = qs + OFF_K, vs = qs + OFF_V, gs = qs + OFF_G;
                if (!LA_CHECK(qs >= sm_lo && qs + K::STAGE <= sm_hi && pb + K::P_BYTES <= sm_hi &&
                                  sbf_u + K::S_BYTES <= sm_hi,
                              311, qs - sm_lo, k))
                    break;
                if (CAUSAL) {
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16(tA, desc_kmajor(qs, 128, 0, kk), desc_kmajor(ks_, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                    mma_commit(&bar_afull);
                    if (!mbar_wait(&bar_pready, k & 1, &abort_flag)) break;
                }
                if ((CAUSAL || k == 0) && !mbar_wait(&bar_sbf, k & 1, &abort_flag)) break;
                if (k > 0 && !mbar_wait(&bar_dofree, (k - 1) & 1, &abort_flag)) break;
                tc_fence_after();
                uint32_t acc = 0;
                if (CAUSAL)
                    for (int kk = 0; kk < C / 16; ++kk, acc = 1)
                        mma_bf16(tO, desc_kmajor(pb, 128, 0, kk), desc_mnmajor(vs, C, 0, kk), idO, acc);
                for (int kk = 0; kk < D / 16; ++kk, acc = 1)
                    mma_bf16(tO, desc_kmajor(qs, 128, 0, kk), desc_mnmajor(sbf_u, D, 0, kk), idO, acc);
                mma_commit(&bar_ofull);
                if (!mbar_wait(&bar_gnready, k & 1, &abort_flag)) break;
                tc_fence_after();
                if (CAUSAL) {
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16(tA, desc_kmajor(gs, 128, 0, kk), desc_kmajor(vs, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                    mma_commit(&bar_dafull);
                    if (!mbar_wait(&bar_dpready, k & 1, &abort_flag)) break;
                    tc_fence_after();
                }
                acc = 0;
                if (CAUSAL)
                    for (int kk = 0; kk < C / 16; ++kk, acc = 1)
                        mma_bf16(tO, desc_kmajor(pb, 128, 0, kk), desc_mnmajor(ks_, C, 0, kk), idO, acc);
                for (int kk = 0; kk < D / 16; ++kk, acc = 1)
                    mma_bf16(tO, desc_kmajor(gs, 128, 0, kk), desc_kmajor(sbf_u, D, 0, kk), idOK, acc);
                mma_commit(&bar_dqfull);
                for (int kk = 0; kk < 128 / 16; ++kk)
                    mma_bf16(tR, desc_mnmajor(qs, 128, 0, kk), desc_mnmajor(gs, 128, 0, kk), idR,
                             (k > 0 || kk > 0) ? 1u : 0u);
                if (CAUSAL) {
                    for (int kk = 0; kk < C / 16; ++kk)
                        mma_bf16(tS, desc_mnmajor(ks_, C, 0, kk), desc_mnmajor(vs, C, 0, kk), idR, 1u);
                    mma_commit(&bar_sfull);
                }
                mma_commit(&bar_empty[s]);
            }
            mma_commit(&bar_fin);
            mbar_drain(&bar_fin, 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- phi prologue (in place on phi(Q) and phi(K) tiles)
        const int i = threadIdx.x - 128;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            ok = ok && warp_wait(&bar_full[s], (k / NS) & 1, &abort_flag);
            if (ok) {
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C;
                const bool qvalid = c0 + (i % C) < t1;
#pragma unroll 4
                for (int c = 0; c < D / 8; ++c) {
                    uint8_t *ch = st + swz_chunk(128, i, c);
                    if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 321, smem_u32(ch) - sm_lo, c))
                        feat8_inplace2(ch, qvalid, p.phi);
                }
                if (CAUSAL)
                    for (int idx = i; idx < C * (D / 8); idx += 128) {
                        const int j = idx / (D / 8), c = idx % (D / 8);
                        uint8_t *ch = st + OFF_K + swz_chunk(C, j, c);
                        if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 322, smem_u32(ch) - sm_lo, idx))
                            feat8_inplace2(ch, c0 + j < t1, p.phi);
                    }
                fence_proxy_async();
            }
            mbar_arrive(&bar_ready[s]);
        }
    } else if (warp >= 8 && warp < 12) {
        // ---------------- row work (thread = query row i) and column sums (thread = d)
        const int i = threadIdx.x - 256;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int r = i / C, ti = i % C;
        const int bh = bh0 + r;
        if (i < D) zf[i] = state[(size_t)i * (D + 1) + D];
        float r_acc = 0.f;
        named_barrier(1, 128);
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            const int c0 = t0 + k * C, t = c0 + ti;
            const bool valid = t < t1;
            uint8_t *st = stage0 + s * K::STAGE;
            const float *z = zf + (CAUSAL ? (k & 1) * D : 0);
            float den_intra = 0.f;
            if (CAUSAL) {
                ok = ok && warp_wait(&bar_afull, k & 1, &abort_flag);
                tc_fence_after();
                if (ok) {
#pragma unroll 1
                    for (int c16 = 0; c16 < C / 16; ++c16) {
                        float v[16];
                        tmem_ld16(tA + lane_off + c16 * 16, v);
                        tmem_ld_wait();
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const int j = c16 * 16 + e;
                            w[e / 2] = pack_bf16x2((j <= ti) ? v[e] : 0.f, (j + 1 <= ti) ? v[e + 1] : 0.f);
                            const float2 f = unpack_bf16x2(w[e / 2]);
                            den_intra += f.x + f.y;
                        }
                        uint8_t *p0 = pbuf + swz_chunk(128, i, 2 * c16), *p1 = pbuf + swz_chunk(128, i, 2 * c16 + 1);
                        if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi), 331,
                                     smem_u32(p0) - sm_lo, c16)) {
                            *reinterpret_cast<uint4 *>(p0) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4 *>(p1) = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                    fence_proxy_async();
                }
                tc_fence_before();
                mbar_arrive(&bar_pready);
            }
            // num, den -> gn (over the grad_out tile), gd
            ok = ok && warp_wait(&bar_ofull, k & 1, &abort_flag);
            tc_fence_after();
            float gd = 0.f;
            if (ok) {
                float dint = 0.f;
#pragma unroll 4
                for (int c = 0; c < D / 8; ++c) {
                    const uint8_t *ch = st + swz_chunk(128, i, c);
                    if (!LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 332, smem_u32(ch) - sm_lo, c)) continue;
                    const uint4 x = *reinterpret_cast<const uint4 *>(ch);
                    const uint32_t *xi = reinterpret_cast<const uint32_t *>(&x);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 f = unpack_bf16x2(xi[h]);
                        dint += f.x * z[c * 8 + 2 * h] + f.y * z[c * 8 + 2 * h + 1];
                    }
                }
                const float den = den_intra + dint + p.eps;
                const float inv = 1.f / den;
                float gdot = 0.f;
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    float v[16];
                    tmem_ld16(tO + lane_off + c16 * 16, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint8_t *ch = st + OFF_G + swz_chunk(128, i, 2 * c16 + h);
                        if (!LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 333, smem_u32(ch) - sm_lo, c16)) continue;
                        uint4 x = *reinterpret_cast<uint4 *>(ch);
                        uint32_t *xi = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 gv = unpack_bf16x2(xi[q]);
                            gdot += gv.x * v[h * 8 + 2 * q] + gv.y * v[h * 8 + 2 * q + 1];
                            xi[q] = valid ? pack_bf16x2(gv.x * inv, gv.y * inv) : 0u;
                        }
                        *reinterpret_cast<uint4 *>(ch) = x;
                    }
                }
                gd = valid ? -gdot * inv * inv : 0.f;
                gds[i] = gd;
                if (valid && LA_CHECK((size_t)bh * p.N + t < (size_t)p.B * p.Hq * p.N, 334, bh, t)) {
                    p.den[(size_t)bh * p.N + t] = den;
                    p.gd[(size_t)bh * p.N + t] = gd;
                }
                fence_proxy_async();
            }
            tc_fence_before();
            mbar_arrive(&bar_gnready);
            if (CAUSAL) {   // dP = mask(dA + gd), into the P buffer (P was consumed by the O product)
                ok = ok && warp_wait(&bar_dafull, k & 1, &abort_flag);
                tc_fence_after();
                if (ok) {
#pragma unroll 1
                    for (int c16 = 0; c16 < C / 16; ++c16) {
                        float v[16];
                        tmem_ld16(tA + lane_off + c16 * 16, v);
                        tmem_ld_wait();
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const int j = c16 * 16 + e;
                            w[e / 2] = pack_bf16x2((j <= ti) ? v[e] + gd : 0.f, (j + 1 <= ti) ? v[e + 1] + gd : 0.f);
                        }
                        uint8_t *p0 = pbuf + swz_chunk(128, i, 2 * c16), *p1 = pbuf + swz_chunk(128, i, 2 * c16 + 1);
                        if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi), 335,
                                     smem_u32(p0) - sm_lo, c16)) {
                            *reinterpret_cast<uint4 *>(p0) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4 *>(p1) = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                    fence_proxy_async();
                }
                tc_fence_before();
                mbar_arrive(&bar_dpready);
            }
            // dq = phi'(q) * (da + gd z)
            ok = ok && warp_wait(&bar_dqfull, k & 1, &abort_flag);
            tc_fence_after();
            if (ok) {
                __nv_bfloat16 *qrow = static_cast<__nv_bfloat16 *>(p.dq) + ((size_t)bh * p.N + t) * D;
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    float v[16];
                    tmem_ld16(tO + lane_off + c16 * 16, v);
                    tmem_ld_wait();
                    if (valid && LA_CHECK(((size_t)bh * p.N + t) * D + c16 * 16 + 16 <= (size_t)p.B * p.Hq * p.N * D,
                                          336, bh, t)) {
                        uint32_t w[8];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 x = *reinterpret_cast<const uint4 *>(st + swz_chunk(128, i, 2 * c16 + h));
                            const uint32_t *xi = reinterpret_cast<const uint32_t *>(&x);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float2 f = unpack_bf16x2(xi[q]);
                                const int d0 = c16 * 16 + h * 8 + 2 * q;
                                w[h * 4 + q] =
                                    pack_bf16x2(feat_grad_from_feat(f.x, p.phi) * (v[h * 8 + 2 * q] + gd * z[d0]),
                                                feat_grad_from_feat(f.y, p.phi) * (v[h * 8 + 2 * q + 1] + gd * z[d0 + 1]));
                            }
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(qrow + c16 * 16);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_dofree);
            named_barrier(1, 128);
            if (ok && i < D) {
                // r += sum_i gd_i phi(q_i)[d] over this chunk's rows (thread d = i)
                for (int row = 0; row < 128; ++row) {
                    const uint8_t *e_ = st + swz_offset(128, row, i);
                    r_acc += gds[row] * __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(e_));
                }
                if (CAUSAL) {   // z for the next chunk
                    float zs = zf[(k & 1) * D + i];
                    for (int j = 0; j < C; ++j)
                        zs += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(st + OFF_K + swz_offset(C, j, i)));
                    zf[((k + 1) & 1) * D + i] = zs;
                }
            }
            mbar_arrive(&bar_empty[s]);
            named_barrier(1, 128);
        }
        if (ok && i < D) rstate[(size_t)i * (D + 1) + D] = r_acc;
    } else if (warp >= 12) {
        // ---------------- state conversion; at the end the segment's R to the workspace
        const int d = threadIdx.x - 384;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        if (wq * 32 < D) {
            const float *row = state + (size_t)d * (D + 1);
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = row[c16 * 16 + e];
                if (CAUSAL) tmem_st16(tS + lane_off + c16 * 16, v);
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                *reinterpret_cast<uint4 *>(sbf + swz_chunk(D, d, 2 * c16)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(sbf + swz_chunk(D, d, 2 * c16 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
            if (CAUSAL) tmem_st_wait();
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_sbf);
        bool ok = true;
        if (CAUSAL) {
            for (int k = 0; k < nchunk; ++k) {
                ok = ok && warp_wait(&bar_sfull, k & 1, &abort_flag);
                tc_fence_after();
                if (ok && wq * 32 < D) {
#pragma unroll 1
                    for (int c16 = 0; c16 < D / 16; ++c16) {
                        float v[16];
                        tmem_ld16(tS + lane_off + c16 * 16, v);
                        tmem_ld_wait();
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                        *reinterpret_cast<uint4 *>(sbf + swz_chunk(D, d, 2 * c16)) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4 *>(sbf + swz_chunk(D, d, 2 * c16 + 1)) =
                            make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(&bar_sbf);
            }
        }
        ok = ok && warp_wait(&bar_fin, 0, &abort_flag);
        tc_fence_after();
        if (ok && wq * 32 < D) {
            float *row = rstate + (size_t)d * (D + 1);
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                float v[16];
                tmem_ld16(tR + lane_off + c16 * 16, v);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) row[c16 * 16 + e] = v[e];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (threadIdx.x == 0 && abort_flag) atomicExch(p.err, kErrTimeout);
}

// ---------------------------------------------------------------------------------------
template <int D, int G, bool CAUSAL>
__global__ void __launch_bounds__(512, 1) k_tc_bwd_dkdv(const __grid_constant__ CUtensorMap map_q,
                                                        const __grid_constant__ CUtensorMap map_k,
                                                        const __grid_constant__ CUtensorMap map_v,
                                                        const __grid_constant__ CUtensorMap map_g, Params p) {
    using K = BwdCfg<D, G>;
    constexpr int C = K::C, NS = K::NS;
    constexpr int OFF_K = K::Q_BYTES, OFF_V = OFF_K + K::K_BYTES, OFF_G = OFF_V + K::V_BYTES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full[NS], bar_ready[NS], bar_empty[NS];
    __shared__ uint64_t bar_afull, bar_pready, bar_outfull, bar_outfree, bar_rfull, bar_rbf, bar_fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::DKDV_SMEM;
    (void)sm_lo;
    (void)sm_hi;
    uint8_t *pbuf = stage0 + NS * K::STAGE;
    uint8_t *dpbuf = pbuf + K::P_BYTES;
    uint8_t *rbf = dpbuf + K::P_BYTES;
    float *gds = reinterpret_cast<float *>(rbf + K::R_BYTES);   // [NS][128]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;
    const int bh0 = b * p.Hq + g * G;
    const float *rstate = p.rstate + ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1));

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_ready[s], 128);
            mbar_init(&bar_empty[s], 1 + 128);
        }
        mbar_init(&bar_afull, 1);
        mbar_init(&bar_pready, 128);
        mbar_init(&bar_outfull, 1);
        mbar_init(&bar_outfree, 128);
        mbar_init(&bar_rfull, 1);
        mbar_init(&bar_rbf, 128);
        mbar_init(&bar_fin, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // tR: R (d rows x e); tA: A, then dk^T; tD: dA, then dv^T
    const uint32_t tR = tmem_base, tA = tmem_base + 128, tD = tmem_base + 256;

    if (warp == 0) {
        // ---------------- TMA producer (chunks in reverse order)
        if (lane == 0) {
            constexpr uint32_t bytes = CAUSAL ? K::STAGE : K::K_BYTES + K::V_BYTES;
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (k >= NS && !mbar_wait(&bar_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + (nchunk - 1 - k) * C;
                if (!LA_CHECK(in_smem(st, K::STAGE, sm_lo, sm_hi) && c0 < p.N, 401, smem_u32(st) - sm_lo, c0)) break;
                mbar_arrive_expect_tx(&bar_full[s], bytes);
                if (CAUSAL)
                    for (int r = 0; r < G; ++r)
                        for (int blk = 0; blk < K::DB; ++blk) {
                            tma_load_3d(st + blk * 128 * 128 + r * C * 128, &map_q, &bar_full[s], blk * 64, c0,
                                        bh0 + r);
                            tma_load_3d(st + OFF_G + blk * 128 * 128 + r * C * 128, &map_g, &bar_full[s], blk * 64,
                                        c0, bh0 + r);
                        }
                for (int blk = 0; blk < K::DB; ++blk) {
                    tma_load_3d(st + OFF_K + blk * C * 128, &map_k, &bar_full[s], blk * 64, c0, bg);
                    tma_load_3d(st + OFF_V + blk * C * 128, &map_v, &bar_full[s], blk * 64, c0, bg);
                }
                issued = k + 1;
            }
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k) mbar_drain(&bar_full[k % NS], (k / NS) & 1);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idA = idesc_bf16(128, C, false, false);
            constexpr uint32_t idMM = idesc_bf16(128, C, true, true);
            constexpr uint32_t idMK = idesc_bf16(128, C, true, false);
            constexpr uint32_t idR = idesc_bf16(128, D, true, true);
            const uint32_t pb = smem_u32(pbuf), dpb = smem_u32(dpbuf), rb = smem_u32(rbf);
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (!mbar_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) break;
                if (k > 0 && !mbar_wait(&bar_outfree, (k - 1) & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), ks_ = qs + OFF_K, vs = qs + OFF_V, gs = qs + OFF_G;
                if (!LA_CHECK(qs >= sm_lo && qs + K::STAGE <= sm_hi && rb + K::R_BYTES <= sm_hi, 411, qs - sm_lo, k))
                    break;
                if (CAUSAL) {
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16(tA, desc_kmajor(qs, 128, 0, kk), desc_kmajor(ks_, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16(tD, desc_kmajor(gs, 128, 0, kk), desc_kmajor(vs, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                    mma_commit(&bar_afull);
                    if (!mbar_wait(&bar_pready, k & 1, &abort_flag)) break;
                }
                if ((CAUSAL || k == 0) && !mbar_wait(&bar_rbf, k & 1, &abort_flag)) break;
                tc_fence_after();
                // dk^T = phi(Q)^T dP + R_bf V^T
                uint32_t acc = 0;
                if (CAUSAL)
                    for (int kk = 0; kk < 128 / 16; ++kk, acc = 1)
                        mma_bf16(tA, desc_mnmajor(qs, 128, 0, kk), desc_mnmajor(dpb, 128, 0, kk), idMM, acc);
                for (int kk = 0; kk < D / 16; ++kk, acc = 1)
                    mma_bf16(tA, desc_kmajor(rb, 128, 0, kk), desc_kmajor(vs, C, 0, kk), idA, acc);
                // dv^T = gn^T P + R_bf^T phi(K)^T
                acc = 0;
                if (CAUSAL)
                    for (int kk = 0; kk < 128 / 16; ++kk, acc = 1)
                        mma_bf16(tD, desc_mnmajor(gs, 128, 0, kk), desc_mnmajor(pb, 128, 0, kk), idMM, acc);
                for (int kk = 0; kk < D / 16; ++kk, acc = 1)
                    mma_bf16(tD, desc_mnmajor(rb, 128, 0, kk), desc_kmajor(ks_, C, 0, kk), idMK, acc);
                mma_commit(&bar_outfull);
                if (CAUSAL) {   // this chunk's rows join R for the earlier chunks
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        mma_bf16(tR, desc_mnmajor(qs, 128, 0, kk), desc_mnmajor(gs, 128, 0, kk), idR, 1u);
                    mma_commit(&bar_rfull);
                }
                mma_commit(&bar_empty[s]);
            }
            mma_commit(&bar_fin);
            mbar_drain(&bar_fin, 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- prologue: phi(Q), phi(K) in place; gn = g / den over the g tile
        const int i = threadIdx.x - 128;
        const int r = i / C, ti = i % C;
        const int bh = bh0 + r;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            ok = ok && warp_wait(&bar_full[s], (k / NS) & 1, &abort_flag);
            if (ok) {
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + (nchunk - 1 - k) * C, t = c0 + ti;
                const bool qvalid = t < t1;
                if (CAUSAL) {
                    float inv = 0.f, gdv = 0.f;
                    if (qvalid && LA_CHECK((size_t)bh * p.N + t < (size_t)p.B * p.Hq * p.N, 421, bh, t)) {
                        inv = 1.f / p.den[(size_t)bh * p.N + t];
                        gdv = p.gd[(size_t)bh * p.N + t];
                    }
                    gds[s * 128 + i] = gdv;
#pragma unroll 4
                    for (int c = 0; c < D / 8; ++c) {
                        uint8_t *ch = st + swz_chunk(128, i, c);
                        if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 422, smem_u32(ch) - sm_lo, c))
                            feat8_inplace2(ch, qvalid, p.phi);
                        uint8_t *gch = st + OFF_G + swz_chunk(128, i, c);
                        if (LA_CHECK(in_smem(gch, 16, sm_lo, sm_hi), 423, smem_u32(gch) - sm_lo, c)) {
                            uint4 x = *reinterpret_cast<uint4 *>(gch);
                            uint32_t *xi = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float2 f = unpack_bf16x2(xi[q]);
                                xi[q] = pack_bf16x2(f.x * inv, f.y * inv);
                            }
                            *reinterpret_cast<uint4 *>(gch) = x;
                        }
                    }
                }
                for (int idx = i; idx < C * (D / 8); idx += 128) {
                    const int j = idx / (D / 8), c = idx % (D / 8);
                    uint8_t *ch = st + OFF_K + swz_chunk(C, j, c);
                    if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 424, smem_u32(ch) - sm_lo, idx))
                        feat8_inplace2(ch, c0 + j < t1, p.phi);
                }
                fence_proxy_async();
            }
            mbar_arrive(&bar_ready[s]);
        }
    } else if (warp >= 8 && warp < 12) {
        // ---------------- P / dP conversion (thread = query row) and the dk, dv epilogue
        // (thread = TMEM lane = feature d)
        const int i = threadIdx.x - 256;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int ti = i % C;
        const int d = i;
        float r_d = (d < D) ? rstate[(size_t)d * (D + 1) + D] : 0.f;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            const int c0 = t0 + (nchunk - 1 - k) * C;
            uint8_t *st = stage0 + s * K::STAGE;
            if (CAUSAL) {
                ok = ok && warp_wait(&bar_afull, k & 1, &abort_flag);
                tc_fence_after();
                if (ok) {
                    const float gdi = gds[s * 128 + i];
#pragma unroll 1
                    for (int c16 = 0; c16 < C / 16; ++c16) {
                        float va[16], vd[16];
                        tmem_ld16(tA + lane_off + c16 * 16, va);
                        tmem_ld16(tD + lane_off + c16 * 16, vd);
                        tmem_ld_wait();
                        uint32_t wa[8], wd[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const int j = c16 * 16 + e;
                            const bool m0 = j <= ti, m1 = j + 1 <= ti;
                            wa[e / 2] = pack_bf16x2(m0 ? va[e] : 0.f, m1 ? va[e + 1] : 0.f);
                            wd[e / 2] = pack_bf16x2(m0 ? vd[e] + gdi : 0.f, m1 ? vd[e + 1] + gdi : 0.f);
                        }
                        uint8_t *p0 = pbuf + swz_chunk(128, i, 2 * c16), *p1 = pbuf + swz_chunk(128, i, 2 * c16 + 1);
                        uint8_t *q0 = dpbuf + swz_chunk(128, i, 2 * c16), *q1 = dpbuf + swz_chunk(128, i, 2 * c16 + 1);
                        if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi) &&
                                         in_smem(q0, 16, sm_lo, sm_hi) && in_smem(q1, 16, sm_lo, sm_hi),
                                     431, smem_u32(p0) - sm_lo, c16)) {
                            *reinterpret_cast<uint4 *>(p0) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
                            *reinterpret_cast<uint4 *>(p1) = make_uint4(wa[4], wa[5], wa[6], wa[7]);
                            *reinterpret_cast<uint4 *>(q0) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                            *reinterpret_cast<uint4 *>(q1) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
                        }
                    }
                    fence_proxy_async();
                }
                tc_fence_before();
                mbar_arrive(&bar_pready);
            }
            ok = ok && warp_wait(&bar_outfull, k & 1, &abort_flag);
            tc_fence_after();
            if (ok && wq * 32 < D) {
                __nv_bfloat16 *dkb = static_cast<__nv_bfloat16 *>(p.dk) + (size_t)bg * p.N * D;
                __nv_bfloat16 *dvb = static_cast<__nv_bfloat16 *>(p.dv) + (size_t)bg * p.N * D;
                const uint8_t *kt = st + OFF_K;
#pragma unroll 1
                for (int c16 = 0; c16 < C / 16; ++c16) {
                    float vb[16], vv[16];
                    tmem_ld16(tA + lane_off + c16 * 16, vb);
                    tmem_ld16(tD + lane_off + c16 * 16, vv);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j = c16 * 16 + e, tok = c0 + j;
                        if (tok < t1 && LA_CHECK(((size_t)bg * p.N + tok) * D + d < (size_t)p.B * p.Hkv * p.N * D, 432,
                                                 tok, d)) {
                            const float f = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kt + swz_offset(C, j, d)));
                            dkb[(size_t)tok * D + d] = __float2bfloat16_rn(feat_grad_from_feat(f, p.phi) * (vb[e] + r_d));
                            dvb[(size_t)tok * D + d] = __float2bfloat16_rn(vv[e]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_outfree);
            if (CAUSAL && ok && d < D) {   // this chunk's rows join r for the earlier chunks
                const float *gsd = gds + s * 128;
                for (int row = 0; row < 128; ++row)
                    r_d += gsd[row] * __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(st + swz_offset(128, row, d)));
            }
            mbar_arrive(&bar_empty[s]);
        }
    } else if (warp >= 12) {
        // ---------------- R conversion: TMEM R (fp32) -> R_bf (bf16 operand tile)
        const int d = threadIdx.x - 384;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        if (wq * 32 < D) {
            const float *row = rstate + (size_t)d * (D + 1);
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = row[c16 * 16 + e];
                if (CAUSAL) tmem_st16(tR + lane_off + c16 * 16, v);
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                *reinterpret_cast<uint4 *>(rbf + swz_chunk(128, d, 2 * c16)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(rbf + swz_chunk(128, d, 2 * c16 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
            if (CAUSAL) tmem_st_wait();
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_rbf);
        if (CAUSAL) {
            bool ok = true;
            for (int k = 0; k < nchunk; ++k) {
                ok = ok && warp_wait(&bar_rfull, k & 1, &abort_flag);
                tc_fence_after();
                if (ok && wq * 32 < D) {
#pragma unroll 1
                    for (int c16 = 0; c16 < D / 16; ++c16) {
                        float v[16];
                        tmem_ld16(tR + lane_off + c16 * 16, v);
                        tmem_ld_wait();
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                        *reinterpret_cast<uint4 *>(rbf + swz_chunk(128, d, 2 * c16)) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4 *>(rbf + swz_chunk(128, d, 2 * c16 + 1)) =
                            make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(&bar_rbf);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (threadIdx.x == 0 && abort_flag) atomicExch(p.err, kErrTimeout);
}

// ---------------------------------------------------------------------------------------
// Host side

template <int D, int G, bool CAUSAL>
cudaError_t launch_bwd_kernels(const Params &p, cudaStream_t s) {
    using K = BwdCfg<D, G>;
    CUtensorMap mq{}, mk{}, mv{}, mg{};
    cudaError_t e = make_map(&mq, p.q, p.B * p.Hq, p.N, D, K::C);
    if (e == cudaSuccess) e = make_map(&mk, p.k, p.B * p.Hkv, p.N, D, K::C);
    if (e == cudaSuccess) e = make_map(&mv, p.v, p.B * p.Hkv, p.N, D, K::C);
    if (e == cudaSuccess) e = make_map(&mg, p.g, p.B * p.Hq, p.N, D, K::C);
    if (e == cudaSuccess) e = prepare(k_tc_bwd_dq<D, G, CAUSAL>, K::DQ_SMEM);
    if (e == cudaSuccess) e = prepare(k_tc_bwd_dkdv<D, G, CAUSAL>, K::DKDV_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = p.B * p.Hkv * p.nseg;
    {
        TraceScope ts(CAUSAL ? "tc_bwd_dq_causal" : "tc_bwd_dq_bidir", s);
        k_tc_bwd_dq<D, G, CAUSAL><<<grid, 512, K::DQ_SMEM, s>>>(mq, mk, mv, mg, p);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = scan_segments(p.rstate, p, CAUSAL ? kScanSuffix : kScanTotal, (size_t)D * (D + 1), s);
    if (e != cudaSuccess) return e;
    TraceScope ts(CAUSAL ? "tc_bwd_dkdv_causal" : "tc_bwd_dkdv_bidir", s);
    k_tc_bwd_dkdv<D, G, CAUSAL><<<grid, 512, K::DKDV_SMEM, s>>>(mq, mk, mv, mg, p);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t backward_dg(const Params &p, cudaStream_t s) {
    if constexpr (!BwdCfg<D, G>::FITS) {
        return cudaErrorNotSupported;
    } else {
        cudaError_t e = tc_launch_state(p, s);
        if (e == cudaSuccess)
            e = scan_segments(p.state, p, p.causal ? kScanPrefix : kScanTotal, (size_t)D * (D + 1), s);
        if (e != cudaSuccess) return e;
        return p.causal ? launch_bwd_kernels<D, G, true>(p, s) : launch_bwd_kernels<D, G, false>(p, s);
    }
}

template <int D>
cudaError_t backward_d(const Params &p, cudaStream_t s) {
    switch (p.n_rep) {
        case 1: return backward_dg<D, 1>(p, s);
        case 2: return backward_dg<D, 2>(p, s);
        case 4: return backward_dg<D, 4>(p, s);
        case 8: return backward_dg<D, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool tc_bwd_supported(int n_rep, int D) {
    if (D == 128) return n_rep == 4 || n_rep == 8;
    if (D == 64) return n_rep == 1 || n_rep == 2 || n_rep == 4 || n_rep == 8;
    return false;
}

cudaError_t tc_backward(const Params &p, cudaStream_t s) {
    return p.D == 128 ? backward_d<128>(p, s) : (p.D == 64 ? backward_d<64>(p, s) : cudaErrorNotSupported);
}

}  // namespace la

#ifdef LA_DEBUG
// Debug builds only: the first failed self-check of the backward kernels (id, a, b, block).
extern "C" int la_debug_read_bwd(int *out4) {
    if (cudaMemcpyFromSymbol(out4, la::g_la_debug, 4 * sizeof(int)) != cudaSuccess) return 1;
    const int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(la::g_la_debug, zero, 4 * sizeof(int)) == cudaSuccess ? 0 : 1;
}
#endif
