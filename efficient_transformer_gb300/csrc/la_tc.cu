// la_tc.cu -- tensor-core kernels (tcgen05 / TMEM / TMA) for bfloat16 inputs.
//
// The dense contractions of the chunked linear attention ("chunked causal streaming" and
// "bidirectional parallel reduction" in the linear_attn module docstring) run as
// tcgen05.mma with bf16 operands in 128-byte-swizzled shared memory and fp32 accumulators
// in TMEM; tiles arrive by TMA.  The query rows of one chunk are the n_rep heads of a
// key/value group stacked on the MMA's M = 128 rows (G = n_rep heads x C = 128 / G
// tokens), so one key/value tile serves the whole group (the gqa page's head sharing,
// fused: no expanded k, v).
//
// Forward = k_tc_state (per-segment S = phi(K)^T V, z = colsum phi(K)) -> k_scan
// (exclusive prefix, or total when bidirectional; CUDA cores) -> k_tc_fwd.  Per chunk of
// k_tc_fwd (M = 128 query rows, C keys):
//   MMA1  A   = phi(Q) phi(K)^T                 [128 x C]   (causal)
//   conv  P   = bf16(A masked j <= i); den_intra = rowsum P  (CUDA cores)
//   MMA2  O   = P V + phi(Q) S_bf                [128 x D]
//   epi   out = O / (den_intra + phi(Q) . z + eps)           (CUDA cores, fp32)
//   MMA3  S  += phi(K)^T V                       [D x D]     (causal)
//   conv  S_bf = bf16(S) for the next chunk's readout; z += colsum phi(K) (fp32)
// Warp roles (512 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM owner,
// warps 4-7 phi prologue (in place on the swizzled tiles), warps 8-11 P conversion and
// epilogue, warps 12-15 state conversion.
#include "la_tc_common.cuh"

namespace la {
namespace {

template <int D, int G>
struct FwdCfg {
    static constexpr int C = 128 / G;                  // tokens per chunk
    static constexpr int DB = D / 64;                  // 64-wide blocks per D-wide row
    static constexpr int Q_BYTES = 128 * D * 2;        // 128 query rows
    static constexpr int K_BYTES = C * D * 2;
    static constexpr int V_BYTES = C * D * 2;
    static constexpr int STAGE = Q_BYTES + K_BYTES + V_BYTES;
    static constexpr int P_BYTES = ((C + 63) / 64) * 128 * 128;
    static constexpr int S_BYTES = DB * D * 128;       // D rows (d) x D columns (e)
    static constexpr int FIXED = 2 * P_BYTES + S_BYTES + 2 * D * 4 + 1024;
    static constexpr int NS = (kSmemLimit - FIXED) / STAGE > 4 ? 4 : (kSmemLimit - FIXED) / STAGE;
    static constexpr int SMEM = NS * STAGE + FIXED;
    static_assert(NS >= 2, "not enough shared memory for two stages");
};

template <int D>
struct StateCfg {
    static constexpr int C = 128;
    static constexpr int DB = D / 64;
    static constexpr int K_BYTES = C * D * 2;
    static constexpr int STAGE = 2 * K_BYTES;          // K then V
    static constexpr int NS = (kSmemLimit - 1024) / STAGE > 6 ? 6 : (kSmemLimit - 1024) / STAGE;
    static constexpr int SMEM = NS * STAGE + 1024;
};

// ---------------------------------------------------------------------------------------
// Per-segment state: S = sum_j phi(k_j) v_j^T (MMA, fp32 in TMEM), z = sum_j phi(k_j)
// (CUDA cores, fp32), written to the workspace as [D][D+1] with z in column D.
template <int D>
__global__ void __launch_bounds__(256, 1) k_tc_state(const __grid_constant__ CUtensorMap map_k,
                                                     const __grid_constant__ CUtensorMap map_v, Params p) {
    using K = StateCfg<D>;
    constexpr int C = K::C, NS = K::NS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full[NS], bar_ready[NS], bar_empty[NS], bar_done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::SMEM;
    (void)sm_lo;
    (void)sm_hi;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_ready[s], 128);
            mbar_init(&bar_empty[s], 1);
        }
        mbar_init(&bar_done, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch(&map_k);
            tma_prefetch(&map_v);
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (k >= NS && !mbar_wait(&bar_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C;
                mbar_arrive_expect_tx(&bar_full[s], K::STAGE);
                for (int blk = 0; blk < K::DB; ++blk) {
                    uint8_t *dk_ = st + blk * C * 128, *dv_ = st + K::K_BYTES + blk * C * 128;
                    if (LA_CHECK(in_smem(dk_, C * 128, sm_lo, sm_hi) && (smem_u32(dk_) & 1023) == 0, 101,
                                 smem_u32(dk_) - sm_lo, k) &&
                        LA_CHECK(c0 < p.N && bg < p.B * p.Hkv, 102, c0, bg))
                        tma_load_3d(dk_, &map_k, &bar_full[s], blk * 64, c0, bg);
                    if (LA_CHECK(in_smem(dv_, C * 128, sm_lo, sm_hi) && (smem_u32(dv_) & 1023) == 0, 103,
                                 smem_u32(dv_) - sm_lo, k))
                        tma_load_3d(dv_, &map_v, &bar_full[s], blk * 64, c0, bg);
                }
                issued = k + 1;
            }
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k) mbar_drain(&bar_full[k % NS], (k / NS) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(128, D, true, true);
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (!mbar_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t ks_ = smem_u32(stage0 + s * K::STAGE), vs_ = ks_ + K::K_BYTES;
                // A spans 2 blocks of C rows (M = 128), B spans DB blocks
                if (LA_CHECK(ks_ >= sm_lo && ks_ + 2u * C * 128u <= sm_hi, 111, ks_ - sm_lo, k) &&
                    LA_CHECK(vs_ + (uint32_t)K::DB * C * 128u <= sm_hi, 112, vs_ - sm_lo, k))
                    for (int kk = 0; kk < C / 16; ++kk)
                        mma_bf16(tS, desc_mnmajor(ks_, C, 0, kk), desc_mnmajor(vs_, C, 0, kk), idS,
                                 (k > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bar_empty[s]);
            }
            mma_commit(&bar_done);
            mbar_drain(&bar_done, 0);
        }
    } else if (warp >= 4) {
        const int i = threadIdx.x - 128;           // 0..127: column d for z, lane of TMEM
        float z = 0.f;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            ok = ok && warp_wait(&bar_full[s], (k / NS) & 1, &abort_flag);
            uint8_t *kt = stage0 + s * K::STAGE;
            const int c0 = t0 + k * C;
            if (ok) {
                for (int idx = i; idx < C * (D / 8); idx += 128) {
                    const int j = idx / (D / 8), c = idx % (D / 8);
                    uint8_t *ch = kt + swz_chunk(C, j, c);
                    if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 121, smem_u32(ch) - sm_lo, idx))
                        feat8_inplace(ch, c0 + j < t1, p.phi);
                }
            }
            named_barrier(1, 128);
            if (ok && i < D)
                for (int j = 0; j < C; ++j) {
                    const uint8_t *e_ = kt + swz_offset(C, j, i);
                    if (LA_CHECK(in_smem(e_, 2, sm_lo, sm_hi), 122, smem_u32(e_) - sm_lo, j))
                        z += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(e_));
                }
            fence_proxy_async();
            mbar_arrive(&bar_ready[s]);
        }
        ok = ok && warp_wait(&bar_done, 0, &abort_flag);
        tc_fence_after();
        float *dst = p.state + ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1));
        const int wq = warp % 4;
        if (ok && wq * 32 < D) {
            const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
            float *row = dst + (size_t)i * (D + 1);
            const size_t row_idx = ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1)) + (size_t)i * (D + 1);
            (void)row_idx;
            const bool row_ok = LA_CHECK(row_idx + D + 1 <= (size_t)p.B * p.Hkv * p.nseg * D * (D + 1), 131,
                                         row_idx, i);
            for (int c16 = 0; c16 < D / 16; ++c16) {
                float v[16];
                if (LA_CHECK(c16 * 16 + 16 <= 128, 132, c16, i)) {
                    tmem_ld16(tS + lane_off + c16 * 16, v);
                    tmem_ld_wait();
                }
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (row_ok) row[c16 * 16 + e] = nchunk > 0 ? v[e] : 0.f;
            }
            if (row_ok) row[D] = z;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tS, 128);
    if (threadIdx.x == 0 && abort_flag) atomicExch(p.err, kErrTimeout);
}

// ---------------------------------------------------------------------------------------
// Chunked forward (see the file comment for the per-chunk steps and warp roles).
template <int D, int G, bool CAUSAL>
__global__ void __launch_bounds__(512, 1) k_tc_fwd(const __grid_constant__ CUtensorMap map_q,
                                                   const __grid_constant__ CUtensorMap map_k,
                                                   const __grid_constant__ CUtensorMap map_v, Params p) {
    using K = FwdCfg<D, G>;
    constexpr int C = K::C, NS = K::NS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full[NS], bar_ready[NS], bar_empty[NS];
    __shared__ uint64_t bar_afull, bar_pready, bar_ofull, bar_ofree, bar_sfull, bar_sbf, bar_fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::SMEM;
    (void)sm_lo;
    (void)sm_hi;
    uint8_t *ptile = stage0 + NS * K::STAGE;
    uint8_t *sbf = ptile + 2 * K::P_BYTES;
    float *zf = reinterpret_cast<float *>(sbf + K::S_BYTES);   // [2][D]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;
    const int bh0 = b * p.Hq + g * G;
    const float *state = p.state + ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1));
    const size_t state_base = ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1));
    const size_t state_total = (size_t)p.B * p.Hkv * p.nseg * D * (D + 1);
    (void)state_base;
    (void)state_total;

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
        mbar_init(&bar_ofree, 128);
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
    const uint32_t tS = tmem_base, tO = tmem_base + 128, tA = tmem_base + 256;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            tma_prefetch(&map_q);
            if (CAUSAL) {
                tma_prefetch(&map_k);
                tma_prefetch(&map_v);
            }
            constexpr uint32_t bytes = CAUSAL ? K::STAGE : K::Q_BYTES;
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (k >= NS && !mbar_wait(&bar_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C;
                mbar_arrive_expect_tx(&bar_full[s], bytes);
                for (int r = 0; r < G; ++r)
                    for (int blk = 0; blk < K::DB; ++blk) {
                        uint8_t *dq_ = st + blk * 128 * 128 + r * C * 128;
                        if (LA_CHECK(in_smem(dq_, C * 128, sm_lo, sm_hi) && (smem_u32(dq_) & 1023) == 0, 201,
                                     smem_u32(dq_) - sm_lo, k) &&
                            LA_CHECK(c0 < p.N && bh0 + r < p.B * p.Hq, 202, c0, bh0 + r))
                            tma_load_3d(dq_, &map_q, &bar_full[s], blk * 64, c0, bh0 + r);
                    }
                if (CAUSAL)
                    for (int blk = 0; blk < K::DB; ++blk) {
                        uint8_t *dk_ = st + K::Q_BYTES + blk * C * 128, *dv_ = dk_ + K::K_BYTES;
                        if (LA_CHECK(in_smem(dk_, C * 128, sm_lo, sm_hi) && in_smem(dv_, C * 128, sm_lo, sm_hi) &&
                                         (smem_u32(dk_) & 1023) == 0 && (smem_u32(dv_) & 1023) == 0,
                                     203, smem_u32(dk_) - sm_lo, k)) {
                            tma_load_3d(dk_, &map_k, &bar_full[s], blk * 64, c0, bg);
                            tma_load_3d(dv_, &map_v, &bar_full[s], blk * 64, c0, bg);
                        }
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
            constexpr uint32_t idS = idesc_bf16(128, D, true, true);
            const uint32_t sbf_u = smem_u32(sbf);
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (!mbar_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), ks_ = qs + K::Q_BYTES, vs = ks_ + K::K_BYTES;
                const uint32_t pb = smem_u32(ptile + (k & 1) * K::P_BYTES);
                const bool ranges_ok =
                    LA_CHECK(qs >= sm_lo && qs + K::Q_BYTES <= sm_hi, 211, qs - sm_lo, k) &&
                    LA_CHECK(ks_ + 2u * C * 128u <= sm_hi, 212, ks_ - sm_lo, k) &&
                    LA_CHECK(vs + K::V_BYTES <= sm_hi, 213, vs - sm_lo, k) &&
                    LA_CHECK(pb + K::P_BYTES <= sm_hi, 214, pb - sm_lo, k) &&
                    LA_CHECK(sbf_u + K::S_BYTES <= sm_hi, 215, sbf_u - sm_lo, k);
                if (!ranges_ok) break;
                if (CAUSAL) {
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16(tA, desc_kmajor(qs, 128, 0, kk), desc_kmajor(ks_, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                    mma_commit(&bar_afull);
                    if (!mbar_wait(&bar_pready, k & 1, &abort_flag)) break;
                }
                if ((CAUSAL || k == 0) && !mbar_wait(&bar_sbf, k & 1, &abort_flag)) break;
                if (k > 0 && !mbar_wait(&bar_ofree, (k - 1) & 1, &abort_flag)) break;
                tc_fence_after();
                uint32_t acc = 0;
                if (CAUSAL)
                    for (int kk = 0; kk < C / 16; ++kk, acc = 1)
                        mma_bf16(tO, desc_kmajor(pb, 128, 0, kk), desc_mnmajor(vs, C, 0, kk), idO, acc);
                for (int kk = 0; kk < D / 16; ++kk, acc = 1)
                    mma_bf16(tO, desc_kmajor(qs, 128, 0, kk), desc_mnmajor(sbf_u, D, 0, kk), idO, acc);
                mma_commit(&bar_ofull);
                if (CAUSAL) {
                    for (int kk = 0; kk < C / 16; ++kk)
                        mma_bf16(tS, desc_mnmajor(ks_, C, 0, kk), desc_mnmajor(vs, C, 0, kk), idS, 1u);
                    mma_commit(&bar_sfull);
                }
                mma_commit(&bar_empty[s]);
            }
            mma_commit(&bar_fin);
            mbar_drain(&bar_fin, 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- phi prologue, in place on the swizzled Q and K tiles
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
                    if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 221, smem_u32(ch) - sm_lo, c))
                        feat8_inplace(ch, qvalid, p.phi);
                }
                if (CAUSAL)
                    for (int idx = i; idx < C * (D / 8); idx += 128) {
                        const int j = idx / (D / 8), c = idx % (D / 8);
                        uint8_t *ch = st + K::Q_BYTES + swz_chunk(C, j, c);
                        if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 222, smem_u32(ch) - sm_lo, idx))
                            feat8_inplace(ch, c0 + j < t1, p.phi);
                    }
                fence_proxy_async();
            }
            mbar_arrive(&bar_ready[s]);
        }
    } else if (warp >= 8 && warp < 12) {
        // ---------------- P conversion and epilogue (thread = query row of the chunk)
        const int i = threadIdx.x - 256;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int r = i / C, ti = i % C;
        const int bh = bh0 + r;
        if (i < D && LA_CHECK(state_base + (size_t)i * (D + 1) + D < state_total, 231, i, 0) &&
            LA_CHECK(in_smem(zf + i, 4, sm_lo, sm_hi), 232, i, 0))
            zf[i] = state[(size_t)i * (D + 1) + D];
        named_barrier(1, 128);
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            const int c0 = t0 + k * C, t = c0 + ti;
            uint8_t *st = stage0 + s * K::STAGE;
            float den_intra = 0.f;
            if (CAUSAL) {
                ok = ok && warp_wait(&bar_afull, k & 1, &abort_flag);
                tc_fence_after();
                if (ok) {
                    uint8_t *pb = ptile + (k & 1) * K::P_BYTES;
#pragma unroll 1
                    for (int c16 = 0; c16 < C / 16; ++c16) {
                        float v[16];
                        if (LA_CHECK(256 + c16 * 16 + 16 <= 512, 241, c16, i)) {
                            tmem_ld16(tA + lane_off + c16 * 16, v);
                            tmem_ld_wait();
                        }
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const int j = c16 * 16 + e;
                            const float x0 = (j <= ti) ? v[e] : 0.f, x1 = (j + 1 <= ti) ? v[e + 1] : 0.f;
                            w[e / 2] = pack_bf16x2(x0, x1);
                            const float2 f = unpack_bf16x2(w[e / 2]);
                            den_intra += f.x + f.y;
                        }
                        uint8_t *p0 = pb + swz_chunk(128, i, 2 * c16), *p1 = pb + swz_chunk(128, i, 2 * c16 + 1);
                        if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi), 242,
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
            ok = ok && warp_wait(&bar_ofull, k & 1, &abort_flag);
            tc_fence_after();
            if (ok) {
                // den = rowsum P + phi(q_i) . z + eps, in fp32
                const float *z = zf + (CAUSAL ? (k & 1) * D : 0);
                float dint = 0.f;
#pragma unroll 4
                for (int c = 0; c < D / 8; ++c) {
                    const uint8_t *ch = st + swz_chunk(128, i, c);
                    if (!LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi) && in_smem(z + c * 8, 32, sm_lo, sm_hi), 251,
                                  smem_u32(ch) - sm_lo, c))
                        continue;
                    const uint4 x = *reinterpret_cast<const uint4 *>(ch);
                    const uint32_t *xi = reinterpret_cast<const uint32_t *>(&x);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 f = unpack_bf16x2(xi[h]);
                        dint += f.x * z[c * 8 + 2 * h] + f.y * z[c * 8 + 2 * h + 1];
                    }
                }
                const float inv = 1.f / (den_intra + dint + p.eps);
                __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.out) + ((size_t)bh * p.N + t) * D;
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    float v[16];
                    if (LA_CHECK(128 + c16 * 16 + 16 <= 256, 252, c16, i)) {
                        tmem_ld16(tO + lane_off + c16 * 16, v);
                        tmem_ld_wait();
                    }
                    if (t < t1 && LA_CHECK(((size_t)bh * p.N + t) * D + c16 * 16 + 16 <= (size_t)p.B * p.Hq * p.N * D,
                                           253, bh, t)) {
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e] * inv, v[2 * e + 1] * inv);
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c16 * 16);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_ofree);
            if (CAUSAL && ok && i < D) {   // z for the next chunk: z += colsum phi(K) (fp32)
                const uint8_t *kt = st + K::Q_BYTES;
                float zs = zf[(k & 1) * D + i];
                for (int j = 0; j < C; ++j) {
                    const uint8_t *e_ = kt + swz_offset(C, j, i);
                    if (LA_CHECK(in_smem(e_, 2, sm_lo, sm_hi), 261, smem_u32(e_) - sm_lo, j))
                        zs += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(e_));
                }
                if (LA_CHECK(in_smem(zf + ((k + 1) & 1) * D + i, 4, sm_lo, sm_hi), 262, i, k))
                    zf[((k + 1) & 1) * D + i] = zs;
            }
            mbar_arrive(&bar_empty[s]);
            named_barrier(1, 128);
        }
    } else if (warp >= 12) {
        // ---------------- state conversion: TMEM S (fp32) -> S_bf (bf16 operand tile)
        const int d = threadIdx.x - 384;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        if (wq * 32 < D) {
            const float *row = state + (size_t)d * (D + 1);
            const bool row_ok = LA_CHECK(state_base + (size_t)d * (D + 1) + D + 1 <= state_total, 271, d, 0);
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = row_ok ? row[c16 * 16 + e] : 0.f;
                if (CAUSAL && LA_CHECK(c16 * 16 + 16 <= 128, 272, c16, d)) tmem_st16(tS + lane_off + c16 * 16, v);
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                uint8_t *p0 = sbf + swz_chunk(D, d, 2 * c16), *p1 = sbf + swz_chunk(D, d, 2 * c16 + 1);
                if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi), 273,
                             smem_u32(p0) - sm_lo, d)) {
                    *reinterpret_cast<uint4 *>(p0) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(p1) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            if (CAUSAL) tmem_st_wait();
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_sbf);
        if (CAUSAL) {
            bool ok = true;
            for (int k = 0; k < nchunk; ++k) {
                ok = ok && warp_wait(&bar_sfull, k & 1, &abort_flag);
                tc_fence_after();
                if (ok && wq * 32 < D) {
#pragma unroll 1
                    for (int c16 = 0; c16 < D / 16; ++c16) {
                        float v[16];
                        if (LA_CHECK(c16 * 16 + 16 <= 128, 281, c16, d)) {
                            tmem_ld16(tS + lane_off + c16 * 16, v);
                            tmem_ld_wait();
                        }
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                        uint8_t *p0 = sbf + swz_chunk(D, d, 2 * c16), *p1 = sbf + swz_chunk(D, d, 2 * c16 + 1);
                        if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi), 282,
                                     smem_u32(p0) - sm_lo, d)) {
                            *reinterpret_cast<uint4 *>(p0) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4 *>(p1) = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(&bar_sbf);
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

template <int D>
cudaError_t launch_state(const Params &p, cudaStream_t s) {
    CUtensorMap mk{}, mv{};
    cudaError_t e = make_map(&mk, p.k, p.B * p.Hkv, p.N, D, StateCfg<D>::C);
    if (e == cudaSuccess) e = make_map(&mv, p.v, p.B * p.Hkv, p.N, D, StateCfg<D>::C);
    if (e == cudaSuccess) e = prepare(k_tc_state<D>, StateCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    TraceScope ts("tc_seg_state", s);
    k_tc_state<D><<<p.B * p.Hkv * p.nseg, 256, StateCfg<D>::SMEM, s>>>(mk, mv, p);
    return cudaGetLastError();
}

template <int D, int G, bool CAUSAL>
cudaError_t launch_fwd(const Params &p, cudaStream_t s) {
    using K = FwdCfg<D, G>;
    CUtensorMap mq{}, mk{}, mv{};
    cudaError_t e = make_map(&mq, p.q, p.B * p.Hq, p.N, D, K::C);
    if (e == cudaSuccess) e = make_map(&mk, p.k, p.B * p.Hkv, p.N, D, K::C);
    if (e == cudaSuccess) e = make_map(&mv, p.v, p.B * p.Hkv, p.N, D, K::C);
    if (e == cudaSuccess) e = prepare(k_tc_fwd<D, G, CAUSAL>, K::SMEM);
    if (e != cudaSuccess) return e;
    TraceScope ts(CAUSAL ? "tc_fwd_causal" : "tc_fwd_bidir", s);
    k_tc_fwd<D, G, CAUSAL><<<p.B * p.Hkv * p.nseg, 512, K::SMEM, s>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t forward_dg(const Params &p, cudaStream_t s) {
    cudaError_t e = launch_state<D>(p, s);
#ifdef LA_DEBUG
    const char *stop = getenv("LA_DEBUG_STOP");
    if (stop && stop[0] == 's' && stop[1] == 't') return e;      // "state"
#endif
    if (e == cudaSuccess)
        e = scan_segments(p.state, p, p.causal ? kScanPrefix : kScanTotal, (size_t)D * (D + 1), s);
#ifdef LA_DEBUG
    if (stop && stop[0] == 's' && stop[1] == 'c') return e;      // "scan"
#endif
    if (e != cudaSuccess) return e;
    return p.causal ? launch_fwd<D, G, true>(p, s) : launch_fwd<D, G, false>(p, s);
}

template <int D>
cudaError_t forward_d(const Params &p, cudaStream_t s) {
    switch (p.n_rep) {
        case 1:
            if constexpr (D == 64) return forward_dg<D, 1>(p, s);
            return cudaErrorNotSupported;
        case 2: return forward_dg<D, 2>(p, s);
        case 4: return forward_dg<D, 4>(p, s);
        case 8: return forward_dg<D, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

int tc_chunk(int n_rep) { return 128 / n_rep; }

bool tc_supported(int Hq, int Hkv, int N, int D, la_dtype dt, int P, int causal, int is_bwd) {
    (void)N;
    (void)causal;
    if (dt != LA_BF16 || P != 1) return false;
    const int n_rep = Hq / Hkv;
    if (is_bwd) return tc_bwd_supported(n_rep, D);
    if (D == 128) return n_rep == 2 || n_rep == 4 || n_rep == 8;
    if (D == 64) return n_rep == 1 || n_rep == 2 || n_rep == 4 || n_rep == 8;
    return false;
}

cudaError_t tc_forward(const Params &p, cudaStream_t s) {
    return p.D == 128 ? forward_d<128>(p, s) : (p.D == 64 ? forward_d<64>(p, s) : cudaErrorNotSupported);
}

cudaError_t tc_launch_state(const Params &p, cudaStream_t s) {
    return p.D == 128 ? launch_state<128>(p, s) : (p.D == 64 ? launch_state<64>(p, s) : cudaErrorNotSupported);
}

}  // namespace la

#ifdef LA_DEBUG
// Debug builds only: copy out and clear the first failed self-check (id, a, b, block).
extern "C" int la_debug_read(int *out4) {
    if (cudaMemcpyFromSymbol(out4, la::g_la_debug, 4 * sizeof(int)) != cudaSuccess) return 1;
    const int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(la::g_la_debug, zero, 4 * sizeof(int)) == cudaSuccess ? 0 : 1;
}
#endif
