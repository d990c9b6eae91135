// la_tc_bwd.cu -- tensor-core backward (tcgen05 / TMEM / TMA) for bfloat16 inputs.
//
// The gradient of the linear_attn page's `fwd` (its `bwd` differentiates `fwd`), without
// re-running the forward through autograd.  With gn_i = g_i / den_i and
// gd_i = -(g_i . num_i) / den_i^2, the forward's chunked structure carries over to the
// backward: dA_ij = gn_i . v_j + gd_i (j <= i) plays the role of the scores, and the
// suffix state R = sum_{i after} phi(q_i) gn_i^T, r = sum gd_i phi(q_i) carries the rows
// that come later.  Launch order:
//
//   (the forward: k_tc_state -> scan -> k_tc_fwd, with dq as its output scratch; skipped
//    when the caller's forward workspace gives the states and the per-row den)
//   k_tc_bwd_dq   forward over chunks: dq, per-row h, each segment's R and r, and (causal)
//                 the rows phi_s = phi(q) / den for the next kernel
//   scan (suffix R)
//   k_tc_bwd_dkdv reverse over chunks: dk, dv (summed over the n_rep heads of the group),
//                 reading phi_s where the dq kernel read q
//
// Per chunk of k_tc_bwd_dq (128 stacked query rows, C keys), with the raw grad_out g and
// the forward's den (incl. eps) per row:
//   phi_s = phi(q) / den (bf16, the feature map scales Q's rows in place)
//   A_s = phi_s phi(K)^T,  dA' = g V^T,  X = g S_bf^T,  R += phi_s^T g (= phi(Q)^T gn)
//   g . num / den = phi_s . X + sum_j mask(A_s) dA'      (no O product is needed)
//   h = -(g . num) / den,  gd = h / den,  dP' = mask(dA' + h) = den * dP
//   X += dP' phi(K) + h z = den * da,  dq = phi'(q) / den * X
//   r += phi_s^T h (= phi(Q)^T gd),  S += phi(K)^T V
// Per chunk of k_tc_bwd_dkdv, computed transposed so the 128 query rows stay on the MMA's
// K dimension (and the sum over the group's heads comes for free):
//   dk^T = phi(Q)^T dP + R_bf V^T (+ r),  dv^T = gn^T P + R_bf^T phi(K)^T,  R += phi(Q)^T gn
// Warp roles: warp 0 TMA, warp 1 MMA, warp 2 the TMA stores.  The dq kernel runs the feature
// map on warps 4-7 and 16-23 (16-23 also convert S), its row work and dq on a pool of warps
// 8-15; the dk/dv kernel runs the feature map of K on warps 16-23, R conversion and the dk,
// dv epilogues on warps 8-11, and P' / dP' on warps 12-15 with warps 4-7.
#include "la_tc_common.cuh"

namespace la {
namespace {

// Threads per CTA (80 registers a thread) and feature-map threads (dq: warps 4-7 and 16-23;
// dk/dv: warps 16-23).
constexpr int kDqThreads = 768, kDqPro = 384;
constexpr int kKvThreads = 768, kKvPro = 256;

template <int D, int G>
struct BwdCfg {
    static constexpr int C = 128 / G;
    static constexpr int DB = D / 64;
    static constexpr int CB = (C + 63) / 64;
    static constexpr int Q_BYTES = 128 * D * 2;
    static constexpr int K_BYTES = C * D * 2;
    static constexpr int V_BYTES = C * D * 2;
    static constexpr int G_BYTES = 128 * D * 2;
    static constexpr int STAGE = Q_BYTES + K_BYTES + V_BYTES + G_BYTES;   // [phi(Q) | phi(K) | V | g]
    static constexpr int P_BYTES = CB * 128 * 128;
    static constexpr int S_BYTES = DB * D * 128;            // S_bf: D rows (d) x D columns (e)
    static constexpr int Z_BYTES = DB * 16 * 128;           // z: 16 rows x D columns (rows 0-2: hi, lo, hi)
    static constexpr int ONES_BYTES = CB * 16 * 128;        // ones: 16 rows x C columns
    static constexpr int H_BYTES = 2 * 16 * 128;            // h: 16 rows x 128 query rows (rows 0-2: hi, hi, lo)
    static constexpr int XCH_BYTES = 2 * 128 * 4;           // partial row dots of the two pool halves
    // dq kernel: stages (with the rows' den: 128 floats, padded to keep the stages 1024-byte
    // aligned), dP', S_bf, two z slots, ones, h, exchange
    static constexpr int DEN_BYTES = 1024;
    // each head's C dens land at a 128-byte aligned slot of DPAD floats (a TMA destination in
    // shared memory must be 128-byte aligned): row i = r C + ti sits at r DPAD + ti
    static constexpr int DPAD = C < 32 ? 32 : C;
    static_assert(G * DPAD * 4 <= DEN_BYTES, "den slots");
    static constexpr int STAGE_DQ = STAGE + DEN_BYTES;   // [phi_s | phi(K) | V | g | den]
    static constexpr int DQ_FIXED = P_BYTES + S_BYTES + 2 * Z_BYTES + ONES_BYTES + H_BYTES + XCH_BYTES + 1024;
    static constexpr int NS_DQ = 3 * STAGE_DQ + DQ_FIXED <= kSmemLimit - 512 ? 3 : 2;
    static constexpr int DQ_SMEM = NS_DQ * STAGE_DQ + DQ_FIXED;
    // dk/dv kernel: stages, P', dP', R_bf, h (a 16 x 128 tile unless it fits as two spare
    // columns of dP' next to the C keys)
    static constexpr bool H_IN_DP = C % 64 != 0 && C % 64 + 16 <= 64;
    static constexpr int RBF_BYTES = D * 128 * 2;           // R_bf: D rows x 128 columns
    static constexpr int PT_BYTES = C * 256;                // P'^T: C rows (keys) x 128 columns
    // dk and dv leave through a staging tile of their own (C rows x D columns, one after the
    // other), so that the [K | V] region goes back to the loader before the epilogue; for
    // C > 32 the outputs are written over phi(K) and V instead
    static constexpr bool OUT_STAGE = C <= 32;
    static constexpr int OUT_BYTES = OUT_STAGE ? C * D * 2 : 0;
    static constexpr int KV_FIXED = PT_BYTES + P_BYTES + RBF_BYTES + (H_IN_DP ? 0 : H_BYTES) + OUT_BYTES + 1024;
    static constexpr int NS = 3 * STAGE + KV_FIXED <= kSmemLimit - 512 ? 3 : 2;
    static constexpr int DKDV_SMEM = NS * STAGE + KV_FIXED;
    static constexpr bool FITS = DQ_SMEM <= kSmemLimit - 512 && DKDV_SMEM <= kSmemLimit - 512;
    // dk/dv kernel TMEM columns: R, then NB_KV buffers of [A_s | dA' | dk^T | r part | dv^T]
    // when dk^T and dv^T fit in columns of their own (KV_SEP), else of
    // [A_s then dk^T | dA' then dv^T | r part]; the r part (16 columns) takes phi_s^T h
    static constexpr int KT_R = 0;
    static constexpr int KT_AD = D;
    static constexpr bool KV_SEP = KT_AD + 4 * C + 16 <= 512;
    static constexpr int KV_BW = KV_SEP ? 4 * C + 16 : 2 * C + 16;
    static constexpr int NB_KV = KT_AD + 2 * KV_BW <= 512 ? 2 : 1;
    // phi_s^T h rides on the dk^T product as 16 extra columns of dP' (h in dP')
    static constexpr bool MERGE_H = KV_SEP && H_IN_DP;
    // dq kernel TMEM columns: [S | z], (16 free), A_s, dA', X (then den * da), [R | r]
    static constexpr int T_S = 0;
    static constexpr int T_A = D + 32;
    static constexpr int T_A2 = T_A + C;
    static constexpr int T_X = T_A2 + C;
    static constexpr int T_R = T_X + D;
    static constexpr bool TMEM_FITS = T_R + D + 16 <= 512 && KT_AD + KV_BW <= 512;
    static_assert(T_S == 0 && KT_R == 0, "S (dq kernel) and R (dk/dv kernel) start the TMEM allocation");
    static_assert(NB_KV == 1 || NB_KV == 2, "one or two dk/dv TMEM buffers");
};

// phi'(k) from phi(k): elu+1: phi = x + 1 > 1 for x > 0 (derivative 1), phi = exp(x) <= 1
// otherwise (derivative exp(x) = phi); relu: 1 where phi > thr = 0; identity: 1 (thr = -inf,
// so that relu and identity share one comparison).
__device__ __forceinline__ float feat_grad_threshold(int phi) { return phi == LA_PHI_IDENTITY ? -INFINITY : 0.f; }
__device__ __forceinline__ float feat_grad_from_feat(float f, bool elu, float thr) {
    return elu ? fminf(f, 1.f) : (f > thr ? 1.f : 0.f);
}
// ... and w phi'(k) from the weighted feature f = w phi(k) (w >= 0): min(f, w) for elu+1.
__device__ __forceinline__ float feat_grad_from_feat_w(float f, bool elu, float thr, float w) {
    return elu ? fminf(f, w) : (f > thr ? w : 0.f);
}

// W (16 or 32) consecutive TMEM columns of the thread's lane into v; the caller's
// tmem_wait_regs<W>(v) orders every use of v after the load.
template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float *v) {
    static_assert(W == 16 || W == 32, "16 or 32 columns");
    if constexpr (W == 32)
        tmem_ld32(taddr, v);
    else
        tmem_ld16(taddr, v);
}

// z (fp32) into column d of a z tile as the rows (z_hi, z_lo, z_hi), z = z_hi + z_lo.
template <int D>
__device__ __forceinline__ void store_split_z(uint8_t *zt, int d, float z) {
    const __nv_bfloat16 zh = __float2bfloat16_rn(z);
    const __nv_bfloat16 zl = __float2bfloat16_rn(z - __bfloat162float(zh));
    *reinterpret_cast<__nv_bfloat16 *>(zt + swz_offset(16, 0, d)) = zh;
    *reinterpret_cast<__nv_bfloat16 *>(zt + swz_offset(16, 1, d)) = zl;
    *reinterpret_cast<__nv_bfloat16 *>(zt + swz_offset(16, 2, d)) = zh;
}

// One 16-column slice of an R row (bf16) into the swizzled R_bf tile (D rows, 128 columns).
template <int D>
__device__ __forceinline__ void store_rbf_row(uint8_t *rbf, int d, const float *v, int c16) {
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
    *reinterpret_cast<uint4 *>(rbf + swz_chunk(D, d, 2 * c16)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4 *>(rbf + swz_chunk(D, d, 2 * c16 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Eight dq values from eight phi_s = phi(q) / den (bf16) and the matching den * da (fp32):
// dq = phi'(q) / den * (den da), with phi'(q) / den = min(phi_s, 1 / den) for elu+1
// (phi' = min(phi, 1)), 1 / den where phi_s > 0 for relu and 1 / den for identity.
template <int PHI>
__device__ __forceinline__ uint4 dq_piece(uint4 u, const float *x, float inv) {
    const uint32_t *ui = reinterpret_cast<const uint32_t *>(&u);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = unpack_bf16x2(ui[q]);
        const float m0 = PHI == LA_PHI_ELU1 ? fminf(f.x, inv) : PHI == LA_PHI_IDENTITY ? inv : (f.x > 0.f ? inv : 0.f);
        const float m1 = PHI == LA_PHI_ELU1 ? fminf(f.y, inv) : PHI == LA_PHI_IDENTITY ? inv : (f.y > 0.f ? inv : 0.f);
        w[q] = pack_bf16x2(m0 * x[2 * q], m1 * x[2 * q + 1]);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// dq_piece's eight values in float32 (the cos/sin passes add the two terms before rounding);
// with position weights, inv = w / den: the feature is w phi(q), whose derivative is w phi'(q),
// and min(phi_s, w / den) = w min(phi, 1) / den for elu+1.
template <int PHI>
__device__ __forceinline__ void dq_vals(uint4 u, const float *x, float inv, float *o) {
    const uint32_t *ui = reinterpret_cast<const uint32_t *>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = unpack_bf16x2(ui[q]);
        const float m0 = PHI == LA_PHI_ELU1 ? fminf(f.x, inv) : PHI == LA_PHI_IDENTITY ? inv : (f.x > 0.f ? inv : 0.f);
        const float m1 = PHI == LA_PHI_ELU1 ? fminf(f.y, inv) : PHI == LA_PHI_IDENTITY ? inv : (f.y > 0.f ? inv : 0.f);
        o[2 * q] = m0 * x[2 * q];
        o[2 * q + 1] = m1 * x[2 * q + 1];
    }
}

// ---------------------------------------------------------------------------------------
// MASK: the group has fewer heads (n_rep) than the tile's G; the rows past them are masked.
// WT: one of the two passes of the cos/sin-weighted backward (p.pass: 1 cos, 2 sin; see
// backward_two_pass): features w phi, h = -g . out given in p.gd, and dq summed over the passes.
template <int D, int G, bool CAUSAL, bool MASK, bool WT>
__global__ void __launch_bounds__(kDqThreads, 1) k_tc_bwd_dq(const __grid_constant__ CUtensorMap map_q,
                                                              const __grid_constant__ CUtensorMap map_k,
                                                              const __grid_constant__ CUtensorMap map_v,
                                                              const __grid_constant__ CUtensorMap map_g,
                                                              const __grid_constant__ CUtensorMap map_dq,
                                                              const __grid_constant__ CUtensorMap map_ps,
                                                              const __grid_constant__ CUtensorMap map_den, Params p) {
    using K = BwdCfg<D, G>;
    constexpr int C = K::C, NS = K::NS_DQ, STAGE = K::STAGE_DQ;
    constexpr int OFF_K = K::Q_BYTES, OFF_V = OFF_K + K::K_BYTES, OFF_G = OFF_V + K::V_BYTES;
    constexpr int OFF_DEN = OFF_G + K::G_BYTES;   // den + eps of the 128 rows (fp32)
    constexpr int HALF = D / 2;   // feature columns per pool half
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();
    LA_SPAN(2, 0);
    // rdone is per stage: the store warp waits for chunk k's r product, and a single barrier could
    // run two phases ahead of it (the next chunk's product may finish first)
    __shared__ uint64_t bar_fulla[NS], bar_fullg[NS], bar_ready[NS], bar_empty[NS], bar_dqready[NS][2], bar_rdone[NS];
    __shared__ uint64_t bar_mfull, bar_sfull, bar_gnready, bar_dqfull, bar_xfree, bar_sbf, bar_fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::DQ_SMEM;
    (void)sm_lo;
    (void)sm_hi;
    uint8_t *pbuf = stage0 + NS * STAGE;         // dP' (query rows x keys)
    uint8_t *sbf = pbuf + K::P_BYTES;            // S_bf [D][D]
    // z and h enter the products as two-term bf16 splits (v = v_hi + v_lo): the z tile holds
    // rows (z_hi, z_lo, z_hi) and the h tile rows (h_hi, h_hi, h_lo), so that one K = 16
    // product gives h_hi z_hi + h_hi z_lo + h_lo z_hi
    uint8_t *ztile = sbf + K::S_BYTES;           // two slots of 16 x D
    uint8_t *ones = ztile + 2 * K::Z_BYTES;      // 16 x C, row 0 = 1
    uint8_t *htile = ones + K::ONES_BYTES;       // 16 x 128 (query rows)
    float *xch = reinterpret_cast<float *>(htile + K::H_BYTES);   // [2][128] partial row dots

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;
    // the group's gr = n_rep heads fill rows [0, gr C) of the 128 MMA rows; with gr < G the
    // other rows are masked: their phi_s rows are zeros (feature map), their g rows zeros
    // (cleared here, never loaded, and the dq epilogue writes zeros back), so every product
    // over them adds nothing, and nothing is stored for them
    const int gr = MASK ? p.n_rep : G;
    const int bh0 = b * p.Hq + g * gr;
    const size_t seg_state = ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1));
    const float *state_head = p.state + (size_t)bg * p.nseg * (size_t)(D * (D + 1));   // segment 0's state
    constexpr int kJoin = CAUSAL ? kScanPrefix : kScanTotal;
    float *rstate = p.rstate + seg_state;

    fill_ones_tile(ones, C);
    for (int idx = threadIdx.x; idx < (2 * K::Z_BYTES + K::H_BYTES) / 16; idx += blockDim.x) {
        uint8_t *t = idx < 2 * K::Z_BYTES / 16 ? ztile + idx * 16 : htile + (idx - 2 * K::Z_BYTES / 16) * 16;
        *reinterpret_cast<uint4 *>(t) = make_uint4(0u, 0u, 0u, 0u);
    }
    if constexpr (MASK) {
        if (gr < G) {   // the masked g rows of every stage: NS stages x DB blocks x (128 - gr C) rows
            const int mrows = 128 - gr * C;
            for (int idx = threadIdx.x; idx < NS * K::DB * mrows * 8; idx += blockDim.x) {
                const int row = gr * C + (idx / 8) % mrows, blk = (idx / (8 * mrows)) % K::DB, s = idx / (8 * mrows * K::DB);
                *reinterpret_cast<uint4 *>(stage0 + s * STAGE + OFF_G + blk * 128 * 128 + row * 128 + (idx % 8) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    fence_proxy_async();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_fulla[s], 1);
            mbar_init(&bar_fullg[s], 1);
            mbar_init(&bar_ready[s], kDqPro);
            mbar_init(&bar_empty[s], 1);
            mbar_init(&bar_dqready[s][0], 128);
            mbar_init(&bar_dqready[s][1], 128);
            mbar_init(&bar_rdone[s], 1);
        }
        mbar_init(&bar_mfull, 1);
        mbar_init(&bar_sfull, 1);
        mbar_init(&bar_gnready, 256);
        mbar_init(&bar_dqfull, 1);
        mbar_init(&bar_xfree, 256);
        mbar_init(&bar_sbf, 256);
        mbar_init(&bar_fin, 1);
        fence_barrier_init();
        // the forward's record of what it was run on: a workspace that another call wrote is
        // reported through the device error word (la_get_status: LA_ERR_WORKSPACE)
        if (blockIdx.x == 0 && p.hdr) {
            const int want[kHdrWords] = {kHdrMagic, p.B, p.Hq, p.Hkv, p.N, p.D, p.causal, p.phi, p.P,
                                         __float_as_int(p.eps), p.nseg, p.chunk,
                                         (int)reinterpret_cast<uintptr_t>(p.q),
                                         (int)(reinterpret_cast<uintptr_t>(p.q) >> 32),
                                         (int)reinterpret_cast<uintptr_t>(p.k), (int)reinterpret_cast<uintptr_t>(p.v)};
            bool same = true;
            for (int w = 0; w < kHdrWords; ++w) same = same && p.hdr[w] == want[w];
            if (!same) atomicExch(p.err, kErrStaleWorkspace);
        }
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base + K::T_S, tA = tmem_base + K::T_A, tA2 = tmem_base + K::T_A2,
                   tX = tmem_base + K::T_X, tR = tmem_base + K::T_R;

    if (warp == 0) {
        // ---------------- TMA producer: K, Q, V and the rows' den (what the feature map and the
        // first products need) on one barrier, grad_out on another
        {   // the whole warp, one lane issuing
            const uint32_t bytes_a = (uint32_t)(gr * C * D * 2 + gr * C * 4) +
                                     (CAUSAL ? (uint32_t)(K::K_BYTES + K::V_BYTES) : 0u);
            const uint32_t bytes_g = (uint32_t)(gr * C * D * 2);
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (k >= NS && !warp_wait(&bar_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                uint8_t *st = stage0 + s * STAGE;
                const int c0 = t0 + k * C;
                if (!LA_CHECK(in_smem(st, STAGE, sm_lo, sm_hi) && c0 < p.N && gr <= G && bh0 + gr <= p.B * p.Hq, 301,
                              smem_u32(st) - sm_lo, c0))
                    break;
                LA_TL(k, 0);
                mbar_arrive_expect_tx_w(&bar_fulla[s], bytes_a);
                if (CAUSAL)
                    for (int blk = 0; blk < K::DB; ++blk)
                        tma_load_4d_w(st + OFF_K + blk * C * 128, &map_k, &bar_fulla[s], blk * 64, c0, g, b);
                for (int r = 0; r < gr; ++r) {
                    tma_load_2d_w(st + OFF_DEN + r * K::DPAD * 4, &map_den, &bar_fulla[s], c0, bh0 + r);
                    for (int blk = 0; blk < K::DB; ++blk)
                        tma_load_4d_w(st + blk * 128 * 128 + r * C * 128, &map_q, &bar_fulla[s], blk * 64, c0, g * gr + r, b);
                }
                if (CAUSAL)
                    for (int blk = 0; blk < K::DB; ++blk)
                        tma_load_4d_w(st + OFF_V + blk * C * 128, &map_v, &bar_fulla[s], blk * 64, c0, g, b);
                mbar_arrive_expect_tx_w(&bar_fullg[s], bytes_g);
                for (int r = 0; r < gr; ++r)
                    for (int blk = 0; blk < K::DB; ++blk)
                        tma_load_4d_w(st + OFF_G + blk * 128 * 128 + r * C * 128, &map_g, &bar_fullg[s], blk * 64, c0,
                                      g * gr + r, b);
                issued = k + 1;
            }
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k) {
                warp_drain(&bar_fulla[k % NS], (k / NS) & 1);
                warp_drain(&bar_fullg[k % NS], (k / NS) & 1);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer.  Iteration k finishes chunk k - 1 (X += dP' phi(K) + h z,
        // then r) and starts chunk k (A_s, X, dA', then R and the state update).  Products that
        // share an A operand are issued back to back so that A is read from shared memory once.
        {   // the whole warp, one lane issuing
            constexpr uint32_t idA = idesc_bf16(128, C, false, false);
            constexpr uint32_t idX = idesc_bf16(128, D, false, false);
            constexpr uint32_t idDK = idesc_bf16(128, D, false, true);
            constexpr uint32_t idHZ = idesc_bf16(128, D, true, true);
            constexpr uint32_t idR = idesc_bf16(128, D, true, true);
            constexpr uint32_t idR16 = idesc_bf16(128, 16, true, false);
            const uint32_t sbf_u = smem_u32(sbf), pb = smem_u32(pbuf), on = smem_u32(ones), ht = smem_u32(htile);
            for (int k = 0; k <= nchunk; ++k) {
                if (k > 0) {
                    const int kp = k - 1, sp = kp % NS;
                    if (!warp_wait(&bar_gnready, kp & 1, &abort_flag)) break;
                    LA_TL(kp, 5);
                    tc_fence_after();
                    const uint32_t qs = smem_u32(stage0 + sp * STAGE), ks_ = qs + OFF_K;
                    // X += dP' phi(K) + h z^T   (X becomes den * da)
                    const uint32_t zt = smem_u32(ztile + (CAUSAL ? (kp & 1) : 0) * K::Z_BYTES);
                    if (CAUSAL)
                        for (int kk = 0; kk < C / 16; ++kk)
                            mma_bf16_w(tX, desc_kmajor(pb, 128, 0, kk), desc_mnmajor(ks_, C, 0, kk), idDK, 1u);
                    mma_bf16_w(tX, desc_mnmajor(ht, 16, 0, 0), desc_mnmajor(zt, 16, 0, 0), idHZ, 1u);
                    mma_commit_w(&bar_dqfull);
                    // r += phi_s^T h  (phi_s = phi(Q) / den)
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        mma_bf16_w(tR + D, desc_mnmajor(qs, 128, 0, kk), desc_kmajor(ht, 16, 0, kk), idR16,
                                   (kp > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_w(&bar_rdone[sp]);
                }
                if (k == nchunk) break;
                const int s = k % NS;
                if (!warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) break;
                if (!warp_wait(&bar_fullg[s], (k / NS) & 1, &abort_flag)) break;
                if ((CAUSAL || k == 0) && !warp_wait(&bar_sbf, k & 1, &abort_flag)) break;
                LA_TL(k, 3);
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * STAGE), ks_ = qs + OFF_K, vs = qs + OFF_V, gs = qs + OFF_G;
                if (!LA_CHECK(qs >= sm_lo && qs + STAGE <= sm_hi && ht + K::H_BYTES <= sm_hi, 311, qs - sm_lo, k))
                    break;
                // A_s = phi_s phi(K)^T
                if (CAUSAL)
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16_w(tA, desc_kmajor(qs, 128, 0, kk), desc_kmajor(ks_, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                if (k > 0 && !warp_wait(&bar_xfree, (k - 1) & 1, &abort_flag)) break;
                LA_TL(k, 4);
                tc_fence_after();
                // X = g S_bf^T and dA' = g V^T share g
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ag = desc_kmajor(gs, 128, 0, kk);
                    if (CAUSAL) {
                        mma_bf16_fill_w(tX, ag, desc_kmajor(sbf_u, D, 0, kk), idX, kk > 0 ? 1u : 0u);
                        mma_bf16_lastuse_w(tA2, ag, desc_kmajor(vs, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                    } else {
                        mma_bf16_w(tX, ag, desc_kmajor(sbf_u, D, 0, kk), idX, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit_w(&bar_mfull);
                if (CAUSAL) {   // S += phi(K)^T V, z += phi(K)^T 1 (one read of phi(K)), after X has
                                // read S_bf; the state conversion for the next chunk waits for it
                    for (int kk = 0; kk < C / 16; ++kk) {
                        const uint64_t ak = desc_mnmajor(ks_, C, 0, kk);
                        mma_bf16_fill_w(tS, ak, desc_mnmajor(vs, C, 0, kk), idR, 1u);
                        mma_bf16_lastuse_w(tS + D, ak, desc_kmajor(on, 16, 0, kk), idR16, 1u);
                    }
                    mma_commit_w(&bar_sfull);
                }
                // R += phi_s^T g (= phi(Q)^T gn); done before this chunk's dqfull, after which the
                // dq epilogue writes over the g tile
                for (int kk = 0; kk < 128 / 16; ++kk)
                    mma_bf16_w(tR, desc_mnmajor(qs, 128, 0, kk), desc_mnmajor(gs, 128, 0, kk), idR,
                               (k > 0 || kk > 0) ? 1u : 0u);
                LA_TL(k, 6);
            }
            mma_commit_w(&bar_fin);
            warp_drain(&bar_fin, 0);
        }
    } else if (warp == 2) {
        // ---------------- stores.  Causal: phi_s = phi(q) / den, left in the Q tile by the
        // feature map, goes to the workspace for the dk/dv kernel.  Then each pool half leaves
        // its D/2 columns of dq over the g tile; TMA writes them out, and the stage is released
        // once the copies have read it and the chunk's last products (r) are done
        {   // the whole warp, one lane issuing
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                uint8_t *st = stage0 + s * STAGE;
                const int c0 = t0 + k * C;
                bool ok = true;
                if (CAUSAL) {
                    ok = warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag);
                    if (ok) {
                        for (int r = 0; r < gr; ++r)
                            for (int blk = 0; blk < K::DB; ++blk)
                                tma_store_3d_w(&map_ps, st + blk * 128 * 128 + r * C * 128, blk * 64, c0, bh0 + r);
                        bulk_commit();
                    }
                }
                // with D = 128 each half is one 64-column block and goes out on its own;
                // with D = 64 both halves share the block
                for (int hh = 0; hh < 2; ++hh) {
                    ok = ok && warp_wait(&bar_dqready[s][hh], (k / NS) & 1, &abort_flag);
                    if (!ok) break;
                    if (hh == 0) LA_TL(k, 13);
                    if ((K::DB == 2 || hh == 1) && !(WT && p.pass == 1)) {   // (cos pass: dq partials in fp32)
                        const int blk = K::DB == 2 ? hh : 0;
                        for (int r = 0; r < gr; ++r)
                            tma_store_3d_w(&map_dq, st + OFF_G + blk * 128 * 128 + r * C * 128, blk * 64, c0, bh0 + r);
                    }
                }
                if (ok) {
                    bulk_commit();
                    bulk_wait_read();
                    LA_TL(k, 14);
                }
                ok = ok && warp_wait(&bar_rdone[s], (k / NS) & 1, &abort_flag);
                mbar_arrive_w(&bar_empty[s]);
                if (!ok) break;
            }
            bulk_wait_all();
        }
    } else if ((warp >= 4 && warp < 8) || warp >= 16) {
        // ---------------- phi prologue, in place: phi_s = phi(q) / den on the Q tile (den from
        // the forward, in the stage) and phi(k) on the K tile; both warpgroups share every chunk
        // (16-byte pieces dealt round-robin)
        const int pi = warp >= 16 ? threadIdx.x - 384 : threadIdx.x - 128;   // 0 .. kDqPro - 1
        // thread pi owns 16-byte column piece c of rows r0, r0 + RPP, ...; RPP is a multiple
        // of 8, so the piece's swizzled position is the same in all of them
        constexpr int CPR = D / 8, RPP = kDqPro / CPR;
        static_assert(RPP % 8 == 0, "rows per pass");
        const int c = pi % CPR, r0 = pi / CPR;
        const uint32_t pos = (uint32_t)(((c & 7) ^ (r0 & 7)) << 4);
        const uint32_t offq = (uint32_t)(c >> 3) * 128u * 128u + pos, offk = (uint32_t)(c >> 3) * C * 128u + pos;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            ok = ok && warp_wait(&bar_fulla[s], (k / NS) & 1, &abort_flag);
            if (pi == 0) LA_TL(k, 1);
            if (ok) {
                uint8_t *st = stage0 + s * STAGE;
                const float *dent = reinterpret_cast<const float *>(st + OFF_DEN);
                const int c0 = t0 + k * C;
                const int nvalid = t1 - c0;   // tokens of this chunk inside the segment
                constexpr int NQ = (128 + RPP - 1) / RPP, NK = CAUSAL ? (C + RPP - 1) / RPP : 0;
                uint8_t *pp[NQ + NK + 1];
                bool pres[NQ + NK + 1], val[NQ + NK + 1];
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    const int row = r0 + n * RPP;
                    pp[n] = st + offq + row * 128;
                    pres[n] = row < 128 && LA_CHECK(in_smem(pp[n], 16, sm_lo, sm_hi), 321, smem_u32(pp[n]) - sm_lo, row);
                    val[n] = row < gr * C && row % C < nvalid;
                }
#pragma unroll
                for (int n = 0; n < NK; ++n) {
                    const int j = r0 + n * RPP;
                    pp[NQ + n] = st + OFF_K + offk + j * 128;
                    pres[NQ + n] = j < C && LA_CHECK(in_smem(pp[NQ + n], 16, sm_lo, sm_hi), 322, smem_u32(pp[NQ + n]) - sm_lo, j);
                    val[NQ + n] = j < nvalid;
                }
                if constexpr (WT) {   // w phi(q) / den and w phi(k), phi in float32
                    float sc[NQ + NK + 1];
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        const int row = r0 + n * RPP;
                        sc[n] = val[n] ? p.wrow[c0 + row % C] / dent[(row / C) * K::DPAD + row % C] : 0.f;
                    }
#pragma unroll
                    for (int n = 0; n < NK; ++n) sc[NQ + n] = val[NQ + n] ? p.wrow[c0 + r0 + n * RPP] : 0.f;
                    if (p.phi == LA_PHI_ELU1)
                        feat8_batch_scaled<LA_PHI_ELU1, NQ + NK>(pp, pres, val, sc);
                    else if (p.phi == LA_PHI_RELU)
                        feat8_batch_scaled<LA_PHI_RELU, NQ + NK>(pp, pres, val, sc);
                    else
                        feat8_batch_scaled<LA_PHI_IDENTITY, NQ + NK>(pp, pres, val, sc);
                } else {   // the Q pieces' rows r0 + n RPP, each divided by its den
                    if (p.phi == LA_PHI_ELU1)
                        feat8_batch_rowscale<LA_PHI_ELU1, NQ + NK, C, K::DPAD>(pp, pres, val, dent, r0, RPP, NQ);
                    else if (p.phi == LA_PHI_RELU)
                        feat8_batch_rowscale<LA_PHI_RELU, NQ + NK, C, K::DPAD>(pp, pres, val, dent, r0, RPP, NQ);
                    else
                        feat8_batch_rowscale<LA_PHI_IDENTITY, NQ + NK, C, K::DPAD>(pp, pres, val, dent, r0, RPP, NQ);
                }
                fence_proxy_async();
            }
            if (pi == 0) LA_TL(k, 2);
            mbar_arrive_warp(&bar_ready[s]);
            // ---- warps 16-23: S, z after chunk k -> operand tiles for chunk k + 1, in two
            // halves of D/2 columns (thread = TMEM lane), between this chunk's feature map and
            // the next one's
            if (CAUSAL && warp >= 16) {
                const int h = (warp - 16) / 4, wq = warp % 4, i = wq * 32 + lane;
                const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
                ok = ok && warp_wait(&bar_sfull, k & 1, &abort_flag);
                tc_fence_after();
                if (i == 0 && h == 0) LA_TL(k, 9);
                if (ok && wq * 32 < D) {
#pragma unroll
                    for (int c16 = 0; c16 < HALF / 16; ++c16) {
                        float v[16];
                        tmem_ld16(tS + lane_off + h * HALF + c16 * 16, v);
                        tmem_wait_regs<16>(v);
                        store_state_row<D>(sbf, i, v, (h * HALF) / 16 + c16);
                    }
                    if (h == 0) {
                        float zd = tmem_ld1(tS + lane_off + D);
                        tmem_wait_regs<1>(&zd);
                        store_split_z<D>(ztile + ((k + 1) & 1) * K::Z_BYTES, i, zd);
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                if (i == 0 && h == 0) LA_TL(k, 10);
                mbar_arrive_warp(&bar_sbf);
            }
        }
    } else if (warp >= 8 && warp < 16) {
        // ---------------- row pool: two warpgroups, thread = query row i (TMEM lane), each
        // half owning D/2 feature columns and every second 16-key piece of the chunk.  Per
        // chunk: row work (g . num / den, h, dP'), then dq.
        const int h = (warp - 8) / 4;
        const int wq = warp % 4;
        const int i = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int r = i / C, ti = i % C;
        const int bh = bh0 + r;
        // initial S, z of the segment: TMEM (causal) and the operand tiles (slot 0)
        if (wq * 32 < D) {
#pragma unroll 1
            for (int c16 = h * (HALF / 16); c16 < (h + 1) * (HALF / 16); ++c16) {
                float v[16];
                seg_state_load16<D>(state_head, seg, p.nseg, kJoin, p.scan_in_kernel, i, c16, v);
                if (CAUSAL) tmem_st16(tS + lane_off + c16 * 16, v);
                store_state_row<D>(sbf, i, v, c16);
            }
            if (h == 0) {
                float zv[16];
                zv[0] = seg_state_z<D>(state_head, seg, p.nseg, kJoin, p.scan_in_kernel, i);
#pragma unroll
                for (int e = 1; e < 16; ++e) zv[e] = 0.f;
                if (CAUSAL) tmem_st16(tS + lane_off + D, zv);
                store_split_z<D>(ztile, i, zv[0]);
            }
            if (CAUSAL) tmem_st_wait();
        }
        fence_proxy_async();
        tc_fence_before();
        if (i == 0 && h == 0) LA_TL(0, 15);   // the segment's starting S, z are in TMEM and S_bf
        mbar_arrive_warp(&bar_sbf);
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            const int t = t0 + k * C + ti;
            const bool valid = t < t1 && r < gr;
            uint8_t *st = stage0 + s * STAGE;
            // ---- row work: with phi_s = phi(q) / den and A_s = phi_s phi(K)^T,
            // g . num / den = phi_s . X + sum_j mask(A_s) dA';  h = -(g . num) / den;
            // dP' = mask(dA' + h)
            ok = ok && warp_wait(&bar_mfull, k & 1, &abort_flag);
            tc_fence_after();
            if (i == 0 && h == 0) LA_TL(k, 7);
            float hval = 0.f, inv = 0.f;
            if (WT && ok && valid) hval = p.gd[(size_t)bh * p.N + t];   // h = -g . out, given
            if (ok) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (CAUSAL && !WT) {
#pragma unroll 1
                    for (int c16 = 0; c16 < C / 16; ++c16) {
                        if ((c16 & 1) != h) continue;
                        float va[16], vd[16];
                        tmem_ld16(tA + lane_off + c16 * 16, va);
                        tmem_ld16(tA2 + lane_off + c16 * 16, vd);
                        tmem_wait_regs<16>(va);
                        tmem_wait_regs<16>(vd);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c16 * 16 + e <= ti) acc[e & 3] = fmaf(va[e], vd[e], acc[e & 3]);
                    }
                }
                // phi_s . X over this half's feature columns, XW at a time (one TMEM round trip each)
                constexpr int XW = HALF >= 32 ? 32 : 16;
#pragma unroll 1
                for (int cx = 0; cx < (WT ? 0 : HALF / XW); ++cx) {
                    const int col0 = h * HALF + cx * XW;
                    float xv[XW];
                    tmem_ld_cols<XW>(tX + lane_off + col0, xv);
                    uint4 u[XW / 8];
#pragma unroll
                    for (int q8 = 0; q8 < XW / 8; ++q8) u[q8] = *reinterpret_cast<const uint4 *>(st + swz_chunk(128, i, col0 / 8 + q8));
                    tmem_wait_regs<XW>(xv);
#pragma unroll
                    for (int q8 = 0; q8 < XW / 8; ++q8) {
                        const uint32_t *ui = reinterpret_cast<const uint32_t *>(&u[q8]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = unpack_bf16x2(ui[q]);
                            acc[q] = fmaf(f.x, xv[q8 * 8 + 2 * q], acc[q]);
                            acc[q] = fmaf(f.y, xv[q8 * 8 + 2 * q + 1], acc[q]);
                        }
                    }
                }
                xch[h * 128 + i] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                // (masked rows: 0, so that their dq is zeros, which keeps their g rows zero; with
                // weights w / den, for rows inside the sequence)
                if constexpr (WT)
                    inv = valid ? p.wrow[t] / reinterpret_cast<const float *>(st + OFF_DEN)[r * K::DPAD + ti] : 0.f;
                else
                    inv = r < gr ? 1.f / reinterpret_cast<const float *>(st + OFF_DEN)[r * K::DPAD + ti] : 0.f;
            }
            named_barrier(3, 256);
            if (ok) {
                if (!WT) {
                    const float gnum = xch[i] + xch[128 + i];   // g . num / den
                    hval = valid ? -gnum : 0.f;
                }
                if (CAUSAL)
                    for (int c16 = h; c16 < C / 16; c16 += 2) {
                        float vd[16];
                        tmem_ld16(tA2 + lane_off + c16 * 16, vd);
                        tmem_wait_regs<16>(vd);
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const int j = c16 * 16 + e;
                            w[e / 2] = pack_bf16x2((j <= ti) ? vd[e] + hval : 0.f, (j + 1 <= ti) ? vd[e + 1] + hval : 0.f);
                        }
                        uint8_t *p0 = pbuf + swz_chunk(128, i, 2 * c16), *p1 = pbuf + swz_chunk(128, i, 2 * c16 + 1);
                        if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi), 335,
                                     smem_u32(p0) - sm_lo, c16)) {
                            *reinterpret_cast<uint4 *>(p0) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4 *>(p1) = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                if (h == 0) {
                    const __nv_bfloat16 hh = __float2bfloat16_rn(hval);
                    const __nv_bfloat16 hl = __float2bfloat16_rn(hval - __bfloat162float(hh));
                    *reinterpret_cast<__nv_bfloat16 *>(htile + swz_offset(16, 0, i)) = hh;
                    *reinterpret_cast<__nv_bfloat16 *>(htile + swz_offset(16, 1, i)) = hh;
                    *reinterpret_cast<__nv_bfloat16 *>(htile + swz_offset(16, 2, i)) = hl;
                    if (!WT && valid && LA_CHECK((size_t)bh * p.N + t < (size_t)p.B * p.Hq * p.N, 334, bh, t))
                        p.gd[(size_t)bh * p.N + t] = hval;   // h = den * gd for the dk/dv kernel
                }
                fence_proxy_async();
            }
            tc_fence_before();
            if (i == 0 && h == 0) LA_TL(k, 8);
            mbar_arrive_warp(&bar_gnready);
            // ---- dq = phi'(q) / den * (den da), written over the g tile (its last reader, the R
            // product, is done before dqfull) for the TMA store
            ok = ok && warp_wait(&bar_dqfull, k & 1, &abort_flag);
            tc_fence_after();
            if (i == 0 && h == 0) LA_TL(k, 11);
            // 16 columns of X per TMEM round trip: 32 here (as in the row pass) spilled registers
            // and made the long-context step 3 % slower
            constexpr int XE = 16;
#pragma unroll 1
            for (int cx = 0; cx < HALF / XE; ++cx) {
                const int col0 = h * HALF + cx * XE;
                float xv[XE];
                if (ok) tmem_ld_cols<XE>(tX + lane_off + col0, xv);
                uint8_t *ch[XE / 8];
                uint4 u[XE / 8];
#pragma unroll
                for (int q8 = 0; q8 < XE / 8; ++q8) {   // every load before any store
                    ch[q8] = st + swz_chunk(128, i, col0 / 8 + q8);
                    u[q8] = *reinterpret_cast<const uint4 *>(ch[q8]);
                }
                if (ok) tmem_wait_regs<XE>(xv);
                if (cx + 1 == HALF / XE) {   // every column of X is in registers
                    tc_fence_before();
                    mbar_arrive_warp(&bar_xfree);
                }
                if (!ok) continue;
                if constexpr (WT) {   // cos pass: dq terms (fp32) to the workspace, chunk-blocked (a
                                      // warp's rows form one run per column); sin pass: plus those
                    if (p.pass == 2 && cx == 0 && h == 0 && i == 0 && k + 1 < nchunk)   // the next chunk's block
                        for (int r2 = 0; r2 < gr; ++r2)                                 // of them into L2
                            prefetch_l2_bulk(p.part_dq + blocked_index(bh0 + r2, t0 + (k + 1) * C, 0, p.N, D, C),
                                             (uint32_t)(D * C * 4));
                    float *pq = p.part_dq + (valid ? blocked_index(bh, t, col0, p.N, D, C) : 0);
                    float prev[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) prev[e] = p.pass == 2 && valid ? __ldg(pq + (size_t)e * C) : 0.f;
#pragma unroll
                    for (int q8 = 0; q8 < 2; ++q8) {
                        float o[8];
                        if (p.phi == LA_PHI_ELU1)
                            dq_vals<LA_PHI_ELU1>(u[q8], xv + q8 * 8, inv, o);
                        else if (p.phi == LA_PHI_RELU)
                            dq_vals<LA_PHI_RELU>(u[q8], xv + q8 * 8, inv, o);
                        else
                            dq_vals<LA_PHI_IDENTITY>(u[q8], xv + q8 * 8, inv, o);
                        if (p.pass == 1) {
                            if (valid)
#pragma unroll
                                for (int e = 0; e < 8; ++e) pq[(size_t)(q8 * 8 + e) * C] = o[e];
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[e] += prev[q8 * 8 + e];
                            if (LA_CHECK(in_smem(ch[q8] + OFF_G, 16, sm_lo, sm_hi), 342, smem_u32(ch[q8]) - sm_lo, q8))
                                *reinterpret_cast<uint4 *>(ch[q8] + OFF_G) =
                                    make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                               pack_bf16x2(o[6], o[7]));
                        }
                    }
                } else {
#pragma unroll
                    for (int q8 = 0; q8 < XE / 8; ++q8)
                        if (LA_CHECK(in_smem(ch[q8] + OFF_G, 16, sm_lo, sm_hi), 341, smem_u32(ch[q8]) - sm_lo, q8))
                            *reinterpret_cast<uint4 *>(ch[q8] + OFF_G) =
                                p.phi == LA_PHI_ELU1   ? dq_piece<LA_PHI_ELU1>(u[q8], xv + q8 * 8, inv)
                                : p.phi == LA_PHI_RELU ? dq_piece<LA_PHI_RELU>(u[q8], xv + q8 * 8, inv)
                                                       : dq_piece<LA_PHI_IDENTITY>(u[q8], xv + q8 * 8, inv);
                }
            }
            fence_proxy_async();
            if (i == 0 && h == 0) LA_TL(k, 12);
            mbar_arrive_warp(&bar_dqready[s][h]);
        }
        // the segment's R, r -> workspace
        ok = ok && warp_wait(&bar_fin, 0, &abort_flag);
        tc_fence_after();
        if (ok && wq * 32 < D) {
#pragma unroll 1
            for (int c16 = h * (HALF / 16); c16 < (h + 1) * (HALF / 16); ++c16) {
                float v[16];
                tmem_ld16(tR + lane_off + c16 * 16, v);
                tmem_wait_regs<16>(v);
                state_store16<D>(rstate, i, c16, v);
            }
            if (h == 0) {
                float rd[16];   // r = phi_s^T h_hi (column 0) + phi_s^T h_lo (column 2)
                tmem_ld16(tR + lane_off + D, rd);
                tmem_wait_regs<16>(rd);
                state_store_z<D>(rstate, i, rd[0] + rd[2]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (threadIdx.x == 0 && abort_flag) atomicExch(p.err, kErrTimeout);
    LA_SPAN(2, 1);
}

// ---------------------------------------------------------------------------------------
template <int D, int G, bool CAUSAL, bool MASK, bool WT>
__global__ void __launch_bounds__(kKvThreads, 1) k_tc_bwd_dkdv(const __grid_constant__ CUtensorMap map_q,
                                                                const __grid_constant__ CUtensorMap map_k,
                                                                const __grid_constant__ CUtensorMap map_v,
                                                                const __grid_constant__ CUtensorMap map_g,
                                                                const __grid_constant__ CUtensorMap map_dk,
                                                                const __grid_constant__ CUtensorMap map_dv, Params p) {
    using K = BwdCfg<D, G>;
    constexpr int C = K::C, NS = K::NS, NB = K::NB_KV;
    constexpr int OFF_K = K::Q_BYTES, OFF_V = OFF_K + K::K_BYTES, OFF_G = OFF_V + K::V_BYTES;
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();
    LA_SPAN(3, 0);
    // each stage is two regions: [Q | g] (free once the chunk's products are done) and
    // [K | V] (dk is written over phi(K) and dv over V, and the region is free once the TMA
    // stores of dk and dv have read it)
    __shared__ uint64_t bar_fullq[NS], bar_fullg[NS], bar_fullkv[NS], bar_ready[NS], bar_emptyqg[NS],
        bar_emptykv[NS], bar_dkready[NS], bar_dvready[NS];
    __shared__ uint64_t bar_afull[2], bar_outfull[2], bar_outfree[2];
    __shared__ uint64_t bar_pready, bar_rbf, bar_rfull, bar_stfree, bar_fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::DKDV_SMEM;
    (void)sm_lo;
    (void)sm_hi;
    uint8_t *ptbuf = stage0 + NS * K::STAGE;     // P'^T = mask(phi_s phi(K)^T)^T  [keys][query rows]
    uint8_t *dpbuf = ptbuf + K::PT_BYTES;        // dP' = mask(g V^T + h), then h  [query rows][keys | h_hi h_lo]
    uint8_t *rbf = dpbuf + K::P_BYTES;           // R_bf [D rows d][128 columns e]
    uint8_t *htile = rbf + K::RBF_BYTES;         // h as 16 x 128 (rows h_hi, h_lo) when it is not in dP'
    uint8_t *obuf = htile + (K::H_IN_DP ? 0 : K::H_BYTES);   // dk, then dv [keys][D] (OUT_STAGE)
    constexpr bool OUT_STAGE = K::OUT_STAGE;
    constexpr bool PSPLIT = CAUSAL && C / 16 >= 2;   // two warpgroups convert P' and dP'
    // DVSPLIT: the dv epilogue runs on warps 20-23 beside the dk epilogue on warps 8-11 (and the
    // feature map of K on warps 16-19 only).  With C > 32 (one buffer of TMEM outputs, outputs
    // written over phi(K) and V) the two epilogues are the tail of a chain that the next
    // chunk's products wait for: the TMEM buffer is free once both have read it.
    constexpr bool DVSPLIT = !OUT_STAGE && !WT;
    constexpr int KVPRO = DVSPLIT ? kKvPro / 2 : kKvPro;   // feature-map threads

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;
    // rows of masked heads (gr < G; see k_tc_bwd_dq): zero phi_s and g rows, never loaded, and
    // a zero h, so that they add nothing to dk, dv, R or r
    const int gr = MASK ? p.n_rep : G;
    const int bh0 = b * p.Hq + g * gr;
    const float *rstate_head = p.rstate + (size_t)bg * p.nseg * (size_t)(D * (D + 1));   // segment 0's R
    constexpr int kJoinR = CAUSAL ? kScanSuffix : kScanTotal;

    for (int idx = threadIdx.x; idx < (K::P_BYTES + (K::H_IN_DP ? 0 : K::H_BYTES)) / 16; idx += blockDim.x) {
        uint8_t *t = idx < K::P_BYTES / 16 ? dpbuf + idx * 16 : htile + (idx - K::P_BYTES / 16) * 16;
        *reinterpret_cast<uint4 *>(t) = make_uint4(0u, 0u, 0u, 0u);
    }
    if constexpr (MASK) {
        if (gr < G) {   // NS stages x {phi_s, g} x DB blocks x (128 - gr C) rows
            const int mrows = 128 - gr * C;
            for (int idx = threadIdx.x; idx < NS * 2 * K::DB * mrows * 8; idx += blockDim.x) {
                const int row = gr * C + (idx / 8) % mrows, blk = (idx / (8 * mrows)) % K::DB;
                const int which = (idx / (8 * mrows * K::DB)) % 2, s = idx / (8 * mrows * K::DB * 2);
                *reinterpret_cast<uint4 *>(stage0 + s * K::STAGE + (which ? OFF_G : 0) + blk * 128 * 128 + row * 128 +
                                           (idx % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    fence_proxy_async();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_fullq[s], 1);
            mbar_init(&bar_fullg[s], 1);
            mbar_init(&bar_fullkv[s], 1);
            mbar_init(&bar_ready[s], KVPRO);
            mbar_init(&bar_emptyqg[s], 1);
            mbar_init(&bar_emptykv[s], OUT_STAGE ? 128 : 1);
            mbar_init(&bar_dkready[s], 128);
            mbar_init(&bar_dvready[s], 128);
        }
        mbar_init(&bar_afull[0], 1);
        mbar_init(&bar_afull[1], 1);
        mbar_init(&bar_pready, PSPLIT ? 256 : 128);
        for (int bb = 0; bb < 2; ++bb) {
            mbar_init(&bar_outfull[bb], 1);
            mbar_init(&bar_outfree[bb], DVSPLIT ? 256 : 128);
        }
        mbar_init(&bar_rbf, 128);
        mbar_init(&bar_rfull, 1);
        mbar_init(&bar_stfree, 1);
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
    // TMEM: R, then per buffer bb the scores A_s (tA), dA' (tD), the outputs dk^T (tK), dv^T
    // (tV) and the r part phi_s^T [h_hi h_lo] (tRp, two of 16 columns).  With KV_SEP the
    // outputs have columns of their own and tRp follows dk^T; otherwise dk^T overwrites A_s
    // and dv^T overwrites dA'.
    constexpr bool SEP = K::KV_SEP, MERGE_H = K::MERGE_H;
    const uint32_t tR = tmem_base + K::KT_R;
    auto tBuf = [=](int bb) { return tmem_base + (uint32_t)(K::KT_AD + bb * K::KV_BW); };
    auto tA = [=](int bb) { return tBuf(bb); };
    auto tD = [=](int bb) { return tBuf(bb) + (uint32_t)C; };
    auto tK = [=](int bb) { return tBuf(bb) + (uint32_t)(SEP ? 2 * C : 0); };
    auto tRp = [=](int bb) { return tBuf(bb) + (uint32_t)(SEP ? 3 * C : 2 * C); };
    auto tV = [=](int bb) { return tBuf(bb) + (uint32_t)(SEP ? 3 * C + 16 : C); };

    if (warp == 0) {
        // ---------------- TMA producer (chunks in reverse order)
        {   // the whole warp, one lane issuing
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + (nchunk - 1 - k) * C;
                if (!LA_CHECK(in_smem(st, K::STAGE, sm_lo, sm_hi) && c0 < p.N && gr <= G && bh0 + gr <= p.B * p.Hq, 401,
                              smem_u32(st) - sm_lo, c0))
                    break;
                if (CAUSAL && k >= NS && !warp_wait(&bar_emptyqg[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                LA_TL2(k, 0);
                if (CAUSAL) {
                    mbar_arrive_expect_tx_w(&bar_fullq[s], (uint32_t)(gr * C * D * 2));
                    for (int r = 0; r < gr; ++r)
                        for (int blk = 0; blk < K::DB; ++blk)
                            tma_load_4d_w(st + blk * 128 * 128 + r * C * 128, &map_q, &bar_fullq[s], blk * 64, c0,
                                        g * gr + r, b);
                    mbar_arrive_expect_tx_w(&bar_fullg[s], (uint32_t)(gr * C * D * 2));
                    for (int r = 0; r < gr; ++r)
                        for (int blk = 0; blk < K::DB; ++blk)
                            tma_load_4d_w(st + OFF_G + blk * 128 * 128 + r * C * 128, &map_g, &bar_fullg[s], blk * 64,
                                        c0, g * gr + r, b);
                }
                if (k >= NS && !warp_wait(&bar_emptykv[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                mbar_arrive_expect_tx_w(&bar_fullkv[s], K::K_BYTES + K::V_BYTES);
                for (int blk = 0; blk < K::DB; ++blk) {
                    tma_load_4d_w(st + OFF_K + blk * C * 128, &map_k, &bar_fullkv[s], blk * 64, c0, g, b);
                    tma_load_4d_w(st + OFF_V + blk * C * 128, &map_v, &bar_fullkv[s], blk * 64, c0, g, b);
                }
                issued = k + 1;
            }
            // a chunk whose K, V wait gave up has Q and g in flight: wait for those too
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k) {
                if (CAUSAL) {
                    warp_drain(&bar_fullq[k % NS], (k / NS) & 1);
                    warp_drain(&bar_fullg[k % NS], (k / NS) & 1);
                }
                warp_drain(&bar_fullkv[k % NS], (k / NS) & 1);
            }
            if (issued < nchunk && CAUSAL) {
                const int k = issued;
                warp_drain(&bar_fullq[k % NS], (k / NS) & 1);
                warp_drain(&bar_fullg[k % NS], (k / NS) & 1);
            }
        }
    } else if (warp == 2) {
        // ---------------- dk, dv stores.  With OUT_STAGE both go out of the staging tile,
        // dk first, and each copy frees the tile for the next output; otherwise TMA writes the
        // two tiles left over phi(K) and V, and the [K | V] region is released once the copies
        // have read it
        {   // the whole warp, one lane issuing
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                uint8_t *st = stage0 + s * K::STAGE;
                uint8_t *src_k = OUT_STAGE ? obuf : st + OFF_K, *src_v = OUT_STAGE ? obuf : st + OFF_V;
                const int c0 = t0 + (nchunk - 1 - k) * C;
                bool ok = warp_wait(&bar_dkready[s], (k / NS) & 1, &abort_flag);
                const bool store = !(WT && p.pass == 1);   // cos pass: dk, dv partials in fp32
                if (ok && store) {
                    LA_TL2(k, 12);
                    for (int blk = 0; blk < K::DB; ++blk) tma_store_3d_w(&map_dk, src_k + blk * C * 128, blk * 64, c0, bg);
                    bulk_commit();
                }
                if (OUT_STAGE) {
                    bulk_wait_read();
                    mbar_arrive_w(&bar_stfree);
                }
                ok = ok && warp_wait(&bar_dvready[s], (k / NS) & 1, &abort_flag);
                if (ok && store) {
                    for (int blk = 0; blk < K::DB; ++blk) tma_store_3d_w(&map_dv, src_v + blk * C * 128, blk * 64, c0, bg);
                    bulk_commit();
                }
                bulk_wait_read();
                if (ok) LA_TL2(k, 13);
                mbar_arrive_w(OUT_STAGE ? &bar_stfree : &bar_emptykv[s]);
                if (!ok) break;
            }
            bulk_wait_all();
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer.  Per chunk k: start (A_s, dA'; causal), the R part
        // (dk^T = R_bf V^T, dv^T = R_bf^T phi(K)^T and R += phi_s^T g, none of which needs P'),
        // which the tensor pipe works on while the pool converts P' and dP', then the finish
        // (dk^T += phi_s^T [dP' | h], dv^T += g^T P').  With two buffers, chunk k + 1's start
        // goes before chunk k's finish when its inputs are already there.  Without KV_SEP the
        // outputs share columns with A_s and dA', and the whole chunk runs after P' (finish_alias).
        {   // the whole warp, one lane issuing
            constexpr uint32_t idA = idesc_bf16(128, C, false, false);
            constexpr uint32_t idMM = idesc_bf16(128, C, true, true);
            constexpr uint32_t idMH = idesc_bf16(128, MERGE_H ? C + 16 : C, true, true);
            constexpr uint32_t idMK = idesc_bf16(128, C, true, false);
            constexpr uint32_t idR = idesc_bf16(128, D, true, true);
            constexpr uint32_t idH = idesc_bf16(128, 16, true, K::H_IN_DP);
            const uint32_t pb = smem_u32(ptbuf), dpb = smem_u32(dpbuf), rb = smem_u32(rbf), ht = smem_u32(htile);
            auto stage_ok = [&](uint32_t qs, int k) {
                return LA_CHECK(qs >= sm_lo && qs + K::STAGE <= sm_hi && rb + K::RBF_BYTES <= sm_hi, 411, qs - sm_lo, k);
            };
            auto start = [&](int k) -> bool {
                const int s = k % NS, bb = k % NB;
                if (!warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) return false;
                if (!warp_wait(&bar_fullq[s], (k / NS) & 1, &abort_flag)) return false;
                if (!warp_wait(&bar_fullg[s], (k / NS) & 1, &abort_flag)) return false;
                // sharing columns, A_s and dA' overwrite dk^T and dv^T of chunk k - NB
                if (!SEP && k >= NB && !warp_wait(&bar_outfree[bb], ((k - NB) / NB) & 1, &abort_flag)) return false;
                LA_TL2(k, 3);
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), ks_ = qs + OFF_K, vs = qs + OFF_V, gs = qs + OFF_G;
                if (!stage_ok(qs, k)) return false;
                for (int kk = 0; kk < D / 16; ++kk)   // A_s = phi_s phi(K)^T
                    mma_bf16_w(tA(bb), desc_kmajor(qs, 128, 0, kk), desc_kmajor(ks_, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                for (int kk = 0; kk < D / 16; ++kk)   // dA' = g V^T
                    mma_bf16_w(tD(bb), desc_kmajor(gs, 128, 0, kk), desc_kmajor(vs, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                mma_commit_w(&bar_afull[bb]);
                LA_TL2(k, 4);
                return true;
            };
            // dk^T (+)= R_bf V^T, dv^T (+)= R_bf^T phi(K)^T
            auto rbf_terms = [&](uint32_t qs, int bb, uint32_t acc_k, uint32_t acc_v) {
                const uint32_t ks_ = qs + OFF_K, vs = qs + OFF_V;
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_w(tK(bb), desc_kmajor(rb, D, 0, kk), desc_kmajor(vs, C, 0, kk), idA, kk > 0 ? 1u : acc_k);
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_w(tV(bb), desc_mnmajor(rb, D, 0, kk), desc_kmajor(ks_, C, 0, kk), idMK, kk > 0 ? 1u : acc_v);
            };
            // R += phi_s^T g
            auto r_update = [&](uint32_t qs) {
                for (int kk = 0; kk < 128 / 16; ++kk)
                    mma_bf16_w(tR, desc_mnmajor(qs, 128, 0, kk), desc_mnmajor(qs + OFF_G, 128, 0, kk), idR, 1u);
            };
            auto rpart = [&](int k) -> bool {
                const int s = k % NS, bb = k % NB;
                if ((CAUSAL || k == 0) && !warp_wait(&bar_rbf, k & 1, &abort_flag)) return false;
                if (!CAUSAL && !warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) return false;
                if (k >= NB && !warp_wait(&bar_outfree[bb], ((k - NB) / NB) & 1, &abort_flag)) return false;
                LA_TL2(k, 14);
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE);
                if (!stage_ok(qs, k)) return false;
                rbf_terms(qs, bb, 0u, 0u);
                if (CAUSAL) {
                    r_update(qs);
                    mma_commit_w(&bar_rfull);
                } else {
                    mma_commit_w(&bar_outfull[bb]);
                }
                return true;
            };
            auto finish = [&](int k) -> bool {   // causal, KV_SEP
                const int s = k % NS, bb = k % NB;
                if (!warp_wait(&bar_pready, k & 1, &abort_flag)) return false;
                LA_TL2(k, 5);
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), gs = qs + OFF_G;
                if (!stage_ok(qs, k)) return false;
                for (int kk = 0; kk < 128 / 16; ++kk) {   // dk^T += phi_s^T dP', r part = phi_s^T h
                    const uint64_t as = desc_mnmajor(qs, 128, 0, kk);
                    mma_bf16_w(tK(bb), as, desc_mnmajor(dpb, 128, 0, kk), idMH, 1u);
                    if (!MERGE_H)
                        mma_bf16_w(tRp(bb), as, K::H_IN_DP ? desc_mnmajor(dpb + C * 2, 128, 0, kk) : desc_kmajor(ht, 16, 0, kk),
                                 idH, kk > 0 ? 1u : 0u);
                }
                for (int kk = 0; kk < 128 / 16; ++kk)   // dv^T += g^T P'
                    mma_bf16_w(tV(bb), desc_mnmajor(gs, 128, 0, kk), desc_kmajor(pb, C, 0, kk), idMK, 1u);
                mma_commit_w(&bar_outfull[bb]);
                mma_commit_w(&bar_emptyqg[s]);
                LA_TL2(k, 6);
                return true;
            };
            auto finish_alias = [&](int k) -> bool {   // !KV_SEP: everything after P' (one buffer)
                const int s = k % NS, bb = k % NB;
                if (CAUSAL && !warp_wait(&bar_pready, k & 1, &abort_flag)) return false;
                if ((CAUSAL || k == 0) && !warp_wait(&bar_rbf, k & 1, &abort_flag)) return false;
                if (!CAUSAL) {
                    if (!warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) return false;
                    if (k >= NB && !warp_wait(&bar_outfree[bb], ((k - NB) / NB) & 1, &abort_flag)) return false;
                }
                LA_TL2(k, 5);
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), gs = qs + OFF_G;
                if (!stage_ok(qs, k)) return false;
                if (CAUSAL) {
                    for (int kk = 0; kk < 128 / 16; ++kk) {   // dk^T = phi_s^T dP', r part = phi_s^T h
                        const uint64_t as = desc_mnmajor(qs, 128, 0, kk);
                        mma_bf16_w(tK(bb), as, desc_mnmajor(dpb, 128, 0, kk), idMM, kk > 0 ? 1u : 0u);
                        mma_bf16_w(tRp(bb), as, K::H_IN_DP ? desc_mnmajor(dpb + C * 2, 128, 0, kk) : desc_kmajor(ht, 16, 0, kk),
                                 idH, kk > 0 ? 1u : 0u);
                    }
                    r_update(qs);
                    for (int kk = 0; kk < 128 / 16; ++kk)   // dv^T = g^T P'
                        mma_bf16_w(tV(bb), desc_mnmajor(gs, 128, 0, kk), desc_kmajor(pb, C, 0, kk), idMK, kk > 0 ? 1u : 0u);
                }
                rbf_terms(qs, bb, CAUSAL ? 1u : 0u, CAUSAL ? 1u : 0u);
                mma_commit_w(&bar_outfull[bb]);
                if (CAUSAL) {
                    mma_commit_w(&bar_rfull);
                    mma_commit_w(&bar_emptyqg[s]);
                }
                LA_TL2(k, 6);
                return true;
            };
            if (SEP) {
                int started = -1;
                bool okm = true;
                if (CAUSAL && nchunk > 0) {
                    okm = start(0);
                    started = 0;
                }
                for (int k = 0; okm && k < nchunk; ++k) {
                    if (!rpart(k)) break;
                    const int kn = k + 1, sn = kn % NS;
                    if (CAUSAL && NB == 2 && kn < nchunk && warp_test(&bar_ready[sn], (kn / NS) & 1) &&
                        warp_test(&bar_fullq[sn], (kn / NS) & 1) && warp_test(&bar_fullg[sn], (kn / NS) & 1)) {
                        if (!start(kn)) break;
                        started = kn;
                    }
                    if (CAUSAL && !finish(k)) break;
                    if (CAUSAL && kn < nchunk && started < kn) {
                        if (!start(kn)) break;
                        started = kn;
                    }
                }
            } else {
                for (int k = 0; k < nchunk; ++k) {
                    if (CAUSAL && !start(k)) break;
                    if (!finish_alias(k)) break;
                }
            }
            mma_commit_w(&bar_fin);
            warp_drain(&bar_fin, 0);
        }
    } else if (DVSPLIT && warp >= 20) {
        // ---------------- warps 20-23 (thread = value column e = d): dv = row e of dv^T, written
        // over V for the TMA store, beside warps 8-11's dk
        const int wq = warp % 4;
        const int d = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS, bb = k % NB;
            ok = ok && warp_wait(&bar_outfull[bb], (k / NB) & 1, &abort_flag);
            tc_fence_after();
            uint8_t *vw = stage0 + s * K::STAGE + OFF_V;
#pragma unroll 1
            for (int c16 = 0; c16 < C / 16; ++c16) {
                float v[16];
                if (ok && d < D) {
                    tmem_ld16(tV(bb) + lane_off + c16 * 16, v);
                    tmem_wait_regs<16>(v);
                }
                if (c16 + 1 == C / 16) {
                    tc_fence_before();
                    mbar_arrive_warp(&bar_outfree[bb]);
                }
                if (!ok || d >= D) continue;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    *reinterpret_cast<__nv_bfloat16 *>(vw + swz_offset(C, c16 * 16 + e, d)) = __float2bfloat16_rn(v[e]);
            }
            fence_proxy_async();
            mbar_arrive_warp(&bar_dvready[s]);
        }
    } else if (warp >= 16) {
        // ---------------- prologue (warps 16-23, or 16-19 with DVSPLIT, on every chunk): phi(K)
        // over the K tile, in place (the Q tile arrives as phi_s = phi(q) / den, written by the
        // dq kernel)
        const int pi = threadIdx.x - 512;   // 0 .. KVPRO - 1
        constexpr int CPR = D / 8, RPP = KVPRO / CPR;
        static_assert(RPP % 8 == 0, "rows per pass");
        const int c = pi % CPR, r0 = pi / CPR;
        const uint32_t pos = (uint32_t)(((c & 7) ^ (r0 & 7)) << 4);
        const uint32_t offk = (uint32_t)(c >> 3) * C * 128u + pos;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            const int c0 = t0 + (nchunk - 1 - k) * C;
            const int nvalid = t1 - c0;
            uint8_t *st = stage0 + s * K::STAGE;
            ok = ok && warp_wait(&bar_fullkv[s], (k / NS) & 1, &abort_flag);
            if (pi == 0) LA_TL2(k, 1);
            if (ok) {
                constexpr int NK = (C + RPP - 1) / RPP;
                uint8_t *pp[NK];
                bool pres[NK], val[NK];
#pragma unroll
                for (int n = 0; n < NK; ++n) {
                    const int j = r0 + n * RPP;
                    pp[n] = st + OFF_K + offk + (j < C ? j : 0) * 128;
                    pres[n] = j < C && LA_CHECK(in_smem(pp[n], 16, sm_lo, sm_hi), 422, smem_u32(pp[n]) - sm_lo, j);
                    val[n] = j < nvalid;
                }
                if constexpr (WT) {   // w phi(k), phi in float32
                    float sc[NK];
#pragma unroll
                    for (int n = 0; n < NK; ++n) sc[n] = pres[n] && val[n] ? p.wrow[c0 + r0 + n * RPP] : 0.f;
                    if (p.phi == LA_PHI_ELU1)
                        feat8_batch_scaled<LA_PHI_ELU1, NK>(pp, pres, val, sc);
                    else if (p.phi == LA_PHI_RELU)
                        feat8_batch_scaled<LA_PHI_RELU, NK>(pp, pres, val, sc);
                    else
                        feat8_batch_scaled<LA_PHI_IDENTITY, NK>(pp, pres, val, sc);
                } else {
                    if (p.phi == LA_PHI_ELU1)
                        feat8_batch<LA_PHI_ELU1, NK>(pp, pres, val);
                    else if (p.phi == LA_PHI_RELU)
                        feat8_batch<LA_PHI_RELU, NK>(pp, pres, val);
                    else
                        feat8_batch<LA_PHI_IDENTITY, NK>(pp, pres, val);
                }
            }
            fence_proxy_async();
            if (pi == 0) LA_TL2(k, 2);
            mbar_arrive_warp(&bar_ready[s]);
        }
    } else if (warp >= 8 && warp < 12) {
        // ---------------- warpgroup A (thread = feature d): R conversion, dk and dv
        const int wq = warp % 4;
        const int d = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        float r_prev = 0.f;   // r before the current chunk
        const float grad_thr = feat_grad_threshold(p.phi);
        if (d < D) {
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                float v[16];
                seg_state_load16<D>(rstate_head, seg, p.nseg, kJoinR, p.scan_in_kernel, d, c16, v);
                if (CAUSAL) tmem_st16(tR + lane_off + c16 * 16, v);
                store_rbf_row<D>(rbf, d, v, c16);
            }
            r_prev = seg_state_z<D>(rstate_head, seg, p.nseg, kJoinR, p.scan_in_kernel, d);
        }
        if (MERGE_H)   // the r part (its two read columns) accumulates onto dk^T's product: clear it
            for (int bb = 0; bb < NB; ++bb) tmem_zero2(tRp(bb) + lane_off);
        if (CAUSAL || MERGE_H) tmem_st_wait();
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive_warp(&bar_rbf);
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS, bb = k % NB;
            if (CAUSAL) {   // the chunk's R part (its first products) is done
                ok = ok && warp_wait(&bar_rfull, k & 1, &abort_flag);
                tc_fence_after();
                if (d == 0) LA_TL2(k, 15);
            }
            // OUT_STAGE: phi(k) of column d, kept in registers so that the [K | V] region goes
            // back to the loader as soon as no MMA reads it (causal: after the R part, which
            // rfull says; bidirectional: after the chunk's products)
            const uint8_t *kr = stage0 + s * K::STAGE + OFF_K;
            uint32_t fk2[OUT_STAGE ? C / 2 : 1];
            if constexpr (OUT_STAGE) {
                if (!CAUSAL) {
                    ok = ok && warp_wait(&bar_outfull[bb], (k / NB) & 1, &abort_flag);
                    tc_fence_after();
                }
                const int dd = d < D ? d : 0;
#pragma unroll
                for (int j = 0; j < C; j += 2)
                    fk2[j / 2] = pack_bf16x2(__bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kr + swz_offset(C, j, dd))),
                                             __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kr + swz_offset(C, j + 1, dd))));
                mbar_arrive_warp(&bar_emptykv[s]);
            }
            if (CAUSAL) {   // R after this chunk -> R_bf for the next one
                if (ok && d < D) {
#pragma unroll
                    for (int c16 = 0; c16 < D / 16; ++c16) {
                        float v[16];
                        tmem_ld16(tR + lane_off + c16 * 16, v);
                        tmem_wait_regs<16>(v);
                        store_rbf_row<D>(rbf, d, v, c16);
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive_warp(&bar_rbf);
                if (d == 0) LA_TL2(k, 8);
            }
            if (!OUT_STAGE || CAUSAL) {
                ok = ok && warp_wait(&bar_outfull[bb], (k / NB) & 1, &abort_flag);
                tc_fence_after();
            }
            if (d == 0) LA_TL2(k, 7);
            float r_chunk = 0.f;   // phi_s^T h of this chunk (h split in two bf16 parts)
            if (CAUSAL && ok && d < D) {
                float rv[2];
                tmem_ld2(tRp(bb) + lane_off, rv);
                tmem_wait_regs<2>(rv);
                r_chunk = rv[0] + rv[1];
            }
            // the r part accumulates onto the next dk^T product of this buffer: clear it
            if (MERGE_H && ok) tmem_zero2(tRp(bb) + lane_off);
            // dk = phi'(k) * (dk^T + r) for column d of the chunk's C keys, then dv (row e = d
            // of dv^T), each written into the staging tile once the previous copy out of it
            // has read it (OUT_STAGE), else over phi(K) and V; each thread reads and writes only
            // its own column
            uint8_t *kw = OUT_STAGE ? obuf : stage0 + s * K::STAGE + OFF_K;
            uint8_t *vw = OUT_STAGE ? obuf : stage0 + s * K::STAGE + OFF_V;
            if (OUT_STAGE && k > 0) ok = ok && warp_wait(&bar_stfree, 1u, &abort_flag);   // dv of chunk k - 1
#pragma unroll 1
            for (int c16 = 0; c16 < C / 16; ++c16) {
                if (!ok || d >= D) break;
                float v[16];
                tmem_ld16(tK(bb) + lane_off + c16 * 16, v);
                tmem_wait_regs<16>(v);
                float fk[16];   // the column's 16 phi(k) values, all loaded before any store
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    if constexpr (OUT_STAGE) {
                        const float2 u = unpack_bf16x2(fk2[(c16 * 16 + e) / 2 % (OUT_STAGE ? C / 2 : 1)]);
                        fk[e] = (e & 1) ? u.y : u.x;
                    } else {
                        fk[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kw + swz_offset(C, c16 * 16 + e, d)));
                    }
                }
                if constexpr (WT) {   // w phi'(k) (dk^T + r); cos pass: to the workspace (fp32),
                                      // sin pass: plus the cos pass's (every load before any store)
                    const int c0 = t0 + (nchunk - 1 - k) * C;
                    if (p.pass == 2 && c16 == 0 && d == 0 && k + 1 < nchunk) {   // the next (earlier) chunk's
                        const size_t nx = ((size_t)bg * p.N + (c0 - C)) * D;   // C x D blocks into L2
                        prefetch_l2_bulk(p.part_dk + nx, (uint32_t)(C * D * 4));
                        prefetch_l2_bulk(p.part_dv + nx, (uint32_t)(C * D * 4));
                    }
#pragma unroll
                    for (int e8 = 0; e8 < 16; e8 += 8) {
                        float wv[8], prev[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = c16 * 16 + e8 + e;
                            const bool kv = c0 + j < t1;
                            wv[e] = kv ? __ldg(p.wrow + c0 + j) : 0.f;
                            prev[e] = kv && p.pass == 2 ? __ldg(p.part_dk + ((size_t)bg * p.N + c0 + j) * D + d) : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = c16 * 16 + e8 + e;
                            const float val =
                                feat_grad_from_feat_w(fk[e8 + e], p.phi == LA_PHI_ELU1, grad_thr, wv[e]) * (v[e8 + e] + r_prev);
                            if (p.pass == 1) {
                                if (c0 + j < t1) p.part_dk[((size_t)bg * p.N + c0 + j) * D + d] = val;
                            } else {
                                *reinterpret_cast<__nv_bfloat16 *>(kw + swz_offset(C, j, d)) = __float2bfloat16_rn(val + prev[e]);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        *reinterpret_cast<__nv_bfloat16 *>(kw + swz_offset(C, c16 * 16 + e, d)) =
                            __float2bfloat16_rn(feat_grad_from_feat(fk[e], p.phi == LA_PHI_ELU1, grad_thr) * (v[e] + r_prev));
                }
            }
            fence_proxy_async();
            mbar_arrive_warp(&bar_dkready[s]);
            if constexpr (DVSPLIT) {   // dv is written by warps 20-23; dk^T has been read
                tc_fence_before();
                mbar_arrive_warp(&bar_outfree[bb]);
                r_prev += r_chunk;
                continue;
            }
            if (OUT_STAGE) ok = ok && warp_wait(&bar_stfree, 0u, &abort_flag);   // dk of chunk k
#pragma unroll 1
            for (int c16 = 0; c16 < C / 16; ++c16) {
                float v[16];
                if (ok && d < D) {
                    tmem_ld16(tV(bb) + lane_off + c16 * 16, v);
                    tmem_wait_regs<16>(v);
                }
                if (c16 + 1 == C / 16) {
                    if (MERGE_H && ok) tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive_warp(&bar_outfree[bb]);
                }
                if (!ok || d >= D) continue;
                if constexpr (WT) {   // cos pass: dv terms to the workspace; sin pass: plus those
                    const int c0 = t0 + (nchunk - 1 - k) * C;
                    if (p.pass == 1) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + c16 * 16 + e < t1) p.part_dv[((size_t)bg * p.N + c0 + c16 * 16 + e) * D + d] = v[e];
                    } else {
#pragma unroll
                        for (int e8 = 0; e8 < 16; e8 += 8) {
                            float prev[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = c16 * 16 + e8 + e;
                                prev[e] = c0 + j < t1 ? __ldg(p.part_dv + ((size_t)bg * p.N + c0 + j) * D + d) : 0.f;
                            }
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                *reinterpret_cast<__nv_bfloat16 *>(vw + swz_offset(C, c16 * 16 + e8 + e, d)) =
                                    __float2bfloat16_rn(v[e8 + e] + prev[e]);
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        *reinterpret_cast<__nv_bfloat16 *>(vw + swz_offset(C, c16 * 16 + e, d)) = __float2bfloat16_rn(v[e]);
                }
            }
            fence_proxy_async();
            mbar_arrive_warp(&bar_dvready[s]);
            if (d == 0) LA_TL2(k, 9);
            r_prev += r_chunk;
        }
    } else if ((warp >= 12 && warp < 16) || (PSPLIT && warp >= 4 && warp < 8)) {
        // ---------------- warpgroup B (warps 12-15, thread = query row i): P' and dP'; with
        // PSPLIT warps 4-7 take every second 16-key piece of the same rows
        const bool wgb = warp >= 12;
        const int c16_0 = PSPLIT && !wgb ? 1 : 0, c16_step = PSPLIT ? 2 : 1;
        const int wq = warp % 4;
        const int i = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int ti = i % C, bh = bh0 + i / C;
        bool ok = true;
        float hv = 0.f;   // h of this thread's row in chunk k, loaded one step ahead
        if (CAUSAL && nchunk > 0) {
            const int t = t0 + (nchunk - 1) * C + ti;
            if (t < t1 && i / C < gr && LA_CHECK((size_t)bh * p.N + t < (size_t)p.B * p.Hq * p.N, 434, bh, t))
                hv = p.gd[(size_t)bh * p.N + t];
        }
        for (int k = 0; k < nchunk && CAUSAL; ++k) {
            // P'^T = mask(A_s)^T, dP' = mask(dA' + h) for chunk k, and h (split) for the r part,
            // once chunk k - 1's finish has read P' and dP'
            if (k > 0) {
                ok = ok && warp_wait(&bar_outfull[(k - 1) % NB], ((k - 1) / NB) & 1, &abort_flag);
                tc_fence_after();
            }
            const int bb = k % NB;
            ok = ok && warp_wait(&bar_afull[bb], (k / NB) & 1, &abort_flag);
            tc_fence_after();
            if (i == 0 && wgb) LA_TL2(k, 10);
            float hnext = 0.f;
            if (k + 1 < nchunk) {
                const int tn = t0 + (nchunk - 2 - k) * C + ti;
                if (tn < t1 && i / C < gr && LA_CHECK((size_t)bh * p.N + tn < (size_t)p.B * p.Hq * p.N, 435, bh, tn))
                    hnext = p.gd[(size_t)bh * p.N + tn];
            }
            if (ok && wgb) {
                const __nv_bfloat16 hh = __float2bfloat16_rn(hv);
                const __nv_bfloat16 hl = __float2bfloat16_rn(hv - __bfloat162float(hh));
                if (K::H_IN_DP) {
                    *reinterpret_cast<__nv_bfloat16 *>(dpbuf + swz_offset(128, i, C)) = hh;
                    *reinterpret_cast<__nv_bfloat16 *>(dpbuf + swz_offset(128, i, C + 1)) = hl;
                } else {
                    *reinterpret_cast<__nv_bfloat16 *>(htile + swz_offset(16, 0, i)) = hh;
                    *reinterpret_cast<__nv_bfloat16 *>(htile + swz_offset(16, 1, i)) = hl;
                }
            }
            if (ok) {
#pragma unroll 1
                for (int c16 = c16_0; c16 < C / 16; c16 += c16_step) {
                    float va[16], vd[16];
                    tmem_ld16(tA(bb) + lane_off + c16 * 16, va);
                    tmem_ld16(tD(bb) + lane_off + c16 * 16, vd);
                    tmem_wait_regs<16>(va);
                    tmem_wait_regs<16>(vd);
                    uint32_t wd[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const int j = c16 * 16 + e;
                        const bool m0 = j <= ti, m1 = j + 1 <= ti;
                        wd[e / 2] = pack_bf16x2(m0 ? vd[e] + hv : 0.f, m1 ? vd[e + 1] + hv : 0.f);
                    }
                    uint8_t *q0 = dpbuf + swz_chunk(128, i, 2 * c16), *q1 = dpbuf + swz_chunk(128, i, 2 * c16 + 1);
                    uint8_t *pt = ptbuf + swz_offset(C, c16 * 16, i);
                    if (LA_CHECK(in_smem(q0, 16, sm_lo, sm_hi) && in_smem(q1, 16, sm_lo, sm_hi) &&
                                     in_smem(pt, 2, sm_lo, sm_hi) && in_smem(ptbuf + swz_offset(C, c16 * 16 + 15, i), 2, sm_lo, sm_hi),
                                 431, smem_u32(q0) - sm_lo, c16)) {
                        *reinterpret_cast<uint4 *>(q0) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                        *reinterpret_cast<uint4 *>(q1) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
                        // P'^T: row j (key), column i; a warp writes 64 contiguous bytes of a row
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int j = c16 * 16 + e;
                            *reinterpret_cast<__nv_bfloat16 *>(ptbuf + swz_offset(C, j, i)) =
                                __float2bfloat16_rn(j <= ti ? va[e] : 0.f);
                        }
                    }
                }
                fence_proxy_async();
            }
            tc_fence_before();
            if (i == 0 && wgb) LA_TL2(k, 11);
            mbar_arrive_warp(&bar_pready);
            hv = hnext;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (threadIdx.x == 0 && abort_flag) atomicExch(p.err, kErrTimeout);
    LA_SPAN(3, 1);
}

// ---------------------------------------------------------------------------------------
// Host side

template <int D, int G, bool CAUSAL, bool MASK, bool WT>
cudaError_t launch_bwd_kernels(const Params &p, cudaStream_t s) {
    using K = BwdCfg<D, G>;
    CUtensorMap mq{}, mk{}, mv{}, mg{}, mdq{}, mdk{}, mdv{}, mps{}, mqs{}, mden{};
    // inputs through 4-D maps with the caller's strides; outputs (and phi_s) contiguous
    cudaError_t e = make_map_in(&mq, p.q, p.B, p.Hq, p.N, D, p.st_q, K::C);
    if (e == cudaSuccess) e = make_map_rows_f32(&mden, p.den, p.B * p.Hq, p.N, p.den_stride, K::C);
    // phi(q) / den rows: written by the dq kernel (mps), read by the dk/dv kernel in place of q
    // (mqs; bidirectional: q itself, and mps is not used)
    if (e == cudaSuccess) e = make_map(&mps, CAUSAL ? p.phis : p.dq, p.B * p.Hq, p.N, D, K::C);
    if (e == cudaSuccess)
        e = CAUSAL ? make_map_in(&mqs, p.phis, p.B, p.Hq, p.N, D, contiguous_strides(p.Hq, p.N, D), K::C)
                   : make_map_in(&mqs, p.q, p.B, p.Hq, p.N, D, p.st_q, K::C);
    if (e == cudaSuccess) e = make_map_in(&mk, p.k, p.B, p.Hkv, p.N, D, p.st_k, K::C);
    if (e == cudaSuccess) e = make_map_in(&mv, p.v, p.B, p.Hkv, p.N, D, p.st_v, K::C);
    if (e == cudaSuccess) e = make_map_in(&mg, p.g, p.B, p.Hq, p.N, D, p.st_g, K::C);
    if (e == cudaSuccess) e = make_map(&mdq, p.dq, p.B * p.Hq, p.N, D, K::C);
    if (e == cudaSuccess) e = make_map(&mdk, p.dk, p.B * p.Hkv, p.N, D, K::C);
    if (e == cudaSuccess) e = make_map(&mdv, p.dv, p.B * p.Hkv, p.N, D, K::C);
    if (e == cudaSuccess) e = prepare(k_tc_bwd_dq<D, G, CAUSAL, MASK, WT>, K::DQ_SMEM);
    if (e == cudaSuccess) e = prepare(k_tc_bwd_dkdv<D, G, CAUSAL, MASK, WT>, K::DKDV_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = p.B * p.Hkv * p.nseg;
    {
        TraceScope ts(CAUSAL ? "tc_bwd_dq_causal" : "tc_bwd_dq_bidir", s);
        e = launch_pdl(k_tc_bwd_dq<D, G, CAUSAL, MASK, WT>, dim3(grid), dim3(kDqThreads), K::DQ_SMEM, s, mq, mk, mv, mg, mdq,
                       mps, mden, p);
    }
    if (e == cudaSuccess && !p.scan_in_kernel)
        e = scan_segments(p.rstate, p, CAUSAL ? kScanSuffix : kScanTotal, (size_t)D * (D + 1), s);
    if (e != cudaSuccess) return e;
    TraceScope ts(CAUSAL ? "tc_bwd_dkdv_causal" : "tc_bwd_dkdv_bidir", s);
    return launch_pdl(k_tc_bwd_dkdv<D, G, CAUSAL, MASK, WT>, dim3(grid), dim3(kKvThreads), K::DKDV_SMEM, s, mqs, mk, mv, mg,
                      mdk, mdv, p);
}

// h = -g . out per row (out: the forward's float32 output rows, chunk-blocked over its
// C-token chunks): the h of the cos/sin-weighted backward, shared by its two passes.  One
// block per (head, chunk), thread = row, so the out reads of a column are one run.
__global__ void k_h_rows(const __nv_bfloat16 *__restrict__ g, Strides sg, int H, int N, int C,
                         const float *__restrict__ out, float *__restrict__ h, int D) {
    pdl_wait();
    const int nck = (N + C - 1) / C;
    const int bh = blockIdx.x / nck, t = (blockIdx.x % nck) * C + threadIdx.x;
    if (threadIdx.x >= C || t >= N) return;
    const __nv_bfloat16 *gr = g + (long long)(bh / H) * sg.b + (long long)(bh % H) * sg.h + (long long)t * sg.n;
    const float *orow = out + blocked_index(bh, t, 0, N, D, C);
    float acc = 0.f;
    for (int d = 0; d < D; d += 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(gr + d);
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            acc = fmaf(f.x, orow[(size_t)(d + 2 * e) * C], acc);
            acc = fmaf(f.y, orow[(size_t)(d + 2 * e + 1) * C], acc);
        }
    }
    h[(size_t)bh * N + t] = -acc;
}

// The backward with cos/sin weights, W_ij = c_i c_j + s_i s_j, as two passes (cos, then sin)
// of the one-term kernels with the features w phi: with gn = g / den and gd = h / den shared
// by both terms (den, the sum of both terms' plus eps, from the forward; h = -g . out), each
// term's gradient is the one-term backward with those features and that h, times the weight
// where the feature is differentiated (w phi'(q), w phi'(k)); the cos pass leaves dq, dk, dv
// in float32 in the workspace and the sin pass adds its own before rounding.
template <int D, int G, bool MASK>
cudaError_t backward_two_pass(const Params &p, cudaStream_t s) {
    if (!p.cw || !p.sw || !p.part_num || !p.part_dq || !p.part_dk || !p.part_dv) return cudaErrorInvalidValue;
    cudaError_t e = cudaSuccess;
    if (!p.state_given) {   // the forward (two passes), its output to dq as scratch
        Params pf = p;
        pf.out = p.dq;
        e = tc_forward(pf, s);
        if (e != cudaSuccess) return e;
    }
    {
        TraceScope ts("tc_bwd_h_rows", s);
        const int nck = (p.N + p.chunk - 1) / p.chunk;   // the forward's chunks (p.chunk)
        e = launch_pdl(k_h_rows, dim3((unsigned)(p.B * p.Hq * nck)), dim3(p.chunk), 0, s,
                       static_cast<const __nv_bfloat16 *>(p.g), p.st_g, p.Hq, p.N, p.chunk, (const float *)p.part_num, p.gd, D);
    }
    const size_t pass_elems = (size_t)p.B * p.Hkv * p.nseg * D * (D + 1);
    for (int pass = 1; pass <= 2 && e == cudaSuccess; ++pass) {
        Params pp = p;
        pp.pass = pass;
        pp.wrow = pass == 1 ? p.cw : p.sw;
        pp.state = p.state + (size_t)(pass - 1) * pass_elems;
        e = p.causal ? launch_bwd_kernels<D, G, true, MASK, true>(pp, s) : launch_bwd_kernels<D, G, false, MASK, true>(pp, s);
    }
    return e;
}

template <int D, int G, bool MASK = false>
cudaError_t backward_dg(const Params &p, cudaStream_t s) {
    if constexpr (!BwdCfg<D, G>::FITS || !BwdCfg<D, G>::TMEM_FITS) {
        return cudaErrorNotSupported;
    } else {
        if (p.P == 2) return backward_two_pass<D, G, MASK>(p, s);
        if (!p.state_given) {
            // the forward gives the segment states, the per-row den and the record; its output
            // goes to dq, which the dq kernel overwrites
            Params pf = p;
            pf.out = p.dq;
            cudaError_t e = tc_forward(pf, s);
            if (e != cudaSuccess) return e;
        }
        return p.causal ? launch_bwd_kernels<D, G, true, MASK, false>(p, s) : launch_bwd_kernels<D, G, false, MASK, false>(p, s);
    }
}

template <int D>
cudaError_t backward_d(const Params &p, cudaStream_t s) {
    switch (p.n_rep) {   // D = 128, n_rep <= 2: the n_rep = 4 tiles with rows masked (k_tc_bwd_dq)
        case 1:
            if constexpr (D == 128) return backward_dg<D, 4, true>(p, s);
            else return backward_dg<D, 1>(p, s);
        case 2:
            if constexpr (D == 128) return backward_dg<D, 4, true>(p, s);
            else return backward_dg<D, 2>(p, s);
        case 4: return backward_dg<D, 4>(p, s);
        case 8: return backward_dg<D, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool tc_bwd_supported(int n_rep, int D) {
    return (D == 64 || D == 128) && (n_rep == 1 || n_rep == 2 || n_rep == 4 || n_rep == 8);
}

cudaError_t tc_backward(const Params &p, cudaStream_t s) {
    return p.D == 128 ? backward_d<128>(p, s) : (p.D == 64 ? backward_d<64>(p, s) : cudaErrorNotSupported);
}

}  // namespace la

#ifdef LA_TIMELINE
// Timeline builds only: the dq kernel's event clocks ([64][16] long long).
extern "C" int la_timeline_read_bwd(long long *out) {
    return cudaMemcpyFromSymbol(out, la::g_la_tl, sizeof(long long) * 64 * 16) == cudaSuccess ? 0 : 1;
}
// ... and the dk/dv kernel's.
extern "C" int la_timeline_read_bwd2(long long *out) {
    return cudaMemcpyFromSymbol(out, la::g_la_tl2, sizeof(long long) * 64 * 16) == cudaSuccess ? 0 : 1;
}
// ... and the per-block entry and exit times of this file's kernels ([4][256][2], ns).
extern "C" int la_timeline_read_span_bwd(unsigned long long *out) {
    return cudaMemcpyFromSymbol(out, la::g_la_span, sizeof(unsigned long long) * 4 * 256 * 2) == cudaSuccess ? 0 : 1;
}
#endif

#ifdef LA_DEBUG
// Debug builds only: the first failed self-check of the backward kernels (id, a, b, block).
extern "C" int la_debug_read_bwd(int *out4) {
    if (cudaMemcpyFromSymbol(out4, la::g_la_debug, 4 * sizeof(int)) != cudaSuccess) return 1;
    const int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(la::g_la_debug, zero, 4 * sizeof(int)) == cudaSuccess ? 0 : 1;
}
#endif
