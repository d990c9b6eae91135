// la_tc.cu -- tensor-core kernels (tcgen05 / TMEM / TMA) for bfloat16 inputs: forward.
//
// The dense contractions of the chunked linear attention ("chunked causal streaming" and
// "bidirectional parallel reduction" in the linear_attn module docstring) run as
// tcgen05.mma with bf16 operands in 128-byte-swizzled shared memory and fp32 accumulators
// in TMEM; tiles arrive by TMA and the output leaves by TMA.  The query rows of one chunk
// are the n_rep heads of a key/value group stacked on the MMA's M = 128 rows (G = n_rep
// heads x C = 128 / G tokens), so one key/value tile serves the whole group (the gqa
// page's head sharing, fused: no expanded k, v).
//
// z and the inter-chunk part of the denominator also run on the tensor cores, through N = 16
// products against two small K-major tiles: ONES (row 0 all ones) and Z (rows 0 and 1: z
// split into two bf16 terms, z = z_hi + z_lo, so phi(q) . z comes out as two fp32 columns
// with the accuracy of float32).  The intra-chunk part of the denominator, the row sum of
// mask(A), is taken twice: through the bf16 P (a product with a second ones tile whose row 2
// is ones, landing in column D + 2), for out = O / den with the same P in numerator and
// denominator; and in float32 by the warps that build P, which also write the den left to
// the backward: that one must be accurate to float32 rounding (a den error is amplified
// there by the h z term; measured, the bf16 row sum raises the dq error by 30 %).
//
// Forward = k_tc_state (per-segment S = phi(K)^T V, z = phi(K)^T 1) -> k_scan (exclusive
// prefix, or total when bidirectional; CUDA cores) -> k_tc_fwd.  Per chunk of k_tc_fwd
// (M = 128 query rows, C keys):
//   MMA1  A   = phi(Q) phi(K)^T                                [128 x C]   (causal)
//   conv  P   = bf16(A masked j <= i)                                      (causal)
//   MMA2  O   = phi(Q) S_bf + P V                              [128 x D]
//         den = phi(Q) z_hi + phi(Q) z_lo + P 1    (columns D, D + 1, D + 2)
//   epi   out = O / (den + eps)  -> staged in shared memory -> TMA store; den + eps per row
//         to the workspace (the backward's dq kernel reads it)
//   MMA3  S  += phi(K)^T V,  z += phi(K)^T 1                              (causal)
//   conv  S_bf, z_bf = bf16(S, z) for the next chunk
// Warp roles (640 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM owner,
// warps 4-7 and 16-19 phi prologue (in place, bf16x2; even and odd chunks), warps 8-11
// state and P conversion, warps 12-15 epilogue.  O is double-buffered in TMEM when it
// fits, so the epilogue of a chunk overlaps the next chunk's MMAs.
#include "la_tc_common.cuh"

namespace la {
namespace {

constexpr int kFwdThreads = 768, kFwdPro = 384;   // feature map: warps 4-7 and 16-23

#ifdef LA_TEST_HOOKS
__device__ int g_la_test_skip;   // test build: withhold one arrival in k_tc_fwd (see there)
#endif

template <int D, int G>
struct FwdCfg {
    static constexpr int C = 128 / G;                  // tokens per chunk
    static constexpr int DB = D / 64;                  // 64-wide blocks per D-wide row
    static constexpr int CB = (C + 63) / 64;           // 64-wide blocks per C-wide row
    static constexpr int Q_BYTES = 128 * D * 2;        // 128 query rows
    static constexpr int K_BYTES = C * D * 2;
    static constexpr int V_BYTES = C * D * 2;
    static constexpr int STAGE = Q_BYTES + K_BYTES + V_BYTES;
    static constexpr int P_BYTES = CB * 128 * 128;
    static constexpr int S_BYTES = DB * D * 128;       // S_bf: D rows (d) x D columns (e)
    static constexpr int Z_BYTES = DB * 16 * 128;      // z_bf: 16 rows x D columns, K-major
    static constexpr int ONES_BYTES = CB * 16 * 128;   // ones: 16 rows x C columns, K-major
    static constexpr int OUT_BYTES = 128 * 128;        // output staging: 128 rows x 64 columns
    static constexpr int FIXED = P_BYTES + S_BYTES + Z_BYTES + 2 * ONES_BYTES + OUT_BYTES + 1024;
    static constexpr int NS = (kSmemLimit - 1024 - FIXED) / STAGE > 4 ? 4 : (kSmemLimit - 1024 - FIXED) / STAGE;
    static constexpr int SMEM = NS * STAGE + FIXED;
    static_assert(NS >= 2, "not enough shared memory for two stages");
    // TMEM columns: [S | z], O (+ den in column D) in one or two buffers, A
    static constexpr int NW = D + 16;
    static constexpr int T_S = 0;
    static constexpr int T_O0 = align32(NW);
    static constexpr bool O2 = 3 * align32(NW) + C <= 512;
    static constexpr int T_O1 = O2 ? T_O0 + align32(NW) : T_O0;
    static constexpr int T_A = T_O1 + align32(NW);
    static_assert(T_A + C <= 512, "TMEM budget");
};

// k_tc_state: warp 0 TMA, warp 1 MMA, warps 4-15 the feature map (all of them on every
// chunk) and, at the end, warps 4-7 the TMEM readout.
constexpr int kStateThreads = 512;
constexpr int kStatePro = kStateThreads - 128;

template <int D>
struct StateCfg {
    static constexpr int C = 64;
    static constexpr int DB = D / 64;
    static constexpr int K_BYTES = C * D * 2;
    static constexpr int STAGE = 2 * K_BYTES;                  // K, V
    static constexpr int ONES_BYTES = 16 * 128;
    static constexpr int NS = (kSmemLimit - 4096) / STAGE > 6 ? 6 : (kSmemLimit - 4096) / STAGE;
    static constexpr int SMEM = NS * STAGE + ONES_BYTES + 1024;
};

// The state kernel's feature map over a K tile: thread i of kStatePro takes 16-byte pieces
// idx = i, i + kStatePro, ... (row j = idx / (D / 8)); rows at or past t1 become zeros.  WT:
// each row times its position weight w[token].
template <int PHI, int C, int D, bool WT>
__device__ __forceinline__ void state_feature_map(uint8_t *kt, int i, int c0, int t1, const float *w, uint32_t sm_lo,
                                                  uint32_t sm_hi) {
    (void)sm_lo;
    (void)sm_hi;
    (void)w;
#pragma unroll 2
    for (int idx = i; idx < C * (D / 8); idx += kStatePro) {
        const int j = idx / (D / 8), c = idx % (D / 8);
        uint8_t *ch = kt + swz_chunk(C, j, c);
        if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 121, smem_u32(ch) - sm_lo, idx)) {
            const bool valid = c0 + j < t1;
            if constexpr (WT)
                feat8_weighted<PHI>(ch, valid, valid ? w[c0 + j] : 0.f);
            else
                feat8_inplace2<PHI>(ch, valid);
        }
    }
}

// The forward's feature map over one stage: 16-byte piece `offq` of Q rows r0, r0 + RPP, ...
// (valid while row < qrows, the rows of the group's real heads, and row % C < nvalid; the
// other rows become zeros) and, causal, piece `kpiece` of K rows r0, r0 + RPP, ...  WT: each
// row times the position weight w[c0 + token].
template <int PHI, int C, int RPP, bool CAUSAL, bool WT>
__device__ __forceinline__ void fwd_feature_map(uint8_t *st, uint32_t offq, uint8_t *kpiece, int r0, int nvalid,
                                                int qrows, int c0, const float *w, uint32_t sm_lo, uint32_t sm_hi) {
    (void)sm_lo;
    (void)sm_hi;
    (void)c0;
    (void)w;
#pragma unroll 4
    for (int row = r0; row < 128; row += RPP) {
        uint8_t *ch = st + offq + row * 128;
        if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 221, smem_u32(ch) - sm_lo, row)) {
            const bool valid = row < qrows && row % C < nvalid;
            if constexpr (WT)
                feat8_weighted<PHI>(ch, valid, valid ? w[c0 + row % C] : 0.f);
            else
                feat8_inplace2<PHI>(ch, valid);
        }
    }
    if (CAUSAL)
        for (int j = r0; j < C; j += RPP) {
            uint8_t *ch = kpiece + j * 128;
            if (LA_CHECK(in_smem(ch, 16, sm_lo, sm_hi), 222, smem_u32(ch) - sm_lo, j)) {
                if constexpr (WT)
                    feat8_weighted<PHI>(ch, j < nvalid, j < nvalid ? w[c0 + j] : 0.f);
                else
                    feat8_inplace2<PHI>(ch, j < nvalid);
            }
        }
}

// ---------------------------------------------------------------------------------------
// Per-segment state: S = phi(K)^T V and z = phi(K)^T 1 over the segment's tokens (fp32 in
// TMEM), written to the workspace as [D][D+1] (z in column D).  WT: phi(k) rows weighted by
// the pass's position weights (cos or sin).
template <int D, bool WT>
__global__ void __launch_bounds__(kStateThreads, 1) k_tc_state(const __grid_constant__ CUtensorMap map_k,
                                                     const __grid_constant__ CUtensorMap map_v, Params p) {
    using K = StateCfg<D>;
    constexpr int C = K::C, NS = K::NS;
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();
    LA_SPAN(0, 0);
    __shared__ uint64_t bar_full[NS], bar_ready[NS], bar_empty[NS], bar_done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    uint8_t *ones = stage0 + NS * K::STAGE;
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::SMEM;
    (void)sm_lo;
    (void)sm_hi;
    const int warp = threadIdx.x / 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;

    fill_ones_tile(ones, C);
    fence_proxy_async();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_ready[s], kStatePro);
            mbar_init(&bar_empty[s], 1);
        }
        mbar_init(&bar_done, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base;

    if (warp == 0) {
        {   // the whole warp, one lane issuing
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (k >= NS && !warp_wait(&bar_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C;
                if (!LA_CHECK(in_smem(st, K::STAGE, sm_lo, sm_hi) && c0 < p.N, 101, smem_u32(st) - sm_lo, c0)) break;
                mbar_arrive_expect_tx_w(&bar_full[s], K::STAGE);
                for (int blk = 0; blk < K::DB; ++blk) {
                    tma_load_4d_w(st + blk * C * 128, &map_k, &bar_full[s], blk * 64, c0, g, b);
                    tma_load_4d_w(st + K::K_BYTES + blk * C * 128, &map_v, &bar_full[s], blk * 64, c0, g, b);
                }
                issued = k + 1;
            }
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k) warp_drain(&bar_full[k % NS], (k / NS) & 1);
        }
    } else if (warp == 1) {
        {   // the whole warp, one lane issuing
            constexpr uint32_t idS = idesc_bf16(128, D, true, true);
            constexpr uint32_t idZ = idesc_bf16(128, 16, true, false);
            const uint32_t on = smem_u32(ones);
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (!warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t ks_ = smem_u32(stage0 + s * K::STAGE), vs_ = ks_ + K::K_BYTES;
                if (!LA_CHECK(ks_ >= sm_lo && ks_ + (uint32_t)K::STAGE <= sm_hi, 111, ks_ - sm_lo, k)) break;
                for (int kk = 0; kk < C / 16; ++kk) {
                    const uint32_t acc = (k > 0 || kk > 0) ? 1u : 0u;
                    mma_bf16_w(tS, desc_mnmajor(ks_, C, 0, kk), desc_mnmajor(vs_, C, 0, kk), idS, acc);
                    mma_bf16_w(tS + D, desc_mnmajor(ks_, C, 0, kk), desc_kmajor(on, 16, 0, kk), idZ, acc);
                }
                mma_commit_w(&bar_empty[s]);
            }
            mma_commit_w(&bar_done);
            warp_drain(&bar_done, 0);
        }
    } else if (warp >= 4) {
        const int i = threadIdx.x - 128;   // 0 .. kStatePro - 1
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            ok = ok && warp_wait(&bar_full[s], (k / NS) & 1, &abort_flag);
            if (ok) {
                uint8_t *kt = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C;
                if (p.phi == LA_PHI_ELU1)
                    state_feature_map<LA_PHI_ELU1, C, D, WT>(kt, i, c0, t1, p.wrow, sm_lo, sm_hi);
                else if (p.phi == LA_PHI_RELU)
                    state_feature_map<LA_PHI_RELU, C, D, WT>(kt, i, c0, t1, p.wrow, sm_lo, sm_hi);
                else
                    state_feature_map<LA_PHI_IDENTITY, C, D, WT>(kt, i, c0, t1, p.wrow, sm_lo, sm_hi);
                fence_proxy_async();
            }
            mbar_arrive_warp(&bar_ready[s]);
        }
        ok = ok && warp_wait(&bar_done, 0, &abort_flag);
        tc_fence_after();
        // TMEM rows (lane d: S[d][0..D-1], z[d]) -> shared memory in the lane-blocked state
        // layout (the stages are idle now; a warp's 16-byte stores are side by side)
        const int wq = warp % 4;
        float *srow = reinterpret_cast<float *>(stage0);
        if (ok && warp < 8 && wq * 32 < D) {
            const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
#pragma unroll 1
            for (int c16 = 0; c16 <= D / 16; ++c16) {
                float v[16];
                tmem_ld16(tS + lane_off + c16 * 16, v);
                tmem_wait_regs<16>(v);
                if (c16 < D / 16)
                    state_store16<D>(srow, i, c16, v);
                else
                    state_store_z<D>(srow, i, v[0]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    // the segment's D (D + 1) floats are contiguous (and 16-byte aligned) in the workspace:
    // every thread copies 16-byte pieces
    if (!abort_flag) {
        const float4 *src4 = reinterpret_cast<const float4 *>(stage0);
        float4 *dst4 = reinterpret_cast<float4 *>(p.state + ((size_t)bg * p.nseg + seg) * (size_t)(D * (D + 1)));
        static_assert(D * (D + 1) % 4 == 0, "whole 16-byte pieces");
        for (int idx = threadIdx.x; idx < D * (D + 1) / 4; idx += blockDim.x) dst4[idx] = src4[idx];
    }
    if (warp == 1) tmem_dealloc(tS, 256);
    if (threadIdx.x == 0 && abort_flag) atomicExch(p.err, kErrTimeout);
    LA_SPAN(0, 1);
}

// ---------------------------------------------------------------------------------------
// Chunked forward (see the file comment for the per-chunk steps and warp roles).  MASK: the
// group has fewer heads (n_rep) than the tile's G, and the rows past them are masked.  WT: one
// of the two passes of the cos/sin-weighted forward (p.pass: 1 cos, 2 sin; see forward_dg).
template <int D, int G, bool CAUSAL, bool MASK, bool WT>
__global__ void __launch_bounds__(kFwdThreads, 1) k_tc_fwd(const __grid_constant__ CUtensorMap map_q,
                                                           const __grid_constant__ CUtensorMap map_k,
                                                           const __grid_constant__ CUtensorMap map_v,
                                                           const __grid_constant__ CUtensorMap map_o, Params p) {
    using K = FwdCfg<D, G>;
    constexpr int C = K::C, NS = K::NS;
    constexpr int OFF_K = K::Q_BYTES, OFF_V = OFF_K + K::K_BYTES;
    constexpr int NO = K::O2 ? 2 : 1;   // O buffers
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();
    LA_SPAN(1, 0);
    __shared__ uint64_t bar_full[NS], bar_ready[NS], bar_empty[NS], bar_ofull[2], bar_ofree[2];
    __shared__ uint64_t bar_afull, bar_pready, bar_sfull, bar_sbf, bar_fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    const uint32_t sm_lo = smem_u32(smem_raw), sm_hi = sm_lo + K::SMEM;
    (void)sm_lo;
    (void)sm_hi;
    uint8_t *pbuf = stage0 + NS * K::STAGE;
    uint8_t *sbf = pbuf + K::P_BYTES;
    uint8_t *ztile = sbf + K::S_BYTES;
    uint8_t *ones = ztile + K::Z_BYTES;
    uint8_t *ones2 = ones + K::ONES_BYTES;   // row 2 = 1: P 1 into column D + 2
    uint8_t *obuf = ones2 + K::ONES_BYTES;

    const int warp = threadIdx.x / 32;
    const int bg = blockIdx.x / p.nseg, seg = blockIdx.x % p.nseg;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int t0 = seg * p.seg_len, t1 = min(p.N, t0 + p.seg_len);
    const int nchunk = (t1 - t0 + C - 1) / C;
    // the group's gr = n_rep heads fill rows [0, gr C) of the G C = 128 MMA rows; with gr < G
    // (a group smaller than the tile's) the other rows stay zero and nothing is stored for them
    const int gr = MASK ? p.n_rep : G;
    const int bh0 = b * p.Hq + g * gr;
    const float *state_head = p.state + (size_t)bg * p.nseg * (size_t)(D * (D + 1));   // segment 0's state
    constexpr int kJoin = CAUSAL ? kScanPrefix : kScanTotal;

    // the record of this call, checked by a backward that takes this workspace's states and dens
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.hdr) {
        const int rec[kHdrWords] = {kHdrMagic, p.B, p.Hq, p.Hkv, p.N, p.D, p.causal, p.phi, p.P,
                                    __float_as_int(p.eps), p.nseg, p.chunk,
                                    (int)reinterpret_cast<uintptr_t>(p.q), (int)(reinterpret_cast<uintptr_t>(p.q) >> 32),
                                    (int)reinterpret_cast<uintptr_t>(p.k), (int)reinterpret_cast<uintptr_t>(p.v)};
        for (int w = 0; w < kHdrWords; ++w) p.hdr[w] = rec[w];
    }
    // constant tiles: ones (row 0 = 1 over C columns), ones2 (row 2 = 1) and the zero rows of
    // the z tile
    fill_ones_tile(ones, C);
    fill_ones_tile(ones2, C, 2);
    for (int idx = threadIdx.x; idx < K::Z_BYTES / 16; idx += blockDim.x)
        reinterpret_cast<uint4 *>(ztile)[idx] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_ready[s], kFwdPro);
            mbar_init(&bar_empty[s], 1);
        }
        for (int o = 0; o < 2; ++o) {
            mbar_init(&bar_ofull[o], 1);
            mbar_init(&bar_ofree[o], 128);
        }
        mbar_init(&bar_afull, 1);
        mbar_init(&bar_pready, 128);
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
    const uint32_t tS = tmem_base + K::T_S, tA = tmem_base + K::T_A;
    const uint32_t tO0 = tmem_base + K::T_O0, tO1 = tmem_base + K::T_O1;

    if (warp == 0) {
        // ---------------- TMA producer
        {   // the whole warp, one lane issuing
            const uint32_t bytes = (uint32_t)(gr * C * D * 2) + (CAUSAL ? (uint32_t)(K::K_BYTES + K::V_BYTES) : 0u);
            int issued = 0;
            for (int k = 0; k < nchunk; ++k) {
                const int s = k % NS;
                if (k >= NS && !warp_wait(&bar_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C;
                if (!LA_CHECK(in_smem(st, K::STAGE, sm_lo, sm_hi) && c0 < p.N && gr <= G && bh0 + gr <= p.B * p.Hq, 201,
                              smem_u32(st) - sm_lo, c0))
                    break;
                LA_TL(k, 0);
                mbar_arrive_expect_tx_w(&bar_full[s], bytes);
                for (int r = 0; r < gr; ++r)
                    for (int blk = 0; blk < K::DB; ++blk)
                        tma_load_4d_w(st + blk * 128 * 128 + r * C * 128, &map_q, &bar_full[s], blk * 64, c0, g * gr + r, b);
                if (CAUSAL)
                    for (int blk = 0; blk < K::DB; ++blk) {
                        tma_load_4d_w(st + OFF_K + blk * C * 128, &map_k, &bar_full[s], blk * 64, c0, g, b);
                        tma_load_4d_w(st + OFF_V + blk * C * 128, &map_v, &bar_full[s], blk * 64, c0, g, b);
                    }
                issued = k + 1;
            }
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k) warp_drain(&bar_full[k % NS], (k / NS) & 1);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer.  Per chunk k: the inter-chunk part of O (with S_bf and z)
        // and the state update, which the pool then converts for chunk k + 1; once P is ready,
        // chunk k + 1's scores A (when its feature map is done) and the intra-chunk part of O.
        // The epilogue turns A into P as soon as O no longer reads the P tile.
        {   // the whole warp, one lane issuing
            constexpr uint32_t idA = idesc_bf16(128, C, false, false);
            constexpr uint32_t idO = idesc_bf16(128, D, false, true);
            constexpr uint32_t idDen = idesc_bf16(128, 16, false, false);
            constexpr uint32_t idS = idesc_bf16(128, D, true, true);
            constexpr uint32_t idZ = idesc_bf16(128, 16, true, false);
            const uint32_t sbf_u = smem_u32(sbf), pb = smem_u32(pbuf), zt = smem_u32(ztile), on = smem_u32(ones),
                           on2 = smem_u32(ones2);
            // A for chunk k (causal), into the single A buffer once chunk k - 1's P has been read
            auto issue_a = [&](int k) -> bool {
                const int s = k % NS;
                if (!warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) return false;
                LA_TL(k, 3);
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), ks_ = qs + OFF_K;
                if (!LA_CHECK(qs >= sm_lo && qs + K::STAGE <= sm_hi, 212, qs - sm_lo, k)) return false;
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_w(tA, desc_kmajor(qs, 128, 0, kk), desc_kmajor(ks_, C, 0, kk), idA, kk > 0 ? 1u : 0u);
                mma_commit_w(&bar_afull);
                return true;
            };
            bool okm = !CAUSAL || nchunk == 0 || issue_a(0);
            for (int k = 0; okm && k < nchunk; ++k) {
                const int s = k % NS, o = k % NO;
                const uint32_t tO = o ? tO1 : tO0;
                if (!CAUSAL && !warp_wait(&bar_ready[s], (k / NS) & 1, &abort_flag)) break;
                if ((CAUSAL || k == 0) && !warp_wait(&bar_sbf, k & 1, &abort_flag)) break;
                LA_TL(k, 5);
                if (k >= NO && !warp_wait(&bar_ofree[o], ((k / NO) - 1) & 1, &abort_flag)) break;
                LA_TL(k, 6);
                tc_fence_after();
                const uint32_t qs = smem_u32(stage0 + s * K::STAGE), ks_ = qs + OFF_K, vs = qs + OFF_V;
                if (!LA_CHECK(qs >= sm_lo && qs + K::STAGE <= sm_hi && smem_u32(obuf) + K::OUT_BYTES <= sm_hi, 211,
                              qs - sm_lo, k))
                    break;
                // O = phi(Q) S_bf^T, den = phi(Q) z (the state before this chunk)
                for (int kk = 0; kk < D / 16; ++kk) {
                    mma_bf16_w(tO, desc_kmajor(qs, 128, 0, kk), desc_mnmajor(sbf_u, D, 0, kk), idO, kk > 0 ? 1u : 0u);
                    mma_bf16_w(tO + D, desc_kmajor(qs, 128, 0, kk), desc_kmajor(zt, 16, 0, kk), idDen, kk > 0 ? 1u : 0u);
                }
                bool a_next = false;
                if (CAUSAL) {
                    // S += phi(K)^T V, z += phi(K)^T 1; the commit also covers the reads of S_bf and z
                    for (int kk = 0; kk < C / 16; ++kk) {
                        mma_bf16_w(tS, desc_mnmajor(ks_, C, 0, kk), desc_mnmajor(vs, C, 0, kk), idS, 1u);
                        mma_bf16_w(tS + D, desc_mnmajor(ks_, C, 0, kk), desc_kmajor(on, 16, 0, kk), idZ, 1u);
                    }
                    mma_commit_w(&bar_sfull);
                    if (!warp_wait(&bar_pready, k & 1, &abort_flag)) break;
                    LA_TL(k, 4);
                    tc_fence_after();
                    // chunk k + 1's scores go first when its feature map is ready (A is free now)
                    if (k + 1 < nchunk && warp_test(&bar_ready[(k + 1) % NS], ((k + 1) / NS) & 1)) {
                        if (!issue_a(k + 1)) break;
                        a_next = true;
                    }
                    // O += P V, den += P 1 (within the chunk)
                    for (int kk = 0; kk < C / 16; ++kk) {
                        mma_bf16_w(tO, desc_kmajor(pb, 128, 0, kk), desc_mnmajor(vs, C, 0, kk), idO, 1u);
                        mma_bf16_w(tO + D, desc_kmajor(pb, 128, 0, kk), desc_kmajor(on2, 16, 0, kk), idDen, 1u);
                    }
                }
                mma_commit_w(&bar_ofull[o]);
                mma_commit_w(&bar_empty[s]);
                LA_TL(k, 7);
                if (CAUSAL && k + 1 < nchunk && !a_next && !issue_a(k + 1)) break;
            }
            mma_commit_w(&bar_fin);
            warp_drain(&bar_fin, 0);
        }
    } else if ((warp >= 4 && warp < 8) || warp >= 16) {
        // ---------------- phi prologue, in place on the swizzled Q and K tiles; all its
        // warps on every chunk, thread pi owning 16-byte piece c of rows r0, r0 + RPP, ...
        // (RPP a multiple of 8, so the piece's swizzled position is the same in all of them)
        const int pi = warp >= 16 ? threadIdx.x - 384 : threadIdx.x - 128;   // 0 .. kFwdPro - 1
        const int i = pi;
        constexpr int CPR = D / 8, RPP = kFwdPro / CPR;
        static_assert(RPP % 8 == 0, "rows per pass");
        const int c = pi % CPR, r0 = pi / CPR;
        const uint32_t pos = (uint32_t)(((c & 7) ^ (r0 & 7)) << 4);
        const uint32_t offq = (uint32_t)(c >> 3) * 128u * 128u + pos, offk = (uint32_t)(c >> 3) * C * 128u + pos;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int s = k % NS;
            ok = ok && warp_wait(&bar_full[s], (k / NS) & 1, &abort_flag);
            if (i == 0) LA_TL(k, 1);
            if (ok) {
                uint8_t *st = stage0 + s * K::STAGE;
                const int c0 = t0 + k * C, nvalid = t1 - c0;
                if (p.phi == LA_PHI_ELU1)
                    fwd_feature_map<LA_PHI_ELU1, C, RPP, CAUSAL, WT>(st, offq, st + OFF_K + offk, r0, nvalid, gr * C, c0,
                                                                     p.wrow, sm_lo, sm_hi);
                else if (p.phi == LA_PHI_RELU)
                    fwd_feature_map<LA_PHI_RELU, C, RPP, CAUSAL, WT>(st, offq, st + OFF_K + offk, r0, nvalid, gr * C, c0,
                                                                     p.wrow, sm_lo, sm_hi);
                else
                    fwd_feature_map<LA_PHI_IDENTITY, C, RPP, CAUSAL, WT>(st, offq, st + OFF_K + offk, r0, nvalid, gr * C,
                                                                         c0, p.wrow, sm_lo, sm_hi);
                fence_proxy_async();
            }
            if (i == 0) LA_TL(k, 2);
#ifdef LA_TEST_HOOKS
            // test build only: while armed, warp 4 of block 0 withholds its arrival for the
            // first chunk, so the MMA warp's bounded wait for that chunk runs out
            if (g_la_test_skip && blockIdx.x == 0 && k == 0 && warp == 4) continue;
#endif
            mbar_arrive_warp(&bar_ready[s]);
        }
    } else if (warp >= 8 && warp < 12) {
        // ---------------- state conversion (thread = d) and P conversion (thread = query row
        // i): S, z after chunk k for chunk k + 1, then P = mask(A) for chunk k + 1 as soon as
        // chunk k's O products (the readers of the P tile) are done
        const int i = threadIdx.x - 256;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int ti = i % C;
        // initial S, z of the segment: TMEM (causal) and the bf16 operand tiles
        if (wq * 32 < D) {
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                float v[16];
                seg_state_load16<D>(state_head, seg, p.nseg, kJoin, p.scan_in_kernel, i, c16, v);
                if (CAUSAL) tmem_st16(tS + lane_off + c16 * 16, v);
                store_state_row<D>(sbf, i, v, c16);
            }
            float zv[16];
            zv[0] = seg_state_z<D>(state_head, seg, p.nseg, kJoin, p.scan_in_kernel, i);
#pragma unroll
            for (int e = 1; e < 16; ++e) zv[e] = 0.f;
            if (CAUSAL) {
                tmem_st16(tS + lane_off + D, zv);
                tmem_st_wait();
            }
            store_z_split(ztile, i, zv[0]);
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive_warp(&bar_sbf);
        if (CAUSAL) {
            bool ok = true;
            float rs_cur = 0.f;   // fp32 row sum of mask(A) of the chunk last converted
            auto p_conv = [&](int k) {
                ok = ok && warp_wait(&bar_afull, k & 1, &abort_flag);
                tc_fence_after();
                if (i == 0) LA_TL(k, 8);
                float rs = 0.f;
                if (ok) {
#pragma unroll
                    for (int c32 = 0; c32 < (C + 31) / 32; ++c32) {
                        float v[32];
                        if (C >= 32) {
                            tmem_ld32(tA + lane_off + c32 * 32, v);
                        } else {
                            tmem_ld16(tA + lane_off, v);
                        }
                        tmem_wait_regs<(C >= 32 ? 32 : 16)>(v);
#pragma unroll
                        for (int h = 0; h < (C >= 32 ? 2 : 1); ++h) {
                            uint32_t w[8];
                            float pair[8];
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                const int j = c32 * 32 + h * 16 + e;
                                const float a0 = (j <= ti) ? v[h * 16 + e] : 0.f, a1 = (j + 1 <= ti) ? v[h * 16 + e + 1] : 0.f;
                                pair[e / 2] = a0 + a1;
                                w[e / 2] = pack_bf16x2(a0, a1);
                            }
                            rs += ((pair[0] + pair[1]) + (pair[2] + pair[3])) + ((pair[4] + pair[5]) + (pair[6] + pair[7]));
                            const int c16 = c32 * 2 + h;
                            uint8_t *p0 = pbuf + swz_chunk(128, i, 2 * c16), *p1 = pbuf + swz_chunk(128, i, 2 * c16 + 1);
                            if (LA_CHECK(in_smem(p0, 16, sm_lo, sm_hi) && in_smem(p1, 16, sm_lo, sm_hi), 241,
                                         smem_u32(p0) - sm_lo, c16)) {
                                *reinterpret_cast<uint4 *>(p0) = make_uint4(w[0], w[1], w[2], w[3]);
                                *reinterpret_cast<uint4 *>(p1) = make_uint4(w[4], w[5], w[6], w[7]);
                            }
                        }
                    }
                    fence_proxy_async();
                }
                rs_cur = rs;
                tc_fence_before();
                if (i == 0) LA_TL(k, 9);
                mbar_arrive_warp(&bar_pready);
            };
            // the backward's den of chunk k: phi(q) . z (columns D, D + 1 of chunk k's O buffer,
            // read once its products are done and before this warpgroup's next state conversion
            // lets chunk k + 2 reuse the buffer) plus this thread's fp32 row sum of mask(A)
            auto write_den = [&](int k, float rsum) {
                float dz[2] = {0.f, 0.f};
                if (ok) {
                    tmem_ld2((k % NO ? tO1 : tO0) + lane_off + D, dz);
                    tmem_wait_regs<2>(dz);
                }
                const int t = t0 + k * C + ti;
                if (ok && p.den && t < t1 && i / C < gr) {
                    float *dp = p.den + (size_t)(bh0 + i / C) * p.den_stride + t;
                    if (WT && p.pass == 2)   // the sin terms onto the cos pass's den (which has eps)
                        *dp += (dz[0] + dz[1]) + rsum;
                    else
                        *dp = (dz[0] + dz[1]) + rsum + p.eps;
                }
            };
            if (nchunk > 0) p_conv(0);
            for (int k = 0; k < nchunk; ++k) {
                // S, z after chunk k -> operand tiles for chunk k + 1
                ok = ok && warp_wait(&bar_sfull, k & 1, &abort_flag);
                tc_fence_after();
                if (i == 0) LA_TL(k, 10);
                if (ok && wq * 32 < D) {
#pragma unroll 1
                    for (int c32 = 0; c32 < D / 32; ++c32) {
                        float v[32];
                        tmem_ld32(tS + lane_off + c32 * 32, v);
                        tmem_wait_regs<32>(v);
#pragma unroll
                        for (int h = 0; h < 2; ++h) store_state_row<D>(sbf, i, v + 16 * h, c32 * 2 + h);
                    }
                    float zd = tmem_ld1(tS + lane_off + D);
                    tmem_wait_regs<1>(&zd);
                    store_z_split(ztile, i, zd);
                }
                fence_proxy_async();
                tc_fence_before();
                if (i == 0) LA_TL(k, 11);
                mbar_arrive_warp(&bar_sbf);
                if (k + 1 < nchunk) {
                    ok = ok && warp_wait(&bar_ofull[k % NO], (k / NO) & 1, &abort_flag);
                    tc_fence_after();
                    write_den(k, rs_cur);
                    p_conv(k + 1);
                }
            }
            if (nchunk > 0) {
                ok = ok && warp_wait(&bar_ofull[(nchunk - 1) % NO], ((nchunk - 1) / NO) & 1, &abort_flag);
                tc_fence_after();
                write_den(nchunk - 1, rs_cur);
            }
        }
    } else if (warp >= 12 && warp < 16) {
        // ---------------- epilogue (thread = query row of the chunk): out = O / (den + eps),
        // staged in shared memory 64 columns at a time and written by TMA
        const int i = threadIdx.x - 384;
        const int wq = warp % 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        bool ok = true;
        for (int k = 0; k < nchunk; ++k) {
            const int o = k % NO;
            const uint32_t tO = o ? tO1 : tO0;
            const int c0 = t0 + k * C;
            ok = ok && warp_wait(&bar_ofull[o], (k / NO) & 1, &abort_flag);
            tc_fence_after();
            if (i == 0) LA_TL(k, 12);
            const bool rowok = c0 + i % C < t1 && i / C < gr;
            const size_t rg = (size_t)(bh0 + i / C) * p.N + (c0 + i % C);   // the row's index (when rowok)
            if constexpr (WT)   // sin pass: the next chunk's cos partials (one contiguous block a head)
                if (p.pass == 2 && i == 0 && k + 1 < nchunk)   // into L2 while this chunk is written out
                    for (int r = 0; r < gr; ++r)
                        prefetch_l2_bulk(p.part_num + blocked_index(bh0 + r, c0 + C, 0, p.N, D, C), (uint32_t)(D * C * 4));
            float pden = 0.f;   // sin pass: the cos terms' den of the row
            if constexpr (WT)
                if (p.pass == 2 && ok && rowok) pden = p.part_den[rg];
            float den = 0.f;
            if (ok) {
                float dz[4];   // phi(q) . z_hi, phi(q) . z_lo, P 1 (bf16 P), unused
                tmem_ld4(tO + lane_off + D, dz);
                tmem_wait_regs<4>(dz);
                den = (dz[0] + dz[1]) + dz[2];
                // bidirectional: the backward's den (causal: written by the P conversion warps;
                // the sin pass adds its terms to the cos pass's)
                if (!CAUSAL && p.den && rowok) {
                    float *dp = p.den + (size_t)(bh0 + i / C) * p.den_stride + c0 + i % C;
                    if (WT && p.pass == 2)
                        *dp += den;
                    else
                        *dp = den + p.eps;
                }
            }
            if constexpr (WT) {
                if (p.pass == 1) {   // cos pass: the row's numerator (fp32, unnormalised) and den
#pragma unroll 1
                    for (int c32 = 0; c32 < D / 32; ++c32) {
                        float v[32];
                        if (ok) {
                            tmem_ld32(tO + lane_off + c32 * 32, v);
                            tmem_wait_regs<32>(v);
                        }
                        if (ok && rowok) {   // chunk-blocked: a warp's rows form one run per column
                            float *dst = p.part_num + blocked_index(bh0 + i / C, c0 + i % C, c32 * 32, p.N, D, C);
#pragma unroll
                            for (int e = 0; e < 32; ++e) dst[(size_t)e * C] = v[e];
                        }
                    }
                    if (ok && rowok) p.part_den[rg] = den;
                    tc_fence_before();
                    mbar_arrive_warp(&bar_ofree[o]);
                    continue;
                }
            }
            const float inv = 1.f / (den + pden + p.eps);
#pragma unroll 1
            for (int c64 = 0; c64 < D / 64; ++c64) {
                float v[32];   // 32 columns at a time
                if (ok) {
                    tmem_ld32(tO + lane_off + c64 * 64, v);
                    tmem_wait_regs<32>(v);
                }
                if (i < 32) {   // previous stores (lane 0's) have read the staging tile
                    bulk_wait_read();
                    __syncwarp();
                }
                named_barrier(2, 128);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (ok && hh == 1) {
                        tmem_ld32(tO + lane_off + c64 * 64 + 32, v);
                        tmem_wait_regs<32>(v);
                    }
                    if constexpr (WT) {   // sin pass: plus the cos terms' numerator; the float32
                                          // output row goes back in its place (the backward's h)
                        if (p.pass == 2 && ok && rowok) {   // (every load before any store)
                            float *src = p.part_num + blocked_index(bh0 + i / C, c0 + i % C, c64 * 64 + hh * 32, p.N, D, C);
                            float a[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) a[e] = src[(size_t)e * C];
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                v[e] += a[e];
                                src[(size_t)e * C] = v[e] * inv;
                            }
                        }
                    }
                    if (ok) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 w;
                            w.x = pack_bf16x2(v[8 * q + 0] * inv, v[8 * q + 1] * inv);
                            w.y = pack_bf16x2(v[8 * q + 2] * inv, v[8 * q + 3] * inv);
                            w.z = pack_bf16x2(v[8 * q + 4] * inv, v[8 * q + 5] * inv);
                            w.w = pack_bf16x2(v[8 * q + 6] * inv, v[8 * q + 7] * inv);
                            *reinterpret_cast<uint4 *>(obuf + swz_chunk(128, i, hh * 4 + q)) = w;
                        }
                    }
                }
                fence_proxy_async();
                named_barrier(2, 128);
                if (i < 32 && ok) {   // the first warp, lane 0 issuing
                    for (int r = 0; r < gr; ++r) tma_store_3d_w(&map_o, obuf + r * C * 128, c64 * 64, c0, bh0 + r);
                    bulk_commit();
                }
            }
            tc_fence_before();
            if (i == 0) LA_TL(k, 13);
            mbar_arrive_warp(&bar_ofree[o]);
        }
        if (i < 32) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (threadIdx.x == 0 && abort_flag) atomicExch(p.err, kErrTimeout);
    LA_SPAN(1, 1);
}

// ---------------------------------------------------------------------------------------
// Host side

template <int D, bool WT>
cudaError_t launch_state(const Params &p, cudaStream_t s) {
    CUtensorMap mk{}, mv{};
    cudaError_t e = make_map_in(&mk, p.k, p.B, p.Hkv, p.N, D, p.st_k, StateCfg<D>::C);
    if (e == cudaSuccess) e = make_map_in(&mv, p.v, p.B, p.Hkv, p.N, D, p.st_v, StateCfg<D>::C);
    if (e == cudaSuccess) e = prepare(k_tc_state<D, WT>, StateCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    TraceScope ts("tc_seg_state", s);
    return launch_pdl(k_tc_state<D, WT>, dim3(p.B * p.Hkv * p.nseg), dim3(kStateThreads), StateCfg<D>::SMEM, s, mk, mv, p);
}

template <int D, int G, bool CAUSAL, bool MASK, bool WT>
cudaError_t launch_fwd(const Params &p, cudaStream_t s) {
    using K = FwdCfg<D, G>;
    CUtensorMap mq{}, mk{}, mv{}, mo{};
    cudaError_t e = make_map_in(&mq, p.q, p.B, p.Hq, p.N, D, p.st_q, K::C);
    if (e == cudaSuccess) e = make_map_in(&mk, p.k, p.B, p.Hkv, p.N, D, p.st_k, K::C);
    if (e == cudaSuccess) e = make_map_in(&mv, p.v, p.B, p.Hkv, p.N, D, p.st_v, K::C);
    if (e == cudaSuccess) e = make_map(&mo, p.out, p.B * p.Hq, p.N, D, K::C);
    if (e == cudaSuccess) e = prepare(k_tc_fwd<D, G, CAUSAL, MASK, WT>, K::SMEM);
    if (e != cudaSuccess) return e;
    TraceScope ts(CAUSAL ? "tc_fwd_causal" : "tc_fwd_bidir", s);
    return launch_pdl(k_tc_fwd<D, G, CAUSAL, MASK, WT>, dim3(p.B * p.Hkv * p.nseg), dim3(kFwdThreads), K::SMEM, s, mq, mk, mv,
                      mo, p);
}

// The forward with cos/sin weights (the cosFormer modulation of the linear_attn page:
// W_ij = c_i c_j + s_i s_j) as two passes of the one-term kernels, each with its own (S, z)
// and the features c_t phi(x_t), then s_t phi(x_t): out = (num_c + num_s) / (den_c + den_s +
// eps).  The cos pass leaves num_c and den_c (fp32) in the workspace; the sin pass adds them
// in its epilogue, and leaves the float32 output rows where num_c was (the backward's h =
// -g . out).  Each pass's states sit in their own half of the state array; the den left for
// the backward (incl. eps) is the cos pass's plus the sin pass's.
template <int D, int G, bool MASK>
cudaError_t forward_two_pass(const Params &p, cudaStream_t s) {
    const size_t pass_elems = (size_t)p.B * p.Hkv * p.nseg * D * (D + 1);
    cudaError_t e = cudaSuccess;
    for (int pass = 1; pass <= 2 && e == cudaSuccess; ++pass) {
        Params pp = p;
        pp.pass = pass;
        pp.wrow = pass == 1 ? p.cw : p.sw;
        pp.state = p.state + (size_t)(pass - 1) * pass_elems;
        e = launch_state<D, true>(pp, s);
        if (e == cudaSuccess && !pp.scan_in_kernel)
            e = scan_segments(pp.state, pp, pp.causal ? kScanPrefix : kScanTotal, (size_t)D * (D + 1), s);
        if (e == cudaSuccess)
            e = pp.causal ? launch_fwd<D, G, true, MASK, true>(pp, s) : launch_fwd<D, G, false, MASK, true>(pp, s);
    }
    return e;
}

template <int D, int G, bool MASK = false>
cudaError_t forward_dg(const Params &p, cudaStream_t s) {
    if (p.P == 2) {
        if (!p.cw || !p.sw || !p.part_num || !p.part_den) return cudaErrorInvalidValue;
        return forward_two_pass<D, G, MASK>(p, s);
    }
    cudaError_t e = launch_state<D, false>(p, s);
#ifdef LA_DEBUG
    const char *stop = getenv("LA_DEBUG_STOP");
    if (stop && stop[0] == 's' && stop[1] == 't') return e;      // "state"
#endif
    if (e == cudaSuccess && !p.scan_in_kernel)
        e = scan_segments(p.state, p, p.causal ? kScanPrefix : kScanTotal, (size_t)D * (D + 1), s);
#ifdef LA_DEBUG
    if (stop && stop[0] == 's' && stop[1] == 'c') return e;      // "scan"
#endif
    if (e != cudaSuccess) return e;
    return p.causal ? launch_fwd<D, G, true, MASK, false>(p, s) : launch_fwd<D, G, false, MASK, false>(p, s);
}

template <int D>
cudaError_t forward_d(const Params &p, cudaStream_t s) {
    switch (p.n_rep) {
        case 1:   // D = 128: the n_rep = 2 tiles with half the rows masked (see k_tc_fwd)
            if constexpr (D == 64) return forward_dg<D, 1>(p, s);
            else return forward_dg<D, 2, true>(p, s);
        case 2: return forward_dg<D, 2>(p, s);
        case 4: return forward_dg<D, 4>(p, s);
        case 8: return forward_dg<D, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

// Tokens per chunk of the forward's tiles (the plan's chunk): 128 / n_rep, except for D = 128
// with n_rep = 1, whose one head takes half of the n_rep = 2 tiles.
int tc_chunk(int n_rep, int D) { return D == 128 && n_rep == 1 ? 64 : 128 / n_rep; }

bool tc_supported(int Hq, int Hkv, int N, int D, la_dtype dt, int P, int causal, int is_bwd) {
    (void)N;
    (void)causal;
    if (dt != LA_BF16 || (P != 1 && P != 2)) return false;
    const int n_rep = Hq / Hkv;
    if (is_bwd) return tc_bwd_supported(n_rep, D);
    return (D == 64 || D == 128) && (n_rep == 1 || n_rep == 2 || n_rep == 4 || n_rep == 8);
}

cudaError_t tc_forward(const Params &p, cudaStream_t s) {
    return p.D == 128 ? forward_d<128>(p, s) : (p.D == 64 ? forward_d<64>(p, s) : cudaErrorNotSupported);
}


}  // namespace la

#ifdef LA_TEST_HOOKS
// Test builds only: arm (1) or disarm (0) the withheld arrival of k_tc_fwd.
extern "C" int la_test_withhold_arrival(int on) {
    return cudaMemcpyToSymbol(la::g_la_test_skip, &on, sizeof(int)) == cudaSuccess ? 0 : 1;
}
#endif

#ifdef LA_TIMELINE
// Timeline builds only: copy out the forward kernel's event clocks ([64][16] long long).
extern "C" int la_timeline_read(long long *out) {
    return cudaMemcpyFromSymbol(out, la::g_la_tl, sizeof(long long) * 64 * 16) == cudaSuccess ? 0 : 1;
}
// ... and the per-block entry and exit times of this file's kernels ([4][256][2], ns).
extern "C" int la_timeline_read_span(unsigned long long *out) {
    return cudaMemcpyFromSymbol(out, la::g_la_span, sizeof(unsigned long long) * 4 * 256 * 2) == cudaSuccess ? 0 : 1;
}
#endif

#ifdef LA_DEBUG
// Debug builds only: copy out and clear the first failed self-check (id, a, b, block).
extern "C" int la_debug_read(int *out4) {
    if (cudaMemcpyFromSymbol(out4, la::g_la_debug, 4 * sizeof(int)) != cudaSuccess) return 1;
    const int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(la::g_la_debug, zero, 4 * sizeof(int)) == cudaSuccess ? 0 : 1;
}
#endif
