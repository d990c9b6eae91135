// la_lowrank.cu -- the low-rank projection on tensor cores (tcgen05 / TMEM / TMA):
//
//   y = (x V^T) U^T + bias        (module neuralops.core.triton_kernels.low_rank, `fwd`)
//
// with x [M, K_in], V [r, K_in], U [K_out, r], bias [K_out] (bf16, row-major), and its
// gradient (the page's `bwd` differentiates `fwd`):
//
//   t = x V^T,  dt = g U,  dx = dt V,  dU = g^T t,  dV = dt^T x,  dbias = sum_m g[m].
//
// One kernel template does the two chained products of a 128-row tile of A1 [M, K1]:
//
//   T = A1 B1^T  (fp32 in TMEM, K1 in 64-column blocks)  ->  bf16 T in shared memory
//   Y = T B2^T (+ bias)  (fp32 in TMEM, 128 output columns at a time)  ->  bf16 Y by TMA
//
// so the rank-r bottleneck T never leaves the SM.  B1 is [R, K1] (K-major) or [K1, R]
// (MN-major: the same bytes read as rows of K), likewise B2 is [N2, R] or [R, N2]; the
// forward takes x, V, U as they are (both K-major), the backward's dx = (g U) V takes U and
// V as MN-major operands and also stores T (= dt) for the weight gradients.  The weight
// gradients dU = g^T t and dV = dt^T x reduce over the M rows: a second kernel sums them in
// row slices (fp32 partials in the workspace) and a fixed-order reduction finishes them, so
// results never depend on scheduling.
//
// Warp roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM owner, warps
// 4-7 epilogue (thread = row of the tile).  Every wait is bounded; a wait that runs out
// raises the block's abort flag and the call reports LA_ERR_TIMEOUT through la_get_status.
#include "la_tc_common.cuh"

namespace la {
namespace {

constexpr int kLrThreads = 256;
constexpr int kLrChainThreads = 384;   // chain kernel: warp 0 TMA, warp 1 MMA, warps 4-11 epilogue

// 2-D map over a row-major bf16 matrix [rows][cols]: box {64 columns, box_rows rows},
// 128-byte swizzle; elements past either edge read as zeros.
cudaError_t make_map_2d(CUtensorMap *map, const void *ptr, int rows, int cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// RP: the inner (rank) dimension padded to a multiple of 64, at most 256.
template <int RP, bool B1_MN, bool B2_MN>
struct ChainCfg {
    static constexpr int RB = RP / 64;                        // 64-wide rank blocks
    static constexpr int A_BYTES = 128 * 64 * 2;              // A1 block: 128 rows x 64 columns of K1
    static constexpr int B1_BYTES = RP * 64 * 2;              // B1 block: RP x 64 (either layout)
    static constexpr int B2_BYTES = 128 * 64 * 2;             // B2 block: 128 outputs x 64 rank columns
    static constexpr int STAGE = A_BYTES + (B1_BYTES > B2_BYTES ? B1_BYTES : B2_BYTES);
    static constexpr int TBF_BYTES = 128 * RP * 2;            // T (bf16): 128 rows x RP, K-major
    static constexpr int OUT_BYTES = 2 * 128 * 32 * 2;        // Y staging: two tiles of 128 rows x 32 columns
    static constexpr int FIXED = TBF_BYTES + OUT_BYTES + 1024;
    static constexpr int NS = (kSmemLimit - 1024 - FIXED) / STAGE > 4 ? 4 : (kSmemLimit - 1024 - FIXED) / STAGE;
    static constexpr int SMEM = NS * STAGE + FIXED;
    static_assert(NS >= 2, "two pipeline stages");
    // the second product's B2 blocks are small: a stage carries BPS of them, so that as many
    // bytes are in flight as in the first product (the ring runs into L2 latency otherwise)
    static constexpr int BPS = STAGE / B2_BYTES;
    // TMEM: T in [0, RP); four Y buffers of 128 columns: 256, 384 and, once T has been copied
    // out in bf16 (until the next tile's first product), 0 and 128
    static constexpr int T_T = 0;
    static constexpr int NY = 4;
    __host__ __device__ static constexpr int t_y(int b) { return b == 0 ? 256 : b == 1 ? 384 : b == 2 ? 0 : 128; }
};

struct ChainArgs {
    int M, K1, R, N2;      // A1 [M, K1], the rank R (<= RP), N2 output columns
    const void *bias;      // [N2] bf16 or null
    int write_t, write_y;  // which products leave the SM
    int *err;
    void *y;               // [M, N2] bf16, written row by row from the epilogue (set by launch_chain)
};

template <int RP, bool B1_MN, bool B2_MN>
__global__ void __launch_bounds__(kLrChainThreads, 1) k_lr_chain(const __grid_constant__ CUtensorMap map_a1,
                                                             const __grid_constant__ CUtensorMap map_b1,
                                                             const __grid_constant__ CUtensorMap map_b2,
                                                             const __grid_constant__ CUtensorMap map_t, ChainArgs a) {
    using K = ChainCfg<RP, B1_MN, B2_MN>;
    constexpr int NS = K::NS;
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();
    __shared__ uint64_t bar_full[NS], bar_empty[NS], bar_tfull, bar_tbf, bar_yfull[K::NY], bar_yfree[K::NY], bar_fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    uint8_t *tbf = stage0 + NS * K::STAGE;
    uint8_t *obuf = tbf + K::TBF_BYTES;
    const int warp = threadIdx.x / 32;
    const int ntiles = (a.M + 127) / 128;
    const int nk1 = (a.K1 + 63) / 64;
    const int nn2 = a.write_y ? (a.N2 + 127) / 128 : 0;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        mbar_init(&bar_tfull, 1);
        mbar_init(&bar_tbf, 128);
        for (int b = 0; b < K::NY; ++b) {
            mbar_init(&bar_yfull[b], 1);
            mbar_init(&bar_yfree[b], 128);
        }
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
    const uint32_t tT = tmem_base + K::T_T;

    if (warp == 0) {
        // ---------------- TMA producer: per tile, the K1 blocks of A1 and B1, then the
        // (output tile, rank block) blocks of B2, all through one ring of stages
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
            for (int kb = 0; ok && kb < nk1; ++kb, ++it) {
                const int s = it % NS;
                if (it >= NS && !warp_wait(&bar_empty[s], ((it / NS) - 1) & 1, &abort_flag)) { ok = false; break; }
                uint8_t *st = stage0 + s * K::STAGE;
                if (tile == blockIdx.x) LA_TL(kb, 0);
                mbar_arrive_expect_tx_w(&bar_full[s], K::A_BYTES + K::B1_BYTES);
                tma_load_2d_w(st, &map_a1, &bar_full[s], kb * 64, tile * 128);
                if (B1_MN)   // B1 stored [K1][R]: RP/64 boxes of 64 K rows x 64 rank columns
                    for (int rb = 0; rb < K::RB; ++rb)
                        tma_load_2d_w(st + K::A_BYTES + rb * 64 * 128, &map_b1, &bar_full[s], rb * 64, kb * 64);
                else         // B1 stored [R][K1]: one box of RP rows x 64 K columns
                    tma_load_2d_w(st + K::A_BYTES, &map_b1, &bar_full[s], kb * 64, 0);
            }
            // B2 blocks bi = nt RB + rb (output tile nt, rank block rb), BPS to a stage
            const int nb2 = nn2 * K::RB;
            for (int b0 = 0; ok && b0 < nb2; b0 += K::BPS, ++it) {
                const int s = it % NS;
                if (it >= NS && !warp_wait(&bar_empty[s], ((it / NS) - 1) & 1, &abort_flag)) { ok = false; break; }
                const int nb = nb2 - b0 < K::BPS ? nb2 - b0 : K::BPS;
                mbar_arrive_expect_tx_w(&bar_full[s], nb * K::B2_BYTES);
                for (int j = 0; j < nb; ++j) {
                    const int nt = (b0 + j) / K::RB, rb = (b0 + j) % K::RB;
                    uint8_t *st = stage0 + s * K::STAGE + j * K::B2_BYTES;
                    if (B2_MN)   // B2 stored [R][N2]: two boxes of 64 rank rows x 64 output columns
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d_w(st + h * 64 * 128, &map_b2, &bar_full[s], nt * 128 + h * 64, rb * 64);
                    else         // B2 stored [N2][R]: one box of 128 output rows x 64 rank columns
                        tma_load_2d_w(st, &map_b2, &bar_full[s], rb * 64, nt * 128);
                }
            }
        }
        // drain the copies still in flight
        for (int j = it > NS ? it - NS : 0; j < it; ++j) warp_drain(&bar_full[j % NS], (j / NS) & 1);
    } else if (warp == 1) {
        // ---------------- MMA issuer
        constexpr uint32_t id1 = idesc_bf16(128, RP, false, B1_MN);
        constexpr uint32_t id2 = idesc_bf16(128, 128, false, B2_MN);
        const uint32_t tb = smem_u32(tbf);
        int it = 0, yc = 0, tc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++tc) {
            // T's columns are free once the epilogue has read the previous tile's T (tbf) and
            // the Y buffers 2 and 3 that lie in them (their last uses)
            if (tc > 0 && !warp_wait(&bar_tbf, (tc - 1) & 1, &abort_flag)) break;
            for (int b = 2; b < K::NY && ok; ++b) {
                const int uses = yc > b ? (yc - 1 - b) / K::NY + 1 : 0;
                if (uses > 0 && !warp_wait(&bar_yfree[b], (uses - 1) & 1, &abort_flag)) ok = false;
            }
            if (!ok) break;
            tc_fence_after();
            for (int kb = 0; kb < nk1; ++kb, ++it) {
                const int s = it % NS;
                if (!warp_wait(&bar_full[s], (it / NS) & 1, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (tc == 0) LA_TL(kb, 1);
                const uint32_t as = smem_u32(stage0 + s * K::STAGE), bs = as + K::A_BYTES;
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd = B1_MN ? desc_mnmajor(bs, 64, 0, kk) : desc_kmajor(bs, RP, 0, kk);
                    mma_bf16_w(tT, desc_kmajor(as, 128, 0, kk), bd, id1, (kb > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit_w(&bar_empty[s]);
            }
            if (!ok) break;
            mma_commit_w(&bar_tfull);
            if (tc == 0) LA_TL(0, 7);
            if (nn2 == 0) continue;
            if (!warp_wait(&bar_tbf, tc & 1, &abort_flag)) break;   // bf16 T is in shared memory
            tc_fence_after();
            if (tc == 0) LA_TL(1, 7);
            // B2 blocks as the producer packs them: BPS to a stage, output tile nt = bi / RB
            // accumulating into Y buffer yc % NY over its RB rank blocks
            const int nb2 = nn2 * K::RB;
            for (int b0 = 0; ok && b0 < nb2; b0 += K::BPS, ++it) {
                const int s = it % NS;
                if (!warp_wait(&bar_full[s], (it / NS) & 1, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                const int nb = nb2 - b0 < K::BPS ? nb2 - b0 : K::BPS;
                for (int j = 0; j < nb; ++j) {
                    const int rb = (b0 + j) % K::RB, yb = yc % K::NY;
                    const uint32_t tY = tmem_base + K::t_y(yb);
                    if (rb == 0) {   // a new output tile: its Y buffer must have been read
                        if (yc >= K::NY && !warp_wait(&bar_yfree[yb], ((yc / K::NY) - 1) & 1, &abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        if (tc == 0) LA_TL((b0 + j) / K::RB, 2);
                    }
                    const uint32_t bs = smem_u32(stage0 + s * K::STAGE + j * K::B2_BYTES);
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = B2_MN ? desc_mnmajor(bs, 64, 0, kk) : desc_kmajor(bs, 128, 0, kk);
                        mma_bf16_w(tY, desc_kmajor(tb, 128, 0, rb * 4 + kk), bd, id2, (rb > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (rb == K::RB - 1) {
                        mma_commit_w(&bar_yfull[yb]);
                        if (tc == 0) LA_TL((b0 + j) / K::RB, 3);
                        ++yc;
                    }
                }
                mma_commit_w(&bar_empty[s]);
            }
        }
        mma_commit_w(&bar_fin);
        warp_drain(&bar_fin, 0);
    } else if (warp >= 4) {
        // ---------------- epilogue: two warpgroups, thread i = row i of the tile (TMEM lane i).
        // Group 0 (warps 4-7) turns T into its bf16 copy (and writes T out when asked); group g
        // takes the output tiles of Y buffers g and g + 2 (yc % 4 of parity g), so two output
        // tiles are written out at once while the MMA runs up to two more ahead.
        const int grp = (warp - 4) / 4, wq = warp % 4;
        const int i = wq * 32 + threadIdx.x % 32, lane = threadIdx.x % 32;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        uint8_t *stg = obuf + grp * (K::OUT_BYTES / 2);   // this group's staging: 128 rows x 32 columns
        int yc = 0, tc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tc) {
            if (grp == 0) {
                ok = ok && warp_wait(&bar_tfull, tc & 1, &abort_flag);
                tc_fence_after();
                if (a.write_t && tc > 0) {   // the previous tile's copies of T have read the bf16 tile
                    if (i < 32) bulk_wait_read();
                    named_barrier(2, 128);
                }
                // T (fp32) -> bf16 T in shared memory (the operand of the second product), and
                // when asked, out to global memory from there
#pragma unroll 1
                for (int c16 = 0; c16 < RP / 16; ++c16) {
                    float v[16];
                    if (ok) {
                        tmem_ld16(tT + lane_off + c16 * 16, v);
                        tmem_wait_regs<16>(v);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = 0.f;
                    }
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                    *reinterpret_cast<uint4 *>(tbf + swz_chunk(128, i, 2 * c16)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(tbf + swz_chunk(128, i, 2 * c16 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                tc_fence_before();
                fence_proxy_async();
                if (tc == 0 && i == 0) LA_TL(2, 7);
                mbar_arrive_warp(&bar_tbf);
                if (a.write_t) {   // T leaves from the bf16 copy, every 64-column block at once
                    named_barrier(2, 128);
                    if (ok && i < 32) {
                        for (int rb = 0; rb < (a.R + 63) / 64; ++rb)
                            tma_store_2d_w(&map_t, tbf + rb * 128 * 128, rb * 64, tile * 128);
                        bulk_commit();
                    }
                    __syncwarp();
                }
            }
            for (int nt = 0; nt < nn2; ++nt, ++yc) {
                const int yb = yc % K::NY;
                if ((yb & 1) != grp) continue;
                const uint32_t tY = tmem_base + K::t_y(yb);
                // the tile's 128 bias values before the wait for its products: their loads (L2
                // latency, which each 32-column piece exposed) overlap the wait and the TMEM reads
                uint4 bias16[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    bias16[q] = a.bias && nt * 128 + 8 * q < a.N2
                                    ? __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.bias) + nt * 128 + 8 * q))
                                    : make_uint4(0u, 0u, 0u, 0u);
                ok = ok && warp_wait(&bar_yfull[yb], (yc / K::NY) & 1, &abort_flag);
                tc_fence_after();
                if (tc == 0 && i == 0) LA_TL(nt, 4);
                // 32 columns at a time: thread i (row i) writes its 64 bytes into the staging tile
                // (rows in pairs of 128-byte swizzled lines), then each warp copies 8 rows per
                // store instruction, whole 64-byte row pieces.  (A TMA store out of a staging tile
                // queued behind this SM's loads of the next blocks, and a store per thread per
                // row wrote partial lines: 10 k and 7 k cycles per output tile, measured.)
#pragma unroll
                for (int c32 = 0; c32 < 4; ++c32) {
                    const int col0 = nt * 128 + c32 * 32;
                    float v[32];
                    if (ok) {
                        tmem_ld32(tY + lane_off + c32 * 32, v);
                        tmem_wait_regs<32>(v);
                    }
                    if (c32 == 3) {   // every column of this Y buffer is in registers
                        tc_fence_before();
                        mbar_arrive_warp(&bar_yfree[yb]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t *bw = reinterpret_cast<const uint32_t *>(&bias16[c32 * 4 + q]);
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16x2(bw[e]);
                            w[e] = pack_bf16x2(v[8 * q + 2 * e] + f.x, v[8 * q + 2 * e + 1] + f.y);
                        }
                        // row i: line i / 2, chunks (i % 2) 4 + q, swizzled by the line
                        *reinterpret_cast<uint4 *>(stg + swz_chunk(64, i >> 1, (i & 1) * 4 + q)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    named_barrier(2 + grp, 128);
                    // warp wq copies rows wq 32 .. + 31: lane l takes 16-byte piece l % 4 of row
                    // 8 r + l / 4 of its block, r = 0 .. 3
                    const int piece = lane % 4, c = col0 + piece * 8;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int rr = wq * 32 + 8 * r + lane / 4, row = tile * 128 + rr;
                        const uint4 w = *reinterpret_cast<const uint4 *>(stg + swz_chunk(64, rr >> 1, (rr & 1) * 4 + piece));
                        if (ok && row < a.M && c < a.N2)
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.y) + (size_t)row * a.N2 + c) = w;
                    }
                    named_barrier(2 + grp, 128);   // the staging tile is read before the next piece
                }
                if (tc == 0 && i == 0) LA_TL(nt, 5);
            }
        }
        if (grp == 0 && i < 32) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (threadIdx.x == 0 && abort_flag) atomicExch(a.err, kErrTimeout);
}

template <int RP, bool B1_MN, bool B2_MN>
cudaError_t launch_chain(const void *a1, const void *b1, const void *b2, void *t, void *y, const ChainArgs &ca,
                         cudaStream_t s, const char *name) {
    using K = ChainCfg<RP, B1_MN, B2_MN>;
    CUtensorMap m_a1{}, m_b1{}, m_b2{}, m_t{};
    cudaError_t e = make_map_2d(&m_a1, a1, ca.M, ca.K1, 128);
    // B1 as stored: [R][K1] (box RP rows) or [K1][R] (box 64 rows)
    if (e == cudaSuccess) e = B1_MN ? make_map_2d(&m_b1, b1, ca.K1, ca.R, 64) : make_map_2d(&m_b1, b1, ca.R, ca.K1, RP);
    if (e == cudaSuccess && ca.write_y)
        e = B2_MN ? make_map_2d(&m_b2, b2, ca.R, ca.N2, 64) : make_map_2d(&m_b2, b2, ca.N2, ca.R, 128);
    if (e == cudaSuccess && ca.write_t) e = make_map_2d(&m_t, t, ca.M, ca.R, 128);
    if (e == cudaSuccess) e = prepare(k_lr_chain<RP, B1_MN, B2_MN>, K::SMEM);
    if (e != cudaSuccess) return e;
    ChainArgs a = ca;
    a.y = y;
    const int ntiles = (ca.M + 127) / 128;
    const int grid = ntiles < kPlanSms ? ntiles : kPlanSms;
    TraceScope ts(name, s);
    return launch_pdl(k_lr_chain<RP, B1_MN, B2_MN>, dim3(grid), dim3(kLrChainThreads), K::SMEM, s, m_a1, m_b1, m_b2, m_t, a);
}

template <bool B1_MN, bool B2_MN>
cudaError_t chain_dispatch(const void *a1, const void *b1, const void *b2, void *t, void *y, const ChainArgs &ca,
                           cudaStream_t s, const char *name) {
    const int rp = (ca.R + 63) / 64 * 64;
    switch (rp) {
        case 64: return launch_chain<64, B1_MN, B2_MN>(a1, b1, b2, t, y, ca, s, name);
        case 128: return launch_chain<128, B1_MN, B2_MN>(a1, b1, b2, t, y, ca, s, name);
        case 192: return launch_chain<192, B1_MN, B2_MN>(a1, b1, b2, t, y, ca, s, name);
        case 256: return launch_chain<256, B1_MN, B2_MN>(a1, b1, b2, t, y, ca, s, name);
        default: return cudaErrorNotSupported;
    }
}

// ---------------------------------------------------------------------------------------
// Weight gradients: C = A^T B summed over the M rows, A [M, Mc] and B [M, Nc] row-major (both
// read as MN-major operands: rows are the reduction index).  Grid: (Mc / 128) x (Nc / NT)
// output tiles x S row slices; each CTA sums its slice's rows into TMEM and writes an fp32
// partial tile; k_lr_reduce adds the S partials in slice order.  With ROWSUM the CTA also
// sums A over its rows (an N = 16 product against a ones tile): dbias = sum_m g[m].
constexpr int kWgNT = 256;   // output columns per tile

struct WgradArgs {
    int M, Mc, Nc, S, rows_per;   // rows_per: rows of one slice (a multiple of 64)
    float *part;                  // [S][Mc][Nc]
    float *rsum;                  // [S][Mc] (ROWSUM) or null
    int *err;
};

template <bool ROWSUM>
struct WgCfg {
    static constexpr int A_BYTES = 64 * 128 * 2;     // 64 rows x 128 columns (two 64-column blocks)
    static constexpr int B_BYTES = 64 * kWgNT * 2;   // 64 rows x 256 columns (four blocks)
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int ONES_BYTES = 16 * 128;      // 16 x 64 K-major, row 0 = 1
    static constexpr int NS = 4;
    static constexpr int SMEM = NS * STAGE + ONES_BYTES + 1024;
    static constexpr int T_C = 0, T_RS = kWgNT;      // TMEM: C tile, then the row sums (16 columns)
};

template <bool ROWSUM>
__global__ void __launch_bounds__(kLrThreads, 1) k_lr_wgrad(const __grid_constant__ CUtensorMap map_a,
                                                             const __grid_constant__ CUtensorMap map_b, WgradArgs w) {
    using K = WgCfg<ROWSUM>;
    constexpr int NS = K::NS;
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();
    __shared__ uint64_t bar_full[NS], bar_empty[NS], bar_done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t *stage0 = align1024(smem_raw);
    uint8_t *ones = stage0 + NS * K::STAGE;
    const int warp = threadIdx.x / 32;
    const int ntn = (w.Nc + kWgNT - 1) / kWgNT;
    const int sl = blockIdx.x % w.S, tile = blockIdx.x / w.S;
    const int nt = tile % ntn, mt = tile / ntn;
    const int m0 = sl * w.rows_per, m1 = min(w.M, m0 + w.rows_per);
    const int nblk = m1 > m0 ? (m1 - m0 + 63) / 64 : 0;

    if (ROWSUM) fill_ones_tile(ones, 64);
    fence_proxy_async();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        mbar_init(&bar_done, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tC = tmem_base + K::T_C, tRS = tmem_base + K::T_RS;

    if (warp == 0) {
        int issued = 0;
        for (int kb = 0; kb < nblk; ++kb) {
            const int s = kb % NS;
            if (kb >= NS && !warp_wait(&bar_empty[s], ((kb / NS) - 1) & 1, &abort_flag)) break;
            uint8_t *st = stage0 + s * K::STAGE;
            const int r0 = m0 + kb * 64;
            mbar_arrive_expect_tx_w(&bar_full[s], K::STAGE);
            for (int h = 0; h < 2; ++h) tma_load_2d_w(st + h * 64 * 128, &map_a, &bar_full[s], mt * 128 + h * 64, r0);
            for (int h = 0; h < kWgNT / 64; ++h)
                tma_load_2d_w(st + K::A_BYTES + h * 64 * 128, &map_b, &bar_full[s], nt * kWgNT + h * 64, r0);
            issued = kb + 1;
        }
        for (int j = issued > NS ? issued - NS : 0; j < issued; ++j) warp_drain(&bar_full[j % NS], (j / NS) & 1);
    } else if (warp == 1) {
        constexpr uint32_t idC = idesc_bf16(128, kWgNT, true, true);
        constexpr uint32_t idR = idesc_bf16(128, 16, true, false);
        const uint32_t on = smem_u32(ones);
        for (int kb = 0; kb < nblk; ++kb) {
            const int s = kb % NS;
            if (!warp_wait(&bar_full[s], (kb / NS) & 1, &abort_flag)) break;
            tc_fence_after();
            const uint32_t as = smem_u32(stage0 + s * K::STAGE), bs = as + K::A_BYTES;
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                const uint64_t ad = desc_mnmajor(as, 64, 0, kk);
                mma_bf16_w(tC, ad, desc_mnmajor(bs, 64, 0, kk), idC, acc);
                if (ROWSUM) mma_bf16_w(tRS, ad, desc_kmajor(on, 16, 0, 0), idR, acc);
            }
            mma_commit_w(&bar_empty[s]);
        }
        mma_commit_w(&bar_done);
        warp_drain(&bar_done, 0);
    } else if (warp >= 4) {
        // epilogue: thread i = row i of the C tile; fp32 partials to the workspace
        const int i = threadIdx.x - 128, wq = warp - 4;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const bool ok = warp_wait(&bar_done, 0, &abort_flag);
        tc_fence_after();
        const int row = mt * 128 + i;
        float *dst = w.part + ((size_t)sl * w.Mc + row) * (size_t)w.Nc;
#pragma unroll 1
        for (int c16 = 0; c16 < kWgNT / 16; ++c16) {
            float v[16];
            if (ok) {
                tmem_ld16(tC + lane_off + c16 * 16, v);
                tmem_wait_regs<16>(v);
            }
            if (!ok || row >= w.Mc) continue;
            const int col0 = nt * kWgNT + c16 * 16;
            for (int e = 0; e < 16; ++e)
                if (col0 + e < w.Nc) dst[col0 + e] = nblk > 0 ? v[e] : 0.f;
        }
        if (ROWSUM && nt == 0) {
            float v[16];
            if (ok) {
                tmem_ld16(tRS + lane_off, v);
                tmem_wait_regs<16>(v);
            }
            if (ok && row < w.Mc) w.rsum[(size_t)sl * w.Mc + row] = nblk > 0 ? v[0] : 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (threadIdx.x == 0 && abort_flag) atomicExch(w.err, kErrTimeout);
}

// out[e] = bf16(sum over the S slices of part[s][e]), slices in order (deterministic).
__global__ void k_lr_reduce(const float *part, int S, size_t elems, __nv_bfloat16 *out) {
    pdl_wait();
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < elems; e += (size_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < S; ++s) acc += part[(size_t)s * elems + e];
        out[e] = __float2bfloat16_rn(acc);
    }
}

// Slices of the M rows for a weight gradient: as many as keep the CTAs within one wave.
int wgrad_slices(int M, int tiles) {
    int S = kPlanSms / tiles;
    const int blocks = (M + 63) / 64;
    if (S > blocks) S = blocks;
    return S < 1 ? 1 : S;
}

// C = A^T B over M rows into bf16 `out` [Mc][Nc] (and, with rsum_out, the row sums of A).
cudaError_t wgrad(const void *A, const void *Bm, int M, int Mc, int Nc, float *part, float *rsum,
                  void *out, void *rsum_out, int *err, cudaStream_t s, const char *name) {
    CUtensorMap ma{}, mb{};
    cudaError_t e = make_map_2d(&ma, A, M, Mc, 64);
    if (e == cudaSuccess) e = make_map_2d(&mb, Bm, M, Nc, 64);
    const bool rs = rsum_out != nullptr;
    if (e == cudaSuccess) e = rs ? prepare(k_lr_wgrad<true>, WgCfg<true>::SMEM) : prepare(k_lr_wgrad<false>, WgCfg<false>::SMEM);
    if (e != cudaSuccess) return e;
    const int tiles = ((Mc + 127) / 128) * ((Nc + kWgNT - 1) / kWgNT);
    const int S = wgrad_slices(M, tiles);
    const int rows_per = ((M + S - 1) / S + 63) / 64 * 64;
    WgradArgs w{M, Mc, Nc, S, rows_per, part, rsum, err};
    {
        TraceScope ts(name, s);
        e = rs ? launch_pdl(k_lr_wgrad<true>, dim3(tiles * S), dim3(kLrThreads), WgCfg<true>::SMEM, s, ma, mb, w)
               : launch_pdl(k_lr_wgrad<false>, dim3(tiles * S), dim3(kLrThreads), WgCfg<false>::SMEM, s, ma, mb, w);
    }
    if (e != cudaSuccess) return e;
    TraceScope ts("lr_reduce", s);
    const size_t elems = (size_t)Mc * Nc;
    e = launch_pdl(k_lr_reduce, dim3(kPlanSms * 4), dim3(256), 0, s, (const float *)part, S, elems,
                   static_cast<__nv_bfloat16 *>(out));
    if (e == cudaSuccess && rs)
        e = launch_pdl(k_lr_reduce, dim3((unsigned)((Mc + 255) / 256)), dim3(256), 0, s, (const float *)rsum, S, (size_t)Mc,
                       static_cast<__nv_bfloat16 *>(rsum_out));
    return e;
}

}  // namespace

cudaError_t lowrank_forward(const void *x, const void *U, const void *V, const void *bias, void *y, void *t_out, int M,
                            int K_in, int r, int K_out, int *err, cudaStream_t s) {
    // t_out: the bf16 T = x V^T of the first product leaves the SM too (the backward's t)
    ChainArgs ca{M, K_in, r, K_out, bias, t_out ? 1 : 0, 1, err};
    return chain_dispatch<false, false>(x, V, U, t_out, y, ca, s, "lr_fwd");
}

size_t lowrank_bwd_workspace(int M, int K_in, int r, int K_out) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t tb = up((size_t)M * r * 2);   // t and dt, bf16 [M][r]
    const int su = wgrad_slices(M, ((K_out + 127) / 128) * ((r + kWgNT - 1) / kWgNT));
    const int sv = wgrad_slices(M, ((r + 127) / 128) * ((K_in + kWgNT - 1) / kWgNT));
    const size_t pu = up((size_t)su * K_out * r * 4) + up((size_t)su * K_out * 4);
    const size_t pv = up((size_t)sv * r * K_in * 4);
    return 2 * tb + (pu > pv ? pu : pv);
}

cudaError_t lowrank_backward(const void *x, const void *U, const void *V, const void *t_given, const void *g, void *dx,
                             void *dU, void *dV, void *dbias, int M, int K_in, int r, int K_out, void *ws, int *err,
                             cudaStream_t s) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    char *base = static_cast<char *>(ws);
    const void *t = t_given ? t_given : static_cast<const void *>(base);
    void *dt = base + up((size_t)M * r * 2);
    float *part = reinterpret_cast<float *>(base + 2 * up((size_t)M * r * 2));
    cudaError_t e = cudaSuccess;
    if (!t_given) {   // t = x V^T (kept for dU = g^T t), unless the forward left it
        ChainArgs ct{M, K_in, r, 0, nullptr, 1, 0, err};
        e = chain_dispatch<false, false>(x, V, nullptr, base, nullptr, ct, s, "lr_bwd_t");
    }
    // dt = g U (kept for dV = dt^T x), dx = dt V: U and V read as MN-major operands
    ChainArgs cx{M, K_out, r, K_in, nullptr, 1, 1, err};
    if (e == cudaSuccess) e = chain_dispatch<true, true>(g, U, V, dt, dx, cx, s, "lr_bwd_dx");
    // dU = g^T t (and dbias = the row sums of g), then dV = dt^T x
    if (e == cudaSuccess) {
        const int su = wgrad_slices(M, ((K_out + 127) / 128) * ((r + kWgNT - 1) / kWgNT));
        float *rsum = reinterpret_cast<float *>(reinterpret_cast<char *>(part) + up((size_t)su * K_out * r * 4));
        e = wgrad(g, t, M, K_out, r, part, rsum, dU, dbias, err, s, "lr_bwd_dU");
    }
    if (e == cudaSuccess) e = wgrad(dt, x, M, r, K_in, part, nullptr, dV, nullptr, err, s, "lr_bwd_dV");
    return e;
}

}  // namespace la

#ifdef LA_TIMELINE
// Timeline builds only: the low-rank chain kernel's event clocks ([64][16] long long).
extern "C" int la_timeline_read_lr(long long *out) {
    return cudaMemcpyFromSymbol(out, la::g_la_tl, sizeof(long long) * 64 * 16) == cudaSuccess ? 0 : 1;
}
#endif
