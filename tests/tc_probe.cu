// tc_probe.cu -- test-only probe of the tensor-core building blocks of the library: TMA
// tile loads with 128-byte swizzle, hand-swizzled tile writes, the K-major and MN-major
// shared-memory descriptors, the instruction descriptor, tcgen05.mma into TMEM and
// tcgen05.ld back out.  One CTA computes D[m][n] = sum_k A(m, k) B(n, k) for M = 128.
//
// A is given row-major as [M][K] (K-major) or [K][M] (MN-major); B as [N][K] (K-major)
// or [K][N] (MN-major).  With `collector` = 1 every K step is issued twice, first with A
// kept in the collector buffer and then taking A from it, into two accumulators (D is
// then [M][2N]: both halves must equal A B^T); with `collector` = 2 the second MMA has
// N = 16 and takes the first 16 rows (n) of B (D is [M][N + 16]).  `dcol` places the
// accumulator at that TMEM column of a 512-column allocation.  `b_off` (MN-major B only)
// starts B's descriptor `b_off` columns into its tile, inside the first 64-column block:
// B is then stored with N + b_off columns and the product uses columns b_off .. b_off+N-1.  Built by
// tests/test_gpu_tc_layouts.py into tests/_build.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "la_tc_ptx.cuh"

using namespace la::tc;

namespace {

constexpr int kSmemBytes = 200 * 1024;   // far more than the tiles need

__global__ void __launch_bounds__(128) probe_kernel(const __grid_constant__ CUtensorMap map_a,
                                                    const __grid_constant__ CUtensorMap map_b,
                                                    const __nv_bfloat16 *a_src, const __nv_bfloat16 *b_src,
                                                    float *d, int N, int K, int a_mn, int b_mn, int a_manual,
                                                    int b_manual, int collector, int dcol, int b_off, int *err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    const int M = 128;
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int rows_a = a_mn ? K : M, cols_a = a_mn ? M : K;
    const int rows_b = b_mn ? K : N, cols_b = b_mn ? N + b_off : K;
    const int nblk_a = (cols_a + 63) / 64, nblk_b = (cols_b + 63) / 64;
    uint8_t *tile_a = smem;
    uint8_t *tile_b = smem + nblk_a * rows_a * 128;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t ncols = 512;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot + (uint32_t)dcol;

    // unused columns of a partial block are zeroed so nothing undefined is ever read
    for (int i = threadIdx.x; i < (nblk_a * rows_a + nblk_b * rows_b) * 32; i += blockDim.x)
        reinterpret_cast<uint32_t *>(smem)[i] = 0u;
    fence_proxy_async();
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t bytes = 0;
        if (!a_manual) bytes += nblk_a * rows_a * 128;
        if (!b_manual) bytes += nblk_b * rows_b * 128;
        mbar_arrive_expect_tx(&bars[0], bytes);
        if (!a_manual)
            for (int blk = 0; blk < nblk_a; ++blk)
                tma_load_2d(tile_a + blk * rows_a * 128, &map_a, &bars[0], blk * 64, 0);
        if (!b_manual)
            for (int blk = 0; blk < nblk_b; ++blk)
                tma_load_2d(tile_b + blk * rows_b * 128, &map_b, &bars[0], blk * 64, 0);
    }
    if (a_manual)  // threads write A element by element into the swizzled layout
        for (int idx = threadIdx.x; idx < rows_a * cols_a; idx += blockDim.x) {
            const int r = idx / cols_a, c = idx % cols_a;
            *reinterpret_cast<__nv_bfloat16 *>(tile_a + swz_offset(rows_a, r, c)) = a_src[idx];
        }
    if (b_manual)
        for (int idx = threadIdx.x; idx < rows_b * cols_b; idx += blockDim.x) {
            const int r = idx / cols_b, c = idx % cols_b;
            *reinterpret_cast<__nv_bfloat16 *>(tile_b + swz_offset(rows_b, r, c)) = b_src[idx];
        }
    fence_proxy_async();
    __syncthreads();
    bool ok = mbar_wait(&bars[0], 0, &abort_flag);
    if (ok && threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(M, N, a_mn != 0, b_mn != 0);
        const uint32_t ta = smem_u32(tile_a), tb = smem_u32(tile_b);
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint64_t da = a_mn ? desc_mnmajor(ta, rows_a, 0, ks) : desc_kmajor(ta, rows_a, 0, ks);
            const uint64_t db = b_mn ? desc_mnmajor(tb + (uint32_t)b_off * 2u, rows_b, 0, ks) : desc_kmajor(tb, rows_b, 0, ks);
            if (collector == 1) {
                mma_bf16_fill(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
                mma_bf16_lastuse(tmem + (uint32_t)N, da, db, idesc, ks > 0 ? 1u : 0u);
            } else if (collector == 2) {   // the second MMA is N = 16 (first 16 rows of B)
                mma_bf16_fill(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
                mma_bf16_lastuse(tmem + (uint32_t)N, da, db, idesc_bf16(M, 16, a_mn != 0, b_mn != 0),
                                 ks > 0 ? 1u : 0u);
            } else if (collector == 3) {   // fill, use (N = 16), lastuse (N = 16)
                const uint32_t id16 = idesc_bf16(M, 16, a_mn != 0, b_mn != 0);
                mma_bf16_fill(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
                mma_bf16_use(tmem + (uint32_t)N, da, db, id16, ks > 0 ? 1u : 0u);
                mma_bf16_lastuse(tmem + (uint32_t)N + 16u, da, db, id16, ks > 0 ? 1u : 0u);
            } else {
                mma_bf16(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
            }
        }
        mma_commit(&bars[1]);
    }
    __syncwarp();
    ok = ok && mbar_wait(&bars[1], 0, &abort_flag);
    tc_fence_after();
    if (ok) {
        const int row = warp * 32 + lane;
        const int nout = collector == 1 ? 2 * N : (collector == 2 ? N + 16 : (collector == 3 ? N + 32 : N));
        for (int c0 = 0; c0 < nout; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
            tmem_wait_regs<16>(v);
            for (int i = 0; i < 16; ++i) d[row * nout + c0 + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_slot, ncols);
    if (threadIdx.x == 0 && abort_flag) atomicExch(err, 1);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map over a row-major bf16 matrix [rows][cols], box [rows][64], 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *ptr, int rows, int cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Returns 0 on success, 1 bad arguments, 2 tensor-map failure, 3 launch failure,
// 4 a bounded wait ran out.
extern "C" int tc_probe_mma(const void *a, const void *b, float *d, int N, int K, int a_mn, int b_mn,
                            int a_manual, int b_manual, int collector, int dcol, int b_off, int *err_dev) {
    const int M = 128;
    if (N < 16 || N > 256 || N % 16 || K < 16 || K > 256 || K % 16) return 1;
    if (collector < 0 || collector > 3) return 1;
    if (b_off < 0 || b_off % 8 || (b_off && (!b_mn || !b_manual || (b_off % 64) + N > 64))) return 1;
    const int nout = collector == 1 ? 2 * N : (collector == 2 ? N + 16 : (collector == 3 ? N + 32 : N));
    if (dcol < 0 || dcol % 16 || dcol + nout > 512) return 1;
    const int rows_a = a_mn ? K : M, cols_a = a_mn ? M : K;
    const int rows_b = b_mn ? K : N, cols_b = b_mn ? N + b_off : K;
    if ((!a_manual && cols_a % 64) || (!b_manual && cols_b % 64)) return 1;   // TMA: whole blocks
    if (rows_a % 8 || rows_b % 8) return 1;
    CUtensorMap ma{}, mb{};
    if (!a_manual && !make_map(&ma, a, rows_a, cols_a)) return 2;
    if (!b_manual && !make_map(&mb, b, rows_b, cols_b)) return 2;
    if (cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
        return 3;
    probe_kernel<<<1, 128, kSmemBytes>>>(ma, mb, static_cast<const __nv_bfloat16 *>(a),
                                         static_cast<const __nv_bfloat16 *>(b), d, N, K, a_mn, b_mn, a_manual,
                                         b_manual, collector, dcol, b_off, err_dev);
    if (cudaGetLastError() != cudaSuccess) return 3;
    if (cudaDeviceSynchronize() != cudaSuccess) return 3;
    int err = 0;
    if (cudaMemcpy(&err, err_dev, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
    return err ? 4 : 0;
}
