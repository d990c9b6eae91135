// la_tc_common.cuh -- helpers shared by the tensor-core kernels (forward and backward):
// shared-memory alignment, bounded and warp-uniform waits, the feature map on bf16
// chunks, bf16 packing, the optional self-check facility, and TMA tensor-map creation.
#pragma once

#include <cstdlib>
#include <cudaTypedefs.h>

#include "la_internal.cuh"
#include "la_tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kSmemLimit = 227 * 1024;

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// Time-bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kDrainNs) return;
}

// Warp-uniform bounded wait.  A phase that has already completed is seen by one
// non-blocking test; only a wait that has to block reads the abort flag and the timer.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
    const bool ok = (*abort == 0) && mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Warp-uniform non-blocking test (lane 0's view of the phase).
__device__ __forceinline__ bool warp_test(uint64_t *bar, uint32_t parity) {
    return __shfl_sync(0xffffffffu, mbar_test(bar, parity) ? 1 : 0, 0) != 0;
}

// Warp-uniform drain of a barrier phase (bounded; for the exit paths).
__device__ __forceinline__ void warp_drain(uint64_t *bar, uint32_t parity) {
    mbar_drain(bar, parity);
    __syncwarp();
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
}

// Self-check build (compile with -DLA_DEBUG): every shared-memory, TMEM and global access
// of these kernels and every TMA / MMA operand range is checked first; the first failing
// check is recorded in g_la_debug (check id, two values, block) and the access is skipped.
#ifdef LA_DEBUG
__device__ int g_la_debug[4];   // one per translation unit
__device__ __noinline__ bool dbg_fail(int id, long long a, long long b) {
    if (atomicCAS(&g_la_debug[0], 0, id) == 0) {
        g_la_debug[1] = (int)a;
        g_la_debug[2] = (int)b;
        g_la_debug[3] = (int)blockIdx.x;
    }
    return false;
}
#define LA_CHECK(cond, id, a, b) ((cond) ? true : dbg_fail((id), (long long)(a), (long long)(b)))
#else
#define LA_CHECK(cond, id, a, b) true
#endif

// Timeline build (compile with -DLA_TIMELINE): block 0 of a kernel records clock64() at
// fixed events of its first 64 chunks, read back with la_timeline_read().
#ifdef LA_TIMELINE
__device__ long long g_la_tl[64][16];
__device__ long long g_la_tl2[64][16];   // a second kernel of the same translation unit
#define LA_TL(k, ev)                                                  \
    do {                                                              \
        if (blockIdx.x == 0 && (k) < 64) g_la_tl[(k)][(ev)] = clock64(); \
    } while (0)
#define LA_TL2(k, ev)                                                  \
    do {                                                               \
        if (blockIdx.x == 0 && (k) < 64) g_la_tl2[(k)][(ev)] = clock64(); \
    } while (0)
// ... and every block of kernel `kid` records the global timer (ns) at its entry (ev 0) and
// exit (ev 1), read back with la_timeline_read_span()
__device__ unsigned long long g_la_span[4][256][2];
#define LA_SPAN(kid, ev)                                                                            \
    do {                                                                                            \
        if (threadIdx.x == 0 && blockIdx.x < 256) {                                                 \
            unsigned long long t_;                                                                  \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                  \
            g_la_span[(kid)][blockIdx.x][(ev)] = t_;                                                \
        }                                                                                           \
    } while (0)
#else
#define LA_TL(k, ev) \
    do {             \
    } while (0)
#define LA_TL2(k, ev) \
    do {              \
    } while (0)
#define LA_SPAN(kid, ev) \
    do {                 \
    } while (0)
#endif

// Shared-memory range [p, p + bytes) lies inside [lo, hi).
[[maybe_unused]] __device__ __forceinline__ bool in_smem(const void *p, uint32_t bytes, uint32_t lo, uint32_t hi) {
    const uint32_t a = smem_u32(p);
    return a >= lo && a + bytes <= hi;
}

// phi on two bf16 values in bf16x2 arithmetic, branch-free, for the feature map PHI (a
// compile-time constant: the kernels branch on the call's phi once per chunk, outside their
// unrolled loops, which a per-pair branch on a runtime phi slows by ~6 %): elu(x) + 1 = max(x, 0) + exp(m), m = min(x, 0); relu(x) = max(x, 0);
// identity: x.  exp(m) = 2^y with y = m log2(e).  y is formed as yh = bf16(m * c_hi)
// (c_hi = log2(e) rounded to bf16) plus the small remainder r = (m c_hi - yh) + m (log2(e) -
// c_hi), the first term exact in one fused multiply-add; then 2^y = 2^yh 2^r ~ 2^yh (1 + r
// ln 2), with 2^yh from the packed bf16 ex2 instruction.  About ten packed operations per
// pair; at most 0.9 % relative error over bf16 x in [-12, 4].  (A float32 version with a
// single rounding was measured: it lowers the tensor-core dq error by at most 20 % and makes
// the long-context step 10 % slower, the feature map being on every kernel's chunk path.)
template <int PHI>
__device__ __forceinline__ uint32_t feat_bf16x2(uint32_t u) {
    if (PHI == LA_PHI_IDENTITY) return u;
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&u);
    const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
    __nv_bfloat162 y = __hmax2(x, zero);
    if (PHI == LA_PHI_ELU1) {
        const __nv_bfloat162 c_hi = __float2bfloat162_rn(1.4453125f);   // bf16(log2 e)
        const __nv_bfloat162 c_lo = __float2bfloat162_rn(1.4426950408889634f - 1.4453125f);
        const __nv_bfloat162 ln2 = __float2bfloat162_rn(0.6931471805599453f);
        const __nv_bfloat162 m = __hmin2(x, zero);
        const __nv_bfloat162 yh = __hmul2(m, c_hi);
        __nv_bfloat162 r = __hfma2(m, c_hi, __hneg2(yh));
        r = __hfma2(m, c_lo, r);
        uint32_t ei;
        asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(ei) : "r"(*reinterpret_cast<const uint32_t *>(&yh)));
        __nv_bfloat162 e = *reinterpret_cast<__nv_bfloat162 *>(&ei);
        e = __hfma2(e, __hmul2(r, ln2), e);
        y = __hadd2(y, e);
    }
    return *reinterpret_cast<uint32_t *>(&y);
}

// phi on up to NB 16-byte pieces in place (piece n exists when present[n]; it becomes zeros
// when !valid[n], its row being past the end).  Every load is issued before any store:
// in-place updates through computed addresses would otherwise serialise, the compiler being
// unable to tell a later load from an earlier store's address.
template <int PHI, int NB>
__device__ __forceinline__ void feat8_batch(uint8_t *const *ptr, const bool *present, const bool *valid) {
    uint4 x[NB];
#pragma unroll
    for (int n = 0; n < NB; ++n)
        x[n] = present[n] && valid[n] ? *reinterpret_cast<const uint4 *>(ptr[n]) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int n = 0; n < NB; ++n) {
        if (!(present[n] && valid[n])) continue;
        uint32_t *xi = reinterpret_cast<uint32_t *>(&x[n]);
#pragma unroll
        for (int q = 0; q < 4; ++q) xi[q] = feat_bf16x2<PHI>(xi[q]);
    }
#pragma unroll
    for (int n = 0; n < NB; ++n)
        if (present[n]) *reinterpret_cast<uint4 *>(ptr[n]) = x[n];
}

// phi on up to NB 16-byte pieces in place, as feat8_batch; the first NSCALED of them (rows
// r0, r0 + step, ... of a stacked tile whose row r C + ti has its den at den_tile[r DPAD + ti])
// are then divided by their row's den in float32 and rounded to bf16 once more: phi(q) / den.
// (A bf16 multiply by bf16(1 / den) is cheaper but leaves a rounding error shared by the whole
// row, which the h z term of dq amplifies: measured, it doubles the dq error.)
template <int PHI, int NB, int C, int DPAD>
__device__ __forceinline__ void feat8_batch_rowscale(uint8_t *const *ptr, const bool *present, const bool *valid,
                                                     const float *den_tile, int r0, int step, int nscaled) {
    uint4 x[NB];
#pragma unroll
    for (int n = 0; n < NB; ++n)
        x[n] = present[n] && valid[n] ? *reinterpret_cast<const uint4 *>(ptr[n]) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int n = 0; n < NB; ++n) {
        if (!(present[n] && valid[n])) continue;
        uint32_t *xi = reinterpret_cast<uint32_t *>(&x[n]);
        const int row = r0 + n * step;
        const float sc = n < nscaled ? 1.f / den_tile[(row / C) * DPAD + row % C] : 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t f = feat_bf16x2<PHI>(xi[q]);
            if (n < nscaled) {
                const float2 v = unpack_bf16x2(f);
                f = pack_bf16x2(v.x * sc, v.y * sc);
            }
            xi[q] = f;
        }
    }
#pragma unroll
    for (int n = 0; n < NB; ++n)
        if (present[n]) *reinterpret_cast<uint4 *>(ptr[n]) = x[n];
}

// phi on up to NB 16-byte pieces in place, each piece n then times sc[n], as feat8_batch
// (loads first, stores last), with phi in float32 and one rounding to bf16: the weighted
// features w phi(x) of the cos/sin passes, and w phi(q) / den where sc = w / den.
template <int PHI, int NB>
__device__ __forceinline__ void feat8_batch_scaled(uint8_t *const *ptr, const bool *present, const bool *valid,
                                                   const float *sc) {
    uint4 x[NB];
#pragma unroll
    for (int n = 0; n < NB; ++n)
        x[n] = present[n] && valid[n] ? *reinterpret_cast<const uint4 *>(ptr[n]) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int n = 0; n < NB; ++n) {
        if (!(present[n] && valid[n])) continue;
        uint32_t *xi = reinterpret_cast<uint32_t *>(&x[n]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = unpack_bf16x2(xi[q]);
            float a = f.x, b = f.y;
            if (PHI == LA_PHI_ELU1) {
                a = a > 0.f ? a + 1.f : expf(a);
                b = b > 0.f ? b + 1.f : expf(b);
            } else if (PHI == LA_PHI_RELU) {
                a = fmaxf(a, 0.f);
                b = fmaxf(b, 0.f);
            }
            xi[q] = pack_bf16x2(a * sc[n], b * sc[n]);
        }
    }
#pragma unroll
    for (int n = 0; n < NB; ++n)
        if (present[n]) *reinterpret_cast<uint4 *>(ptr[n]) = x[n];
}

// w phi(x) on 8 bf16 values (16 bytes) in place, or zeros for a row past the end: phi in
// float32 (expf for elu+1), times the row's position weight w, rounded to bf16 once.  (The
// cos/sin passes of the forward; one rounding keeps the weighted features as accurate as
// bf16 allows, where the unweighted maps trade that for the packed bf16 arithmetic above.)
template <int PHI>
__device__ __forceinline__ void feat8_weighted(uint8_t *chunk, bool valid, float w) {
    uint4 *ptr = reinterpret_cast<uint4 *>(chunk);
    uint4 x = valid ? *ptr : make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
        uint32_t *xi = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = unpack_bf16x2(xi[q]);
            float a = f.x, b = f.y;
            if (PHI == LA_PHI_ELU1) {
                a = a > 0.f ? a + 1.f : expf(a);
                b = b > 0.f ? b + 1.f : expf(b);
            } else if (PHI == LA_PHI_RELU) {
                a = fmaxf(a, 0.f);
                b = fmaxf(b, 0.f);
            }
            xi[q] = pack_bf16x2(a * w, b * w);
        }
    }
    *ptr = x;
}

// phi applied to 8 bf16 values (16 bytes) in place, or zeros for a row past the end.
template <int PHI>
__device__ __forceinline__ void feat8_inplace2(uint8_t *chunk, bool valid) {
    uint4 *ptr = reinterpret_cast<uint4 *>(chunk);
    uint4 x = valid ? *ptr : make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
        x.x = feat_bf16x2<PHI>(x.x);
        x.y = feat_bf16x2<PHI>(x.y);
        x.z = feat_bf16x2<PHI>(x.z);
        x.w = feat_bf16x2<PHI>(x.w);
    }
    *ptr = x;
}

__host__ __device__ constexpr int align32(int x) { return (x + 31) / 32 * 32; }

// Segment states of the tensor-core kernels (one (S, z) pair, D (D + 1) floats per segment)
// are lane-blocked: S[d][e] sits at ((e / 4) D + d) 4 + e % 4 and z[d] at D D + d.  A warp
// whose threads hold rows d (TMEM lanes d) then moves 16 columns as four runs of 512
// contiguous bytes, where a row-major state costs one 4-byte access per lane and column.  The
// segment scan adds states elementwise and does not depend on the layout.
template <int D>
__device__ __forceinline__ void state_load16(const float *st, int d, int c16, float *v) {
    const float4 *p = reinterpret_cast<const float4 *>(st);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 x = p[(c16 * 4 + q) * D + d];
        v[4 * q] = x.x;
        v[4 * q + 1] = x.y;
        v[4 * q + 2] = x.z;
        v[4 * q + 3] = x.w;
    }
}
template <int D>
__device__ __forceinline__ void state_store16(float *st, int d, int c16, const float *v) {
    float4 *p = reinterpret_cast<float4 *>(st);
#pragma unroll
    for (int q = 0; q < 4; ++q) p[(c16 * 4 + q) * D + d] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
template <int D> __device__ __forceinline__ float state_z(const float *st, int d) { return st[D * D + d]; }

// A segment's starting state, 16 columns of row d (and z[d]): as the scan kernel left it in the
// segment's slot, or (in_kernel) summed here from the per-segment states of its sequence (`head`:
// segment 0's slot) in the scan's own order, so that the bits are the same: the segments before
// `seg` ascending (kScanPrefix), after it descending (kScanSuffix), or all of them (kScanTotal).
template <int D>
__device__ __forceinline__ void seg_state_load16(const float *head, int seg, int nseg, int mode, bool in_kernel, int d,
                                                 int c16, float *v) {
    constexpr int E = D * (D + 1);
    if (!in_kernel) {
        state_load16<D>(head + (size_t)seg * E, d, c16, v);
        return;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = 0.f;
    const bool down = mode == kScanSuffix;
    const int n = mode == kScanPrefix ? seg : mode == kScanSuffix ? nseg - 1 - seg : nseg;
    for (int u = 0; u < n; ++u) {
        float x[16];
        state_load16<D>(head + (size_t)(down ? nseg - 1 - u : u) * E, d, c16, x);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] += x[e];
    }
}
template <int D>
__device__ __forceinline__ float seg_state_z(const float *head, int seg, int nseg, int mode, bool in_kernel, int d) {
    constexpr int E = D * (D + 1);
    if (!in_kernel) return state_z<D>(head + (size_t)seg * E, d);
    const bool down = mode == kScanSuffix;
    const int n = mode == kScanPrefix ? seg : mode == kScanSuffix ? nseg - 1 - seg : nseg;
    float z = 0.f;
    for (int u = 0; u < n; ++u) z += state_z<D>(head + (size_t)(down ? nseg - 1 - u : u) * E, d);
    return z;
}
template <int D> __device__ __forceinline__ void state_store_z(float *st, int d, float z) { st[D * D + d] = z; }

// z (fp32) into column d of a 16-row K-major z tile as rows 0 and 1: z_hi = bf16(z) and
// z_lo = bf16(z - z_hi), so that a product with the tile gives phi . z_hi and phi . z_lo in two
// fp32 columns whose sum carries z to about 16 bits.
__device__ __forceinline__ void store_z_split(uint8_t *zt, int d, float z) {
    const __nv_bfloat16 zh = __float2bfloat16_rn(z);
    *reinterpret_cast<__nv_bfloat16 *>(zt + swz_offset(16, 0, d)) = zh;
    *reinterpret_cast<__nv_bfloat16 *>(zt + swz_offset(16, 1, d)) = __float2bfloat16_rn(z - __bfloat162float(zh));
}

// A 16-row K-major tile with `cols` columns: row `one_row` = 1 for columns < cols, zero
// elsewhere.
__device__ __forceinline__ void fill_ones_tile(uint8_t *t, int cols, int one_row = 0) {
    const int nblk = (cols + 63) / 64;
    for (int idx = threadIdx.x; idx < nblk * 16 * 8; idx += blockDim.x) {
        const int blk = idx / 128, rc = idx % 128, row = rc / 8, c = rc % 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row == one_row) {
            const int col0 = blk * 64 + c * 8;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                w[q] = (col0 + 2 * q < cols ? 0x3F80u : 0u) | (col0 + 2 * q + 1 < cols ? 0x3F800000u : 0u);
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        *reinterpret_cast<uint4 *>(t + swz_chunk(16, row, blk * 8 + c)) = v;
    }
}

// One 16-column slice of an S row (bf16) into the swizzled S_bf tile (D rows).
template <int D>
__device__ __forceinline__ void store_state_row(uint8_t *sbf, int d, const float *v, int c16) {
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
    *reinterpret_cast<uint4 *>(sbf + swz_chunk(D, d, 2 * c16)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4 *>(sbf + swz_chunk(D, d, 2 * c16 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3-D map over a contiguous bf16 tensor [heads][N][D]: box {64, rows, 1}, 128-byte swizzle;
// rows past N read as zeros.
cudaError_t make_map(CUtensorMap *map, const void *ptr, int heads, int N, int D, int rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 4-D map over an input [B, H, N, D] (bf16) with element strides st (b, h, n; d contiguous,
// each a multiple of 8 elements), dims (D, N, H, B): box {64, rows, 1, 1}, 128-byte swizzle;
// loads give the coordinates (d, t, h, b) to tma_load_4d_w.
cudaError_t make_map_in(CUtensorMap *map, const void *ptr, int B, int H, int N, int D, const Strides &st, int rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)st.n * 2, (cuuint64_t)st.h * 2, (cuuint64_t)st.b * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D map over float32 rows [heads][N] with a row stride of `stride` floats (a multiple of
// 4): box {cols, 1}, no swizzle; columns past N read as zeros.
cudaError_t make_map_rows_f32(CUtensorMap *map, const void *ptr, int heads, int N, int stride, int cols) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)heads};
    cuuint64_t strides[1] = {(cuuint64_t)stride * 4};
    cuuint32_t box[2] = {(cuuint32_t)cols, 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename Kern>
cudaError_t prepare(Kern kernel, int smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace
}  // namespace la
