// Prompt-sized Q8_0 contraction on tcgen05 over wide tiles, from operands packed
// for the tensor cores: Y[m][n] = sum_b f32(d_x[m][b]) * f32(d_w[n][b]) * S_b[m][n].
//
// "Filling in the blanks: Inference using Phobos", Fast Decode (prompt
// processing runs on the tensor cores, every weight reused for all prompt rows)
// and GPU Performance Heisenbugs (exact integer values on the tensor cores).
//
// GB300 mapping.  Codes are held as binary16 values (exact: integers in
// [-127, 127]) in plain row-major matrices, weights packed once at load time and
// activations by their quantize kernel, scales as f32 block-major [k/32][ld]
// (ld = rows rounded up to four, so that every block row starts on 16 bytes).
// The contraction is the TMA -> MMA -> TMEM pipeline of the bf16 prompt kernel
// with the per-block rescale the Q8_0 format needs:
//  * one thread copies per K step of 64 codes (two blocks) a 128 x 64 activation
//    slab and a BN x 64 weight slab (128-byte swizzle) and both blocks' scales;
//  * one thread issues, per block, two tcgen05.mma kind::f16 (M = 128, N = BN,
//    K = 16) into that block's own TMEM buffer (two of BN columns), so the block
//    sums S_b come out exact;
//  * BN / 16 epilogue warps (four TMEM lane quarters x 64-column groups) read a
//    block's sums in the 16x256b shape (a thread holds 4 rows x 16 columns, so
//    it needs few scales per block) and accumulate acc += d_x (d_w S_b) with
//    packed f32x2 operations: one rounded product and one fused multiply-add per
//    value and block, as in the streaming GEMV, with the activation scale as the
//    operand that consecutive instructions share.  The tile is then stored
//    through a padded shared-memory transpose.
// BN = 192 makes the 512 x 7168 contraction exactly 152 tiles, one per SM
// (12 epilogue warps and three pipeline stages; BN = 128 has 8 and four).
// Every barrier wait is bounded by the global timer; a stalled pipeline aborts
// (NaN outputs for the tiles left) instead of hanging.
#include <cuda.h>

#include "qg_common.cuh"
#include "qg_tc.cuh"

namespace qg {

// ---------------------------------------------------------------------------
// operand packing
// ---------------------------------------------------------------------------
// Row stride of a block-major scale plane: rows rounded up to four f32, so that
// each block's row starts on the 16-byte boundary a tensor map needs.
__host__ __device__ constexpr int64_t scales_ld(int64_t rows) { return (rows + 3) & ~int64_t(3); }

// Weight planes (int8 codes [n][k], binary16 scales [n][k/32]) -> binary16 codes
// [n][k] and f32 scales [k/32][scales_ld(n)].  One thread per 8 codes.
__global__ void pack_q8_0_f16_kernel(const int8_t *qs, const uint16_t *d, int64_t n, int k, uint16_t *codes,
                                     float *scales_t)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // 8-code group
    const int g = k / 8;
    if (i >= n * g) return;
    const int64_t row = i / g;
    const int c = static_cast<int>(i - row * g) * 8;
    const uint2 w = *reinterpret_cast<const uint2 *>(qs + row * k + c);
    uint32_t f[4];
    s8x4_to_f16x4(w.x, f[0], f[1]);
    s8x4_to_f16x4(w.y, f[2], f[3]);
    *reinterpret_cast<uint4 *>(codes + row * k + c) = make_uint4(f[0], f[1], f[2], f[3]);
    if ((c & 31) == 0) scales_t[static_cast<int64_t>(c / 32) * scales_ld(n) + row] = h2f(d[row * (k / 32) + c / 32]);
}

// Activation rows f32 [m][k] -> Q8_0 with the codes as binary16 [m][k] and the
// scales, rounded to binary16 as the format stores them, as f32 [k/32][scales_ld(m)].  The
// codes and scales are those of quantize_act_q8_0 (same device functions).
// Eight threads per 32-value block, four values each.
__global__ void quantize_act_f16_kernel(const float *x, int64_t m, int k, uint16_t *codes, float *scales_t)
{
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // 4-value group
    const int g = k / 4;
    const bool live = t < m * g;
    const int64_t row = live ? t / g : 0;
    const int c = live ? static_cast<int>(t - row * g) * 4 : 0;
    pdl_trigger();
    pdl_wait();
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) v = *reinterpret_cast<const float4 *>(x + row * k + c);
    float mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    if (!live) return;
    const float dd = div127(mx);
    const float rd = q8_recip(dd);
    const float q[4] = {static_cast<float>(q8_code(v.x, dd, rd)), static_cast<float>(q8_code(v.y, dd, rd)),
                        static_cast<float>(q8_code(v.z, dd, rd)), static_cast<float>(q8_code(v.w, dd, rd))};
    uint32_t h[2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
        h[i] = static_cast<uint32_t>(f2h_rn(q[2 * i])) | (static_cast<uint32_t>(f2h_rn(q[2 * i + 1])) << 16);
    *reinterpret_cast<uint2 *>(codes + row * k + c) = make_uint2(h[0], h[1]);
    if ((c & 31) == 0) scales_t[static_cast<int64_t>(c / 32) * scales_ld(m) + row] = h2f(f2h_rn(dd));
}

// ---------------------------------------------------------------------------
// the contraction
// ---------------------------------------------------------------------------
constexpr int T2_BM = 128;
constexpr int T2_BK = 64;  // codes per K step: two blocks, one 128-byte swizzle row of binary16
constexpr int T2_CW = 64;              // tile columns per epilogue warp
constexpr int T2_XPOSE = 32 * 40 * 4;  // per epilogue warp: a 32 x 32 f32 block in rows of 40 floats

template <int BN>
struct T2Layout {
    static constexpr int A = T2_BM * T2_BK * 2;    // activation codes, 16 KB
    static constexpr int B = BN * T2_BK * 2;       // weight codes
    static constexpr int DX = 2 * T2_BM * 4;       // [2 blocks][128] f32
    static constexpr int DW = 2048;                // [2 blocks][BN] f32, padded to 2 KB
    static constexpr int STAGE = A + B + DX + DW;  // a multiple of 1024
    // warps: EW epilogue (four TMEM lane quarters x BN / 64 column groups), then
    // the copy warp and the MMA warp
    static constexpr int EW = 4 * (BN / T2_CW);
    static constexpr int TMA_WARP = EW;
    static constexpr int MMA_WARP = EW + 1;
    static constexpr int THREADS = (EW + 2) * 32;
    static constexpr int STAGES = EW > 8 ? 3 : 4;
    static constexpr int OFF_XP = STAGES * STAGE;
    static constexpr int BYTES = OFF_XP + EW * T2_XPOSE;
    static_assert(BN % 64 == 0 && BN <= 192 && 2 * BN * 4 <= DW, "tile width");
    static_assert(STAGE % 1024 == 0 && A % 1024 == 0 && B % 1024 == 0, "swizzled slabs need 1024-byte alignment");
    static_assert(BYTES + 1024 <= 227 * 1024, "shared memory");
};

struct PrefillTc2Params {
    float *y;  // [m][n]
    int64_t m;
    int64_t n;
    int k;
    int64_t m_tiles;
    int64_t tiles;  // m_tiles * n_tiles, M fastest
};

template <int BN>
__global__ void __launch_bounds__(T2Layout<BN>::THREADS, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_dw,
                       const PrefillTc2Params p)
{
    using L = T2Layout<BN>;
    constexpr int S = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[S], empty[S], tfull[2], tempty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int lane = t & 31;
    const int nk = (p.k + T2_BK - 1) / T2_BK;

    if (t == 0) {
        abort_flag = 0;
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);                  // the copy thread's expect_tx
            mbar_init(&empty[i], 1 + L::EW);  // MMA commit + every epilogue warp (it reads the scales)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);             // MMA commit of one block
            mbar_init(&tempty[i], L::EW);        // every epilogue warp
        }
    }
    if (warp == L::MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    pdl_wait();  // the activation codes come from the previous kernel
    const uint32_t tmem = tmem_base;

    if (warp == L::TMA_WARP) {
        // ---------------- copies: codes and scales of two blocks per K step ------
        if (lane == 0) {
            uint32_t it = 0;
            int64_t last = -1;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
                const int m0 = static_cast<int>((tile % p.m_tiles) * T2_BM);
                const int n0 = static_cast<int>((tile / p.m_tiles) * BN);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const uint32_t s = it % S, use = it / S;
                    if (!(ok = tc_wait(&empty[s], (use & 1) ^ 1, &abort_flag))) break;
                    uint8_t *st = smem + s * L::STAGE;
                    mbar_expect_tx(&full[s], L::A + L::B + L::DX + 2 * BN * 4);
                    tma_load_2d(st, &tm_x, kb * T2_BK, m0, &full[s]);
                    tma_load_2d(st + L::A, &tm_w, kb * T2_BK, n0, &full[s]);
                    tma_load_2d(st + L::A + L::B, &tm_dx, m0, 2 * kb, &full[s]);
                    tma_load_2d(st + L::A + L::B + L::DX, &tm_dw, n0, 2 * kb, &full[s]);
                    last = it;
                }
            }
            if (!ok && last >= 0) mbar_wait_bounded(&full[last % S], (last / S) & 1, kCopyWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == L::MMA_WARP) {
        // ---------------- MMA issue: per block two K = 16 steps into its own buffer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                   (static_cast<uint32_t>(T2_BM >> 4) << 24);  // D f32, A and B f16, K-major
            uint32_t it = 0;
            int64_t last = -1;  // last block whose MMAs were issued (2 it + j)
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const uint32_t s = it % S, use = it / S;
                    if (!(ok = tc_wait(&full[s], use & 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint32_t a = smem_addr(smem + s * L::STAGE);
                    const uint32_t b = a + L::A;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (!(ok = tc_wait(&tempty[j], (it & 1) ^ 1, &abort_flag))) break;
                        tc_fence_after();
                        const uint32_t d = tmem + j * BN;
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            umma_f16(d, umma_desc_sw128(a + 32 * (2 * j + kk)), umma_desc_sw128(b + 32 * (2 * j + kk)),
                                     idesc, static_cast<uint32_t>(kk));
                        umma_commit(&tfull[j]);
                        last = 2 * static_cast<int64_t>(it) + j;
                    }
                    if (!ok) break;
                    umma_commit(&empty[s]);
                }
            }
            // After an abort, wait (bounded) for the last issued MMAs before TMEM is freed.
            if (!ok && last >= 0) mbar_wait_bounded(&tfull[last & 1], (last >> 1) & 1, kCopyWaitLimitNs);
        }
        __syncwarp();
    } else if (warp < L::EW) {
        // ---------------- epilogue: warp w reads TMEM lanes (tile rows) 32 (w % 4) ..
        // +31 and columns 64 (w / 4) .. +63 in the 16x256b shape, so that thread t
        // holds rows 32 (w % 4) + t / 4 + 8 i (i < 4) and the column pairs
        // 8 c + 2 (t % 4) of its 64 columns: per block it needs four activation
        // scales and eight pairs of weight scales (one shared-memory wavefront each).
        // The second 32-column half of a block is read from TMEM while the first
        // is being accumulated.  Columns come in adjacent pairs in both the TMEM
        // registers and the scale loads, so the f32x2 operands need no repacking.
        constexpr int NP = T2_CW / 8;  // column pairs per thread and row
        const int q = warp & 3;
        const int cbeg = (warp >> 2) * T2_CW;
        const int tr = lane >> 2, tc = 2 * (lane & 3);
        float *xp = reinterpret_cast<float *>(smem + L::OFF_XP + warp * T2_XPOSE);  // [32][40]
        uint32_t it = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
            const int64_t mt = tile % p.m_tiles;
            const int64_t n0 = (tile / p.m_tiles) * BN;
            uint64_t acc[4][NP];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int i = 0; i < NP; ++i) acc[r][i] = 0;
            for (int kb = 0; ok && kb < nk; ++kb, ++it) {
                const uint32_t s = it % S, use = it / S;
                // the stage's scales are read here: see them land (normally long ago)
                ok = __all_sync(0xffffffffu, tc_wait(&full[s], use & 1, &abort_flag));
                if (!ok) break;
                const uint8_t *st = smem + s * L::STAGE;
                const float *dx = reinterpret_cast<const float *>(st + L::A + L::B);
                const float *dw = reinterpret_cast<const float *>(st + L::A + L::B + L::DX);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // tcgen05.ld is warp-collective: the whole warp proceeds or stops
                    ok = __all_sync(0xffffffffu, tc_wait(&tfull[j], it & 1, &abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + j * BN + cbeg;
                    uint32_t v[2][2][16];  // [32-column half][16-lane half]
                    tmem_ld_16x256b_x4(ta, v[0][0]);
                    tmem_ld_16x256b_x4(ta + (16u << 16), v[0][1]);
                    uint64_t dxr[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float x = dx[j * T2_BM + 32 * q + tr + 8 * r];
                        dxr[r] = pack2(x, x);
                    }
                    const float *dwj = dw + j * BN + cbeg + tc;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        tmem_ld_wait_regs(v[c][0], v[c][1]);
                        if (c == 0) {
                            tmem_ld_16x256b_x4(ta + 32, v[1][0]);
                            tmem_ld_16x256b_x4(ta + (16u << 16) + 32, v[1][1]);
                        }
                        uint64_t wp[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) wp[r] = *reinterpret_cast<const uint64_t *>(dwj + 8 * (4 * c + r));
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int r = 0; r < 4; ++r)
#pragma unroll
                                for (int i2 = 0; i2 < 2; ++i2) {
                                    const int rs = 2 * h + i2;  // row tr + 8 rs
                                    const int a = 2 * (4 * c + r);
                                    acc[rs][4 * c + r] = fma2(dxr[rs], mul2(wp[r], pack2u(v[c][h][4 * r + 2 * i2], v[c][h][4 * r + 2 * i2 + 1])),
                                                              acc[rs][4 * c + r]);
                                }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[j]);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if (!ok) {
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int i = 0; i < NP; ++i) acc[r][i] = pack2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
            }
            // through shared memory (row stride 40 floats: the 64-bit writes of a
            // half-warp hit distinct banks), so that each store writes 32 columns of a row
            const int64_t m_base = mt * T2_BM + q * 32;
            const bool rows16 = (p.n & 3) == 0;  // every row of Y starts on 16 bytes
#pragma unroll
            for (int g = 0; g < NP / 4; ++g) {
                // the previous group's row copies have read the buffer
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                __syncwarp();
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        *reinterpret_cast<float2 *>(xp + (tr + 8 * r) * 40 + 8 * kk + tc) = unpack2(acc[r][4 * g + kk]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                const int64_t c0 = n0 + cbeg + 32 * g;
                if (rows16 && c0 + 32 <= p.n) {
                    // lane r sends row r's 32 values (128 bytes) in one bulk copy
                    if (m_base + lane < p.m) {
                        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], 128;" ::"l"(
                                         p.y + (m_base + lane) * p.n + c0),
                                     "r"(smem_addr(xp + lane * 40))
                                     : "memory");
                    }
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                } else {
                    const bool col_ok = c0 + lane < p.n;
#pragma unroll 8
                    for (int r = 0; r < 32; ++r) {
                        const float val = xp[r * 40 + lane];
                        if (m_base + r < p.m && col_ok) p.y[(m_base + r) * p.n + c0 + lane] = val;
                    }
                }
            }
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == L::MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t launch_pack_q8_0_f16(const int8_t *qs, const uint16_t *d, int64_t n, int64_t k, uint16_t *codes,
                                 float *scales_t, cudaStream_t s)
{
    const int64_t groups = n * (k / 8);
    if (groups == 0) return cudaSuccess;
    pack_q8_0_f16_kernel<<<static_cast<unsigned>((groups + 255) / 256), 256, 0, s>>>(qs, d, n, static_cast<int>(k),
                                                                                   codes, scales_t);
    return cudaGetLastError();
}

cudaError_t launch_quantize_act_f16(const float *x, int64_t m, int64_t k, uint16_t *codes, float *scales_t,
                                    cudaStream_t s)
{
    const int64_t groups = m * (k / 4);
    if (groups == 0) return cudaSuccess;
    return launch_pdl(quantize_act_f16_kernel, dim3(static_cast<unsigned>((groups + 255) / 256)), dim3(256), 0, s, x,
                      m, static_cast<int>(k), codes, scales_t);
}

static cudaError_t tc2_map(EncodeTiledFn enc, CUtensorMap *map, CUtensorMapDataType type, const void *base,
                           uint64_t inner, uint64_t ld, uint64_t outer, uint32_t elem, uint32_t box_inner,
                           uint32_t box_outer, CUtensorMapSwizzle swz)
{
    const cuuint64_t dim[2] = {inner, outer};
    const cuuint64_t stride[1] = {ld * elem};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(map, type, 2, const_cast<void *>(base), dim, stride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

template <int BN>
static cudaError_t launch_tc2_bn(EncodeTiledFn enc, const uint16_t *w_codes, const float *w_scales_t, int64_t n,
                                 int64_t k, const uint16_t *x_codes, const float *x_scales_t, int64_t m, float *y,
                                 cudaStream_t s)
{
    using L = T2Layout<BN>;
    const int64_t nb = k / QK;
    CUtensorMap mx, mw, mdx, mdw;
    if (cudaError_t e = tc2_map(enc, &mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x_codes, k, k, m, 2, T2_BK, T2_BM,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        e != cudaSuccess)
        return e;
    if (cudaError_t e = tc2_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w_codes, k, k, n, 2, T2_BK, BN,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        e != cudaSuccess)
        return e;
    if (cudaError_t e = tc2_map(enc, &mdx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x_scales_t, m, scales_ld(m), nb, 4, T2_BM, 2,
                                CU_TENSOR_MAP_SWIZZLE_NONE);
        e != cudaSuccess)
        return e;
    if (cudaError_t e = tc2_map(enc, &mdw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, w_scales_t, n, scales_ld(n), nb, 4, BN, 2,
                                CU_TENSOR_MAP_SWIZZLE_NONE);
        e != cudaSuccess)
        return e;
    PrefillTc2Params p;
    p.y = y;
    p.m = m;
    p.n = n;
    p.k = static_cast<int>(k);
    p.m_tiles = (m + T2_BM - 1) / T2_BM;
    p.tiles = p.m_tiles * ((n + BN - 1) / BN);
    if (cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(prefill_tc2_kernel<BN>),
                                    static_cast<int>(T2Layout<BN>::BYTES + 1024));
        e != cudaSuccess)
        return e;
    const int64_t grid = p.tiles < num_sms() ? p.tiles : num_sms();
    return launch_pdl(prefill_tc2_kernel<BN>, dim3(static_cast<unsigned>(grid)), dim3(L::THREADS),
                      static_cast<size_t>(L::BYTES + 1024), s, mx, mw, mdx, mdw, p);
}

// Tile width 192 or 128: the one whose busiest SM covers the fewest columns.
cudaError_t launch_prefill_tc2(const uint16_t *w_codes, const float *w_scales_t, int64_t n, int64_t k,
                               const uint16_t *x_codes, const float *x_scales_t, int64_t m, float *y, int tile_n,
                               cudaStream_t s)
{
    if (m == 0 || n == 0) return cudaSuccess;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    if (tile_n == 0) {
        const int64_t sms = num_sms(), mt = (m + T2_BM - 1) / T2_BM;
        const int64_t r192 = (mt * ((n + 191) / 192) + sms - 1) / sms, r128 = (mt * ((n + 127) / 128) + sms - 1) / sms;
        tile_n = r192 * 192 <= r128 * 128 ? 192 : 128;
    }
    if (tile_n == 192) return launch_tc2_bn<192>(enc, w_codes, w_scales_t, n, k, x_codes, x_scales_t, m, y, s);
    if (tile_n == 128) return launch_tc2_bn<128>(enc, w_codes, w_scales_t, n, k, x_codes, x_scales_t, m, y, s);
    return cudaErrorInvalidValue;
}

}  // namespace qg
