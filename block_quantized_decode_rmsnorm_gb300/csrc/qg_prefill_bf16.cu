// bf16 prompt-sized projection on tcgen05: Y = x_hat W^T for M prompt rows, with
// the RMSNorm in front (x_hat = bf16((x * r) * gamma) per row) and SiLU(g) * u or
// nothing behind.  The decode form of the same operation is qgemv_bf16.
//
// "One level down: #002 the same compiler on a GPU": The numerical contract
// (bf16 weights and activations, f32 accumulators); Emitting for a GPU (the
// normalization fused with the projection that follows it, the activation with
// the projection before it; the stacked gate|up projection).  "Filling in the
// blanks: Inference using Phobos", Fast Decode (a prompt reuses every weight
// for all of its rows, so that form belongs on the tensor cores).
//
// GB300 mapping.  One small kernel writes x_hat for all M rows (one CTA per row,
// the same compensated norm statistic as the GEMV).  The projection is a
// persistent warp-specialised kernel over 128 x 256 output tiles:
//  * one thread issues TMA copies (128-byte swizzle) of a 128 x 64 x_hat slab and
//    two 128 x 64 weight slabs per K step into a four-stage ring; for SiLU(g) * u
//    the two weight slabs are the gate rows and the matching up rows, so one MMA
//    of N = 256 produces both halves of 128 outputs;
//  * one thread issues four tcgen05.mma kind::f16 (bf16 A and B, M = 128,
//    N = 256, K = 16) per stage into a TMEM accumulator (two of 256 columns, so
//    the epilogue of one tile overlaps the main loop of the next);
//  * eight epilogue warps (two per TMEM lane quarter, each half of the
//    columns) read the accumulator with tcgen05.ld and store f32 outputs
//    (SiLU(g) * u from the two halves where asked, with the fast exponential
//    and division: a few ulp, far inside the bf16 contract's tolerance); each
//    warp turns its 32 x 32 blocks around in shared memory so that every store
//    instruction writes 128 contiguous bytes of one output row.
// Products of bf16 values are exact in f32 and the MMA accumulates in f32, as
// the numerical contract asks; only the summation order differs from a GEMV.
// Every barrier wait is bounded by the global timer; a stalled pipeline aborts
// (NaN outputs for the tiles left) instead of hanging.
#include <cuda.h>

#include "qg_common.cuh"
#include "qg_norm.cuh"
#include "qg_tc.cuh"

namespace qg {

constexpr int PB_BM = 128;      // prompt rows per tile (TMEM lanes)
constexpr int PB_BN = 256;      // accumulator columns per tile (MMA N)
constexpr int PB_BK = 64;       // K per stage: one 128-byte swizzle row of bf16
constexpr int PB_STAGES = 4;
constexpr int PB_A_BYTES = PB_BM * PB_BK * 2;        // 16 KB
constexpr int PB_B_BYTES = PB_BN * PB_BK * 2;        // 32 KB
constexpr int PB_STAGE = PB_A_BYTES + PB_B_BYTES;    // 48 KB, a multiple of 1024
constexpr int PB_XPOSE = 32 * 33 * 4;                // per epilogue warp: a padded 32 x 32 f32 block
constexpr int PB_EPI_WARPS = 8;  // two per TMEM lane quarter, each half of the columns
constexpr int PB_SMEM = PB_STAGES * PB_STAGE + PB_EPI_WARPS * PB_XPOSE + 1024; // + alignment of the base
constexpr int PB_TMA_WARP = 8;
constexpr int PB_MMA_WARP = 9;
constexpr int PB_THREADS = 10 * 32;

struct PrefillBf16Params {
    float *y;         // [m][n_out]
    int64_t m;
    int64_t n_out;    // outputs per row: half (SiLU * u) or n_rows
    int64_t half;     // SiLU * u: up rows start here
    int k;
    int silu;         // 1: outputs are SiLU(g) * u of the stacked halves
    int64_t m_tiles;
    int64_t tiles;    // m_tiles * n_tiles, M fastest
    int n_per_tile;   // outputs per tile: 128 (SiLU * u) or 256
};

// ---------------------------------------------------------------------------
// x_hat for every prompt row
// ---------------------------------------------------------------------------
// One CTA per row: the row is read once in 16-byte pieces kept in registers;
// r from the compensated sum of exact squares (as in the GEMV), then
// x_hat = bf16((x * r) * gamma), two f32 roundings and one bf16 rounding.
constexpr int NR_THREADS = 128;
constexpr int NR_MAXC = 16;  // 16-byte pieces per thread: k <= 16384
__global__ void __launch_bounds__(NR_THREADS) rmsnorm_bf16_rows_kernel(const uint16_t *x, const uint16_t *gamma,
                                                                       int k, float inv_k, float eps, uint16_t *xhat)
{
    __shared__ float scratch[2 * (NR_THREADS / 32) + 1];
    const int64_t row = blockIdx.x;
    const int nc = k / 8;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * k);
    pdl_trigger();
    pdl_wait();
    uint4 v[NR_MAXC];
    f32pair acc = {0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < NR_MAXC; ++j) {
        const int c = static_cast<int>(threadIdx.x) + NR_THREADS * j;
        if (c < nc) {
            v[j] = xr[c];
            const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pair_add_square(acc, __uint_as_float(u[i] << 16));
                pair_add_square(acc, __uint_as_float(u[i] & 0xffff0000u));
            }
        }
    }
    const float r = block_rms_inv(acc, k, inv_k, eps, scratch);
    uint4 *out = reinterpret_cast<uint4 *>(xhat + row * k);
    const uint4 *gr = reinterpret_cast<const uint4 *>(gamma);
#pragma unroll
    for (int j = 0; j < NR_MAXC; ++j) {
        const int c = static_cast<int>(threadIdx.x) + NR_THREADS * j;
        if (c < nc) {
            const uint4 g4 = gr[c];
            const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            const uint32_t gu[4] = {g4.x, g4.y, g4.z, g4.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = __fmul_rn(__fmul_rn(__uint_as_float(u[i] << 16), r), __uint_as_float(gu[i] << 16));
                const float hi = __fmul_rn(__fmul_rn(__uint_as_float(u[i] & 0xffff0000u), r),
                                           __uint_as_float(gu[i] & 0xffff0000u));
                o[i] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
                       (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
            }
            out[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// ---------------------------------------------------------------------------
// the projection
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(PB_THREADS, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                        const PrefillBf16Params p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[PB_STAGES], empty[PB_STAGES], tfull[2], tempty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int lane = t & 31;
    const int nk = (p.k + PB_BK - 1) / PB_BK;

    if (t == 0) {
        abort_flag = 0;
        for (int i = 0; i < PB_STAGES; ++i) {
            mbar_init(&full[i], 1);   // the copy thread's expect_tx
            mbar_init(&empty[i], 1);  // the MMA thread's commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);              // the MMA thread's commit
            mbar_init(&tempty[i], PB_EPI_WARPS);  // one arrival per epilogue warp
        }
    }
    if (warp == PB_MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                     "r"(2 * PB_BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    pdl_wait();  // x_hat comes from the previous kernel
    const uint32_t tmem = tmem_base;

    if (warp == PB_TMA_WARP) {
        // ---------------- copies: x_hat slab and the two weight slabs per K step
        if (lane == 0) {
            uint32_t it = 0;
            int64_t last = -1;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
                const int64_t mt = tile % p.m_tiles, nt = tile / p.m_tiles;
                const int m0 = static_cast<int>(mt * PB_BM);
                const int r0 = static_cast<int>(p.silu ? nt * 128 : nt * PB_BN);
                const int r1 = static_cast<int>(p.silu ? p.half + nt * 128 : nt * PB_BN + 128);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const uint32_t s = it % PB_STAGES, use = it / PB_STAGES;
                    if (!(ok = tc_wait(&empty[s], (use & 1) ^ 1, &abort_flag))) break;
                    mbar_expect_tx(&full[s], PB_STAGE);
                    uint8_t *a = smem + s * PB_STAGE;
                    uint8_t *b = a + PB_A_BYTES;
                    tma_load_2d(a, &tma_a, kb * PB_BK, m0, &full[s]);
                    tma_load_2d(b, &tma_b, kb * PB_BK, r0, &full[s]);
                    tma_load_2d(b + PB_B_BYTES / 2, &tma_b, kb * PB_BK, r1, &full[s]);
                    last = it;
                }
            }
            // After an abort the last copies may still be landing: let them finish
            // (bounded) before the CTA's shared memory goes away.
            if (!ok && last >= 0) mbar_wait_bounded(&full[last % PB_STAGES], (last / PB_STAGES) & 1, kCopyWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == PB_MMA_WARP) {
        // ---------------- MMA issue: four K = 16 steps per stage ------------------
        if (lane == 0) {
            // D f32, A and B bf16, both K-major, N = 256, M = 128
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(PB_BN >> 3) << 17) |
                                   (static_cast<uint32_t>(PB_BM >> 4) << 24);
            uint32_t it = 0, tc = 0;
            int64_t last = -1;  // last stage whose MMAs were issued
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x, ++tc) {
                const uint32_t buf = tc & 1, tuse = tc >> 1;
                if (!(ok = tc_wait(&tempty[buf], (tuse & 1) ^ 1, &abort_flag))) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * PB_BN;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const uint32_t s = it % PB_STAGES, use = it / PB_STAGES;
                    if (!(ok = tc_wait(&full[s], use & 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint32_t a = smem_addr(smem + s * PB_STAGE);
                    const uint32_t b = a + PB_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < PB_BK / 16; ++kk)
                        umma_f16(d, umma_desc_sw128(a + 32 * kk), umma_desc_sw128(b + 32 * kk), idesc,
                                 (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(&empty[s]);
                    last = it;
                }
                if (!ok) break;
                umma_commit(&tfull[buf]);
            }
            // After an abort, wait (bounded) for the last issued MMAs before TMEM is freed.
            if (!ok && last >= 0) mbar_wait_bounded(&empty[last % PB_STAGES], (last / PB_STAGES) & 1, kCopyWaitLimitNs);
        }
        __syncwarp();
    } else if (warp < PB_EPI_WARPS) {
        // ---------------- epilogue: warp w reads TMEM lanes (tile rows)
        // 32 (w % 4) .. +31 and half w / 4 of the tile's columns
        const int q = warp & 3;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const int cw = p.n_per_tile / 2;  // output columns per warp
        const int cbeg = (warp >> 2) * cw;
        float *xp = reinterpret_cast<float *>(smem + PB_STAGES * PB_STAGE + warp * PB_XPOSE);  // [32][33]
        uint32_t tc = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tc) {
            const uint32_t buf = tc & 1, tuse = tc >> 1;
            // tcgen05.ld is warp-collective: the whole warp proceeds or stops
            ok = ok && __all_sync(0xffffffffu, tc_wait(&tfull[buf], tuse & 1, &abort_flag));
            tc_fence_after();
            const int64_t mt = tile % p.m_tiles, nt = tile / p.m_tiles;
            const int64_t n0 = nt * p.n_per_tile;
            const uint32_t ta = tmem + lane_addr + buf * PB_BN;
            for (int c0 = cbeg; c0 < cbeg + cw; c0 += 32) {
                uint32_t a[32], b[32];
                float v[32];
                if (ok) {
                    tmem_ld_32(ta + c0, a);
                    if (p.silu) tmem_ld_32(ta + 128 + c0, b);
                    tmem_ld_wait();
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = !ok ? __int_as_float(0x7fc00000)
                               : p.silu ? silu_mul(__uint_as_float(a[j]), __uint_as_float(b[j])) : __uint_as_float(a[j]);
                // lane l holds row l of the block: through shared memory (row
                // stride 33 floats, conflict-free both ways), then lane l stores
                // column l of each row
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 32; ++j) xp[lane * 33 + j] = v[j];
                __syncwarp();
                const int64_t m_base = mt * PB_BM + q * 32;
                const bool col_ok = n0 + c0 + lane < p.n_out;
#pragma unroll 8
                for (int r = 0; r < 32; ++r) {
                    const float val = xp[r * 33 + lane];
                    if (m_base + r < p.m && col_ok) p.y[(m_base + r) * p.n_out + n0 + c0 + lane] = val;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == PB_MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * PB_BN) : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// TMA needs 16-byte row strides: k a multiple of 8.
bool prefill_bf16_supported(int64_t k) { return k > 0 && k % 8 == 0; }

static cudaError_t bf16_map(EncodeTiledFn enc, CUtensorMap *map, const uint16_t *base, int64_t rows, int64_t k)
{
    const cuuint64_t dim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    const cuuint64_t stride[1] = {static_cast<cuuint64_t>(k) * 2};
    const cuuint32_t box[2] = {PB_BK, 128};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dim, stride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t launch_prefill_bf16(const uint16_t *w, int64_t n_rows, int64_t k, const uint16_t *x, int64_t m,
                                const uint16_t *gamma, float eps, int epi, uint16_t *xhat, float *y, cudaStream_t s)
{
    if (m == 0 || n_rows == 0) return cudaSuccess;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const uint16_t *a = x;
    if (gamma) {
        const float inv_k = 1.0f / static_cast<float>(k);
        if (cudaError_t e = launch_pdl(rmsnorm_bf16_rows_kernel, dim3(static_cast<unsigned>(m)), dim3(NR_THREADS), 0, s, x,
                                       gamma, static_cast<int>(k), inv_k, eps, xhat);
            e != cudaSuccess)
            return e;
        a = xhat;
    }
    CUtensorMap amap, bmap;
    if (cudaError_t e = bf16_map(enc, &amap, a, m, k); e != cudaSuccess) return e;
    if (cudaError_t e = bf16_map(enc, &bmap, w, n_rows, k); e != cudaSuccess) return e;
    PrefillBf16Params p;
    p.y = y;
    p.m = m;
    p.silu = epi == QG_EPI_SILU_MUL_HALVES ? 1 : 0;
    p.half = n_rows / 2;
    p.n_out = p.silu ? p.half : n_rows;
    p.k = static_cast<int>(k);
    p.n_per_tile = p.silu ? 128 : PB_BN;
    p.m_tiles = (m + PB_BM - 1) / PB_BM;
    p.tiles = p.m_tiles * ((p.n_out + p.n_per_tile - 1) / p.n_per_tile);
    if (cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(prefill_bf16_kernel), PB_SMEM); e != cudaSuccess)
        return e;
    const int64_t grid = p.tiles < num_sms() ? p.tiles : num_sms();
    return launch_pdl(prefill_bf16_kernel, dim3(static_cast<unsigned>(grid)), dim3(PB_THREADS), PB_SMEM, s, amap,
                      bmap, p);
}

}  // namespace qg
