// Q8_0 block-scaled matrix-vector product (decode) and the exact block-dot export.
//
// "Filling in the blanks: Inference using Phobos", Fast Decode: decode reads
// every weight once (about 2 ops per byte, memory-bound); the dot products run
// in int8 end to end (dp4a); a warp owns an output row and reduces with
// shuffles; the residual add is folded into the matmul.  "One level down: #002
// the same compiler on a GPU", Emitting for a GPU: gate and up are one stacked
// projection with the activation fused behind it.
//
// GB300 mapping: lane j of a warp owns 32-value blocks j, j+32, ... of a row and
// fetches each block's 32 int8 values with ONE 256-bit load, so a warp reads
// 1 KB of a row per instruction, fully coalesced.  Each lane computes the exact
// int32 block sum with eight dp4a and applies d_w*d_x once per block; the 32
// lane partials are reduced with shuffles.  A warp handles R rows per task (R
// independent 1 KB loads in flight per lane-iteration).  The first task's
// weights are requested before the programmatic-dependent-launch wait, so the
// weight stream overlaps the tail of the kernel that produces the activation.
#include <mutex>
#include <unordered_map>

#include "qg_common.cuh"

namespace qg {

struct GemvParams {
    const int8_t *w_qs;
    const uint16_t *w_d;
    const int8_t *xq;
    const uint16_t *xd;
    const float *residual;
    float *y;
    int64_t n_rows;
    int64_t n_out;    // outputs per batch row
    int64_t n_tasks;  // tasks of R weight rows
    int64_t half;     // n_rows / 2 (stacked gate|up)
    int k;
    int nb;
    int epi;
    int batch;  // live batch rows (<= the compiled width B)
};

constexpr int GEMV_THREADS = 128;

// Weight row of slot s in task t, or -1 past the end.  With the SiLU(g)*u
// epilogue a task covers R/2 outputs, slot pairs (gate row o, up row o + F).
template <int R>
__device__ __forceinline__ int64_t slot_row(const GemvParams &p, int64_t t, int s)
{
    if (p.epi == QG_EPI_SILU_MUL_HALVES) {
        const int64_t o = t * (R / 2) + (s >> 1);
        return o < p.half ? o + (s & 1) * p.half : -1;
    }
    const int64_t r = t * R + s;
    return r < p.n_rows ? r : -1;
}

// Reduce acc over the warp and write the R*B results of task t.  Lane
// (s*B + b) writes slot s of batch row b.
template <int B, int R>
__device__ __forceinline__ void reduce_and_store(const GemvParams &p, int64_t t, int lane, float (&acc)[R][B])
{
    // All R*B sums in one transposed butterfly (R*B - 1 + 5 - log2(R*B)
    // shuffles, the same pairings and order as one warp_sum per value): lane l
    // ends with value v = l >> SH, v = s * B + b.
    // (Batch 2 keeps one warp_sum per value: the butterfly's extra live values
    // cost it registers, and so resident warps, that the few shuffles saved do
    // not pay for.  Both give the same bits.)
    constexpr int NV = R * B;
    constexpr bool MANY = B != 2;
    constexpr int SH = !MANY ? 0 : NV >= 32 ? 0 : NV >= 16 ? 1 : NV >= 8 ? 2 : NV >= 4 ? 3 : NV >= 2 ? 4 : 5;
    float val = 0.0f;
    if constexpr (MANY) {
        float v[NV];
#pragma unroll
        for (int s = 0; s < R; ++s)
#pragma unroll
            for (int b = 0; b < B; ++b) v[s * B + b] = acc[s][b];
        val = warp_sum_many<NV>(v, lane);
    } else {
#pragma unroll
        for (int s = 0; s < R; ++s)
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const float w = warp_sum(acc[s][b]);
                if (lane == s * B + b) val = w;
            }
    }
    const int idx = lane >> SH;
    const bool rep = !MANY ? idx < NV : (lane & ((1 << SH) - 1)) == 0;  // one lane per value stores it
    const int s = idx / B;
    const int b = idx % B;
    if (p.epi == QG_EPI_SILU_MUL_HALVES) {
        const float u = __shfl_down_sync(0xffffffffu, val, B << SH);  // slot s+1 = up row of the pair
        if (rep && (s & 1) == 0 && b < p.batch) {
            const int64_t o = t * (R / 2) + (s >> 1);
            if (o < p.half) p.y[b * p.n_out + o] = silu_mul(val, u);
        }
        return;
    }
    if (rep && b < p.batch) {
        const int64_t row = t * R + s;
        if (row < p.n_rows) {
            float out = val;
            if (p.epi == QG_EPI_RESIDUAL_ADD) out = p.residual[b * p.n_rows + row] + val;
            p.y[b * p.n_out + row] = out;
        }
    }
}

// Fast path: nb <= 32*NBL, activation (B rows x NBL blocks per lane) held in
// registers for the whole kernel.
template <int B, int NBL, int R>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_q8_0_reg_kernel(const GemvParams p)
{
    const int lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * wpc + (threadIdx.x >> 5);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * wpc;

    u32x8 w[R][NBL];
    float wd[R][NBL];

#define QG_LOAD_WEIGHTS(T)                                                                   \
    _Pragma("unroll") for (int s = 0; s < R; ++s)                                            \
    {                                                                                        \
        const int64_t row = slot_row<R>(p, (T), s);                                          \
        _Pragma("unroll") for (int j = 0; j < NBL; ++j)                                      \
        {                                                                                    \
            const int blk = lane + 32 * j;                                                   \
            if (row >= 0 && blk < p.nb) {                                                    \
                w[s][j] = ld_stream_32B(p.w_qs + row * p.k + blk * QK);                      \
                wd[s][j] = h2f(ld_nc_u16(p.w_d + row * p.nb + blk));                         \
            } else {                                                                         \
                _Pragma("unroll") for (int i = 0; i < 8; ++i) w[s][j].v[i] = 0u;             \
                wd[s][j] = 0.0f;                                                             \
            }                                                                                \
        }                                                                                    \
    }

    if (t0 < p.n_tasks) { QG_LOAD_WEIGHTS(t0) }
    pdl_trigger();
    pdl_wait();

    u32x8 xv[B][NBL];
    float xs[B][NBL];
#pragma unroll
    for (int b = 0; b < B; ++b)
#pragma unroll
        for (int j = 0; j < NBL; ++j) {
            const int blk = lane + 32 * j;
            if (blk < p.nb && b < p.batch) {
                const int8_t *src = p.xq + static_cast<int64_t>(b) * p.k + blk * QK;
                const uint4 lo = ld_16B(src);
                const uint4 hi = ld_16B(src + 16);
                xv[b][j].v[0] = lo.x; xv[b][j].v[1] = lo.y; xv[b][j].v[2] = lo.z; xv[b][j].v[3] = lo.w;
                xv[b][j].v[4] = hi.x; xv[b][j].v[5] = hi.y; xv[b][j].v[6] = hi.z; xv[b][j].v[7] = hi.w;
                xs[b][j] = h2f(p.xd[static_cast<int64_t>(b) * p.nb + blk]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) xv[b][j].v[i] = 0u;
                xs[b][j] = 0.0f;
            }
        }

    for (int64_t t = t0; t < p.n_tasks; t += stride) {
        float acc[R][B];
#pragma unroll
        for (int s = 0; s < R; ++s)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[s][b] = 0.0f;
#pragma unroll
        for (int j = 0; j < NBL; ++j)
#pragma unroll
            for (int s = 0; s < R; ++s)
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    int S = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) S = dp4a(w[s][j].v[i], xv[b][j].v[i], S);
                    acc[s][b] = fmaf(small_int_to_float(S), wd[s][j] * xs[b][j], acc[s][b]);
                }
        const int64_t tn = t + stride;
        if (tn < p.n_tasks) { QG_LOAD_WEIGHTS(tn) }  // in flight during the reduction below
        reduce_and_store<B, R>(p, t, lane, acc);
    }
#undef QG_LOAD_WEIGHTS
}

// ---------------------------------------------------------------------------
// Batched GEMV on the int8 tensor cores (batch 2..8, K a multiple of 256)
// ---------------------------------------------------------------------------
// "Filling in the blanks: Inference using Phobos", GPU Performance Heisenbugs:
// exact int8 values on the integer tensor cores.  One mma.sync.m16n8k32 (s8,
// s32 accumulate) is exactly one 32-value block of 16 weight rows against the
// batch (N = 8, unused columns zero), so the block sums come out exact and the
// scales d_w d_x are applied per block as in the dp4a kernel.  A warp owns 16
// rows per task; thread (g = lane / 4, t = lane % 4) loads 8 bytes of rows g
// and g + 8 per block straight from HBM (the four threads of a row cover its
// 32 bytes) and the batch's codes come from shared memory, staged once per CTA.
// The fragment positions of K inside a block are permuted the same way for both
// operands (thread t carries values 8t..8t+7), which leaves every block sum
// unchanged.  With the activations out of registers a thread needs about 70
// registers, so many more warps (and weight bytes) are in flight than in the
// register-tile kernel at the same batch.
constexpr int MMA_ROWS = 16;

__device__ __forceinline__ uint2 ld_stream_8B(const void *p)
{
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ void mma_s8_16832(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// G blocks of weights are requested together per thread (G a multiple of 8 that
// divides the row's block count): 16 keeps 8 KB a warp in flight with 90
// registers (five CTAs, 20 warps an SM), against 4 KB and 28 warps for 8, and
// runs the 262144 x 1024 output head at batch 2-8 in 48.5-49.7 instead of
// 52.4-53.0 us.
template <int G>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_q8_0_mma_kernel(const GemvParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int K = p.k, nb = p.nb;
    const int XS = K + 32;  // row stride of the staged codes: conflict-free 8-byte fragment loads
    int8_t *s_x = reinterpret_cast<int8_t *>(smem);
    float *s_xd = reinterpret_cast<float *>(smem + 8 * XS);  // [nb][8]: a thread's batch pair is one 8-byte load
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int wpc = blockDim.x >> 5;
    const int64_t n_tasks = (p.n_rows + MMA_ROWS - 1) / MMA_ROWS;

    pdl_trigger();
    pdl_wait();
    // batch codes and scales, rows past the batch zero
    for (int i = threadIdx.x; i < 8 * (K / 16); i += blockDim.x) {
        const int b = i / (K / 16), off = (i - b * (K / 16)) * 16;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (b < p.batch) v = ld_16B(p.xq + static_cast<int64_t>(b) * K + off);
        *reinterpret_cast<uint4 *>(s_x + b * XS + off) = v;
    }
    for (int i = threadIdx.x; i < 8 * nb; i += blockDim.x) {
        const int b = i / nb, j = i - b * nb;
        s_xd[j * 8 + b] = b < p.batch ? h2f(p.xd[i]) : 0.0f;
    }
    __syncthreads();

    for (int64_t task = static_cast<int64_t>(blockIdx.x) * wpc + (threadIdx.x >> 5); task < n_tasks;
         task += static_cast<int64_t>(gridDim.x) * wpc) {
        const int64_t rA = task * MMA_ROWS + g, rB = rA + 8;
        const bool vA = rA < p.n_rows, vB = rB < p.n_rows;
        const int8_t *wA = p.w_qs + rA * K + 8 * t;
        const int8_t *wB = p.w_qs + rB * K + 8 * t;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};  // (row g, batch 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
        for (int j0 = 0; j0 < nb; j0 += G) {
            uint2 a[G], b[G];
#pragma unroll
            for (int u = 0; u < G; ++u) {
                a[u] = vA ? ld_stream_8B(wA + (j0 + u) * QK) : make_uint2(0u, 0u);
                b[u] = vB ? ld_stream_8B(wB + (j0 + u) * QK) : make_uint2(0u, 0u);
            }
            // the G blocks' scales of rows g and g + 8, 16 bytes (eight blocks) a load
            uint4 dA[G / 8], dB[G / 8];
#pragma unroll
            for (int q = 0; q < G / 8; ++q) dA[q] = dB[q] = make_uint4(0u, 0u, 0u, 0u);
            if (vA) {
#pragma unroll
                for (int q = 0; q < G / 8; ++q) dA[q] = ld_nc_16B(p.w_d + rA * nb + j0 + 8 * q);
            }
            if (vB) {
#pragma unroll
                for (int q = 0; q < G / 8; ++q) dB[q] = ld_nc_16B(p.w_d + rB * nb + j0 + 8 * q);
            }
            const uint16_t *sdA = reinterpret_cast<const uint16_t *>(dA);
            const uint16_t *sdB = reinterpret_cast<const uint16_t *>(dB);
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const int blk = j0 + u;
                const uint2 xf = *reinterpret_cast<const uint2 *>(s_x + g * XS + blk * QK + 8 * t);
                int c[4] = {0, 0, 0, 0};
                mma_s8_16832(c, a[u].x, b[u].x, a[u].y, b[u].y, xf.x, xf.y);
                const float2 xs2 = *reinterpret_cast<const float2 *>(s_xd + blk * 8 + 2 * t);
                const float x0 = xs2.x, x1 = xs2.y;
                const float wa = h2f(sdA[u]), wb = h2f(sdB[u]);
                acc[0] = fmaf(small_int_to_float(c[0]), wa * x0, acc[0]);
                acc[1] = fmaf(small_int_to_float(c[1]), wa * x1, acc[1]);
                acc[2] = fmaf(small_int_to_float(c[2]), wb * x0, acc[2]);
                acc[3] = fmaf(small_int_to_float(c[3]), wb * x1, acc[3]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t row = (i < 2) ? rA : rB;
            const int bcol = 2 * t + (i & 1);
            if (row < p.n_rows && bcol < p.batch) {
                float out = acc[i];
                if (p.epi == QG_EPI_RESIDUAL_ADD) out = p.residual[bcol * p.n_rows + row] + out;
                p.y[bcol * p.n_out + row] = out;
            }
        }
    }
}

// Generic path: any nb; activation read through L1 per block.
template <int B, int R>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_q8_0_generic_kernel(const GemvParams p)
{
    const int lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * wpc + (threadIdx.x >> 5);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * wpc;
    pdl_trigger();
    pdl_wait();
    for (int64_t t = t0; t < p.n_tasks; t += stride) {
        float acc[R][B];
#pragma unroll
        for (int s = 0; s < R; ++s)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[s][b] = 0.0f;
        int64_t rows[R];
#pragma unroll
        for (int s = 0; s < R; ++s) rows[s] = slot_row<R>(p, t, s);
        for (int j0 = 0; j0 < p.nb; j0 += 32) {
            const int blk = j0 + lane;
            if (blk >= p.nb) continue;
            u32x8 w[R];
            float wd[R];
#pragma unroll
            for (int s = 0; s < R; ++s) {
                if (rows[s] >= 0) {
                    w[s] = ld_stream_32B(p.w_qs + rows[s] * p.k + blk * QK);
                    wd[s] = h2f(ld_nc_u16(p.w_d + rows[s] * p.nb + blk));
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[s].v[i] = 0u;
                    wd[s] = 0.0f;
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (b >= p.batch) break;
                const int8_t *src = p.xq + static_cast<int64_t>(b) * p.k + blk * QK;
                const uint4 lo = ld_16B(src);
                const uint4 hi = ld_16B(src + 16);
                const uint32_t xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                const float xs = h2f(p.xd[static_cast<int64_t>(b) * p.nb + blk]);
#pragma unroll
                for (int s = 0; s < R; ++s) {
                    int S = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) S = dp4a(w[s].v[i], xv[i], S);
                    acc[s][b] = fmaf(small_int_to_float(S), wd[s] * xs, acc[s][b]);
                }
            }
        }
        reduce_and_store<B, R>(p, t, lane, acc);
    }
}

// Exact block sums s[b][n][j] (debug / parity export).  One thread per (b, n, j).
__global__ void __launch_bounds__(256) block_dots_kernel(const int8_t *__restrict__ w_qs, int64_t n_rows, int k,
                                                          const int8_t *__restrict__ xq, int batch,
                                                          int32_t *__restrict__ s)
{
    pdl_wait();
    pdl_trigger();
    const int nb = k / QK;
    const int64_t total = static_cast<int64_t>(batch) * n_rows * nb;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int j = static_cast<int>(i % nb);
    const int64_t n = (i / nb) % n_rows;
    const int64_t b = i / (static_cast<int64_t>(nb) * n_rows);
    const u32x8 w = ld_stream_32B(w_qs + n * k + j * QK);
    const uint4 lo = ld_16B(xq + b * k + j * QK);
    const uint4 hi = ld_16B(xq + b * k + j * QK + 16);
    const uint32_t xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    int acc = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) acc = dp4a(w.v[t], xv[t], acc);
    s[i] = acc;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Resident CTAs per SM of one kernel, cached per kernel (function pointer).
static int max_ctas_per_sm(const void *kernel, size_t smem = 0)
{
    static std::mutex mu;
    static std::unordered_map<const void *, std::pair<size_t, int>> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(kernel);
    if (it != cache.end() && it->second.first == smem) return it->second.second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, GEMV_THREADS, smem) != cudaSuccess || n < 1) n = 1;
    cache[kernel] = {smem, n};
    return n;
}

static cudaError_t launch_gemv(void (*kernel)(GemvParams), const GemvParams &p, cudaStream_t s)
{
    const int occ = max_ctas_per_sm(reinterpret_cast<const void *>(kernel));
    const int wpc = GEMV_THREADS / 32;
    const int64_t need = (p.n_tasks + wpc - 1) / wpc;
    const int64_t cap = static_cast<int64_t>(num_sms()) * occ;
    const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
    return launch_pdl(kernel, dim3(grid), dim3(GEMV_THREADS), 0, s, p);
}

template <int B, int R>
static cudaError_t dispatch_nbl(const GemvParams &p, int nbl, cudaStream_t s)
{
    if constexpr (B == 1 || B == 2) {
        switch (nbl) {
        case 1: return launch_gemv(gemv_q8_0_reg_kernel<B, 1, R>, p, s);
        case 2: return launch_gemv(gemv_q8_0_reg_kernel<B, 2, R>, p, s);
        case 3: return launch_gemv(gemv_q8_0_reg_kernel<B, 3, R>, p, s);
        case 4: return launch_gemv(gemv_q8_0_reg_kernel<B, 4, R>, p, s);
        default: break;
        }
    } else if constexpr (B == 4) {
        switch (nbl) {
        case 1: return launch_gemv(gemv_q8_0_reg_kernel<B, 1, R>, p, s);
        case 2: return launch_gemv(gemv_q8_0_reg_kernel<B, 2, R>, p, s);
        default: break;
        }
    } else {
        if (nbl == 1) return launch_gemv(gemv_q8_0_reg_kernel<B, 1, R>, p, s);
    }
    return launch_gemv(gemv_q8_0_generic_kernel<B, R>, p, s);
}

template <int B>
static cudaError_t dispatch_r(GemvParams p, int nbl, cudaStream_t s)
{
    const bool silu = p.epi == QG_EPI_SILU_MUL_HALVES;
    // Rows per warp task: as many as keep at least ~16 warps per SM busy.
    const int64_t want_warps = static_cast<int64_t>(num_sms()) * 16;
    int R = 4;
    if (p.n_rows / 4 < want_warps) R = 2;
    if (!silu && p.n_rows / 2 < want_warps) R = 1;
    if (B >= 4 && R > 2) R = 2;  // register budget of the batched activation
    const int64_t slots = p.n_rows;
    p.n_tasks = (slots + R - 1) / R;
    if (silu) p.n_tasks = (p.half + R / 2 - 1) / (R / 2);
    switch (R) {
    case 4: return dispatch_nbl<B, 4>(p, nbl, s);
    case 2: return dispatch_nbl<B, 2>(p, nbl, s);
    default: return dispatch_nbl<B, 1>(p, nbl, s);
    }
}

cudaError_t launch_gemv_q8_0(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k, const int8_t *xq,
                             const uint16_t *xd, int64_t batch, int epi, const float *residual, float *y,
                             cudaStream_t s)
{
    if (n_rows == 0) return cudaSuccess;
    GemvParams p;
    p.w_qs = w_qs;
    p.w_d = w_d;
    p.xq = xq;
    p.xd = xd;
    p.residual = residual;
    p.y = y;
    p.n_rows = n_rows;
    p.k = static_cast<int>(k);
    p.nb = static_cast<int>(k / QK);
    p.epi = epi;
    p.half = n_rows / 2;
    p.n_out = (epi == QG_EPI_SILU_MUL_HALVES) ? n_rows / 2 : n_rows;
    p.n_tasks = 0;
    p.batch = static_cast<int>(batch);
    const int nbl = (p.nb + 31) / 32;
    // Batch 1 joins the tensor-core path (its batch padded with zero rows) when
    // there are at least 64 tasks an SM: the 262144 x 1024 output head takes
    // 48.5 us there against 49.6 on the register tile.
    const bool wide = n_rows >= static_cast<int64_t>(num_sms()) * 64 * MMA_ROWS;
    if ((batch >= 2 || wide) && epi != QG_EPI_SILU_MUL_HALVES && k % 256 == 0 && k <= 4096 &&
        (reinterpret_cast<uintptr_t>(w_d) & 15) == 0) {
        // tensor-core path: 16 rows per warp task, the batch's codes staged in shared memory
        void (*kernel)(const GemvParams) = p.nb % 16 == 0 ? gemv_q8_0_mma_kernel<16> : gemv_q8_0_mma_kernel<8>;
        const void *kern = reinterpret_cast<const void *>(kernel);
        const size_t smem = static_cast<size_t>(8) * (k + 32) + static_cast<size_t>(8) * (k / QK) * 4;
        const int occ = max_ctas_per_sm(kern, smem);
        const int wpc = GEMV_THREADS / 32;
        const int64_t need = ((n_rows + MMA_ROWS - 1) / MMA_ROWS + wpc - 1) / wpc;
        const int64_t cap = static_cast<int64_t>(num_sms()) * occ;
        return launch_pdl(kernel, dim3(static_cast<unsigned>(need < cap ? need : cap)), dim3(GEMV_THREADS), smem, s,
                          p);
    }
    if (batch == 1) return dispatch_r<1>(p, nbl, s);
    if (batch == 2) return dispatch_r<2>(p, nbl, s);
    if (batch <= 4) return dispatch_r<4>(p, nbl, s);
    if (batch <= 8) return dispatch_r<8>(p, nbl, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_block_dots(const int8_t *w_qs, int64_t n_rows, int64_t k, const int8_t *xq, int64_t batch,
                              int32_t *s_out, cudaStream_t s)
{
    const int64_t total = batch * n_rows * (k / QK);
    if (total == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((total + 255) / 256);
    return launch_pdl(block_dots_kernel, dim3(grid), dim3(256), 0, s, w_qs, n_rows, static_cast<int>(k), xq,
                      static_cast<int>(batch), s_out);
}

}  // namespace qg
