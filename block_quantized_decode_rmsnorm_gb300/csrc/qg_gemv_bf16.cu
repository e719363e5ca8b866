// bf16-weight matrix-vector product, f32 accumulation, with the RMSNorm fused in
// front and SiLU(g)*u / residual fused behind.
//
// "One level down: #002 the same compiler on a GPU": The numerical contract
// (bf16 weights and activations, f32 accumulators); Emitting for a GPU (rows
// are read as 16-byte groups of eight bf16 values; the stacked gate|up
// projection; the normalization fused with the projection that follows it and
// the activation with the projection before it); Decode: memory decides (the
// matvec is a pure weight stream).
//
// GB300 mapping: every CTA first builds x_hat = bf16((x * r) * gamma) in shared
// memory (x is a few KB, read from L2), stored as f32 in two planes so that a
// lane's eight values come from two conflict-free 16-byte shared loads.  Lane j
// of a warp reads 16-byte group j, j+32, ... of a row (512 bytes per warp
// instruction); a warp handles R rows per task with all of a row's groups
// requested up front.  The first task's weights are requested before the
// dependent-launch wait.
#include <mutex>

#include "qg_common.cuh"
#include "qg_norm.cuh"

namespace qg {

struct Bf16Params {
    const uint16_t *w;
    const uint16_t *x;
    const uint16_t *gamma;
    const float *residual;
    float *y;
    int64_t n_rows;
    int64_t n_out;
    int64_t n_tasks;
    int64_t half;
    int k;
    int n_groups;  // k / 8
    float inv_k;   // fl(1 / k)
    float eps;
    int epi;
};

constexpr int BF16_THREADS = 512;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// x_hat plane index of element e: group g = e / 8 (lane g % 32 of chunk g / 32)
// stores elements 0-3 of its group in plane A and 4-7 in plane B, each at
// float offset 4 * g.
__device__ __forceinline__ int xhat_slot(int e) { return ((e >> 3) << 2) + (e & 3); }

template <int R>
__device__ __forceinline__ int64_t bf16_slot_row(const Bf16Params &p, int64_t t, int s)
{
    if (p.epi == QG_EPI_SILU_MUL_HALVES) {
        const int64_t o = t * (R / 2) + (s >> 1);
        return o < p.half ? o + (s & 1) * p.half : -1;
    }
    const int64_t r = t * R + s;
    return r < p.n_rows ? r : -1;
}

template <int R>
__device__ __forceinline__ void bf16_store(const Bf16Params &p, int64_t t, int lane, float (&acc)[R])
{
    float val = 0.0f;
#pragma unroll
    for (int s = 0; s < R; ++s) {
        const float v = warp_sum(acc[s]);
        if (lane == s) val = v;
    }
    if (p.epi == QG_EPI_SILU_MUL_HALVES) {
        const float u = __shfl_down_sync(0xffffffffu, val, 1);
        if (lane < R && (lane & 1) == 0) {
            const int64_t o = t * (R / 2) + (lane >> 1);
            if (o < p.half) p.y[o] = silu_mul(val, u);
        }
        return;
    }
    if (lane < R) {
        const int64_t row = t * R + lane;
        if (row < p.n_rows) p.y[row] = (p.epi == QG_EPI_RESIDUAL_ADD) ? p.residual[row] + val : val;
    }
}

// A lane holds NCH groups of each of R rows in registers at a time; rows with
// more groups are walked in super-chunks of NCH groups.
template <int R, int NCH>
__global__ void __launch_bounds__(BF16_THREADS) gemv_bf16_kernel(const Bf16Params p)
{
    extern __shared__ float smem[];  // plane A [n_groups*4], plane B [n_groups*4], scratch
    float *planeA = smem;
    float *planeB = smem + p.n_groups * 4;
    float *scratch = smem + p.n_groups * 8;

    const int lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * wpc + (threadIdx.x >> 5);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * wpc;

    uint4 w[R][NCH];
#define QG_LOAD_BF16(T, C0)                                                                      \
    _Pragma("unroll") for (int s = 0; s < R; ++s)                                                \
    {                                                                                            \
        const int64_t row = bf16_slot_row<R>(p, (T), s);                                         \
        _Pragma("unroll") for (int c = 0; c < NCH; ++c)                                          \
        {                                                                                        \
            const int g = lane + 32 * ((C0) + c);                                                \
            if (row >= 0 && g < p.n_groups)                                                      \
                w[s][c] = ld_stream_16B(p.w + row * p.k + g * 8);                                \
            else                                                                                 \
                w[s][c] = make_uint4(0u, 0u, 0u, 0u);                                            \
        }                                                                                        \
    }

    if (t0 < p.n_tasks) { QG_LOAD_BF16(t0, 0) }
    pdl_trigger();
    pdl_wait();

    // ---- prologue: x_hat into shared memory --------------------------------
    const bool norm = p.gamma != nullptr;
    float r = 1.0f;
    if (norm) {
        f32pair acc = {0.0f, 0.0f};
        for (int g = threadIdx.x; g < p.n_groups; g += blockDim.x) {
            const uint4 xv = ld_16B(p.x + g * 8);
            const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pair_add_square(acc, bf16_lo(u[i]));
                pair_add_square(acc, bf16_hi(u[i]));
            }
        }
        r = block_rms_inv(acc, p.k, p.inv_k, p.eps, scratch);
    }
    for (int g = threadIdx.x; g < p.n_groups; g += blockDim.x) {
        const uint4 xv = ld_16B(p.x + g * 8);
        const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = bf16_lo(u[i]);
            v[2 * i + 1] = bf16_hi(u[i]);
        }
        if (norm) {
            const uint4 gv = ld_16B(p.gamma + g * 8);
            const uint32_t gu[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float t0v = __fmul_rn(__fmul_rn(v[2 * i], r), bf16_lo(gu[i]));
                const float t1v = __fmul_rn(__fmul_rn(v[2 * i + 1], r), bf16_hi(gu[i]));
                v[2 * i] = __bfloat162float(__float2bfloat16_rn(t0v));
                v[2 * i + 1] = __bfloat162float(__float2bfloat16_rn(t1v));
            }
        }
        *reinterpret_cast<float4 *>(planeA + 4 * g) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(planeB + 4 * g) = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();

    // ---- main loop ----------------------------------------------------------
    const int n_chunks = (p.n_groups + 31) / 32;
    for (int64_t t = t0; t < p.n_tasks; t += stride) {
        float acc[R];
#pragma unroll
        for (int s = 0; s < R; ++s) acc[s] = 0.0f;
        for (int c0 = 0; c0 < n_chunks; c0 += NCH) {
            if (c0 > 0) { QG_LOAD_BF16(t, c0) }
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int g = lane + 32 * (c0 + c);
                if (g < p.n_groups) {
                    const float4 a = *reinterpret_cast<const float4 *>(planeA + 4 * g);
                    const float4 b = *reinterpret_cast<const float4 *>(planeB + 4 * g);
#pragma unroll
                    for (int s = 0; s < R; ++s) {
                        float q = acc[s];
                        q = fmaf(bf16_lo(w[s][c].x), a.x, q);
                        q = fmaf(bf16_hi(w[s][c].x), a.y, q);
                        q = fmaf(bf16_lo(w[s][c].y), a.z, q);
                        q = fmaf(bf16_hi(w[s][c].y), a.w, q);
                        q = fmaf(bf16_lo(w[s][c].z), b.x, q);
                        q = fmaf(bf16_hi(w[s][c].z), b.y, q);
                        q = fmaf(bf16_lo(w[s][c].w), b.z, q);
                        q = fmaf(bf16_hi(w[s][c].w), b.w, q);
                        acc[s] = q;
                    }
                }
            }
        }
        const int64_t tn = t + stride;
        if (tn < p.n_tasks) { QG_LOAD_BF16(tn, 0) }
        bf16_store<R>(p, t, lane, acc);
    }
#undef QG_LOAD_BF16
}

template <int R, int NCH>
static cudaError_t launch_bf16_nch(const Bf16Params &p, cudaStream_t s)
{
    auto kernel = gemv_bf16_kernel<R, NCH>;
    const size_t smem = (static_cast<size_t>(p.n_groups) * 8 + 2 * (BF16_THREADS / 32) + 1) * sizeof(float);
    if (cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(kernel), 200 * 1024); e != cudaSuccess) return e;
    // occupancy depends on the shared-memory size, i.e. on k: cache the last answer
    static std::mutex mu;
    static size_t occ_smem = 0;
    static int occ_val = 1;
    int occ;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (occ_smem != smem) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, BF16_THREADS, smem) != cudaSuccess || n < 1)
                n = 1;
            occ_smem = smem;
            occ_val = n;
        }
        occ = occ_val;
    }
    const int wpc = BF16_THREADS / 32;
    const int64_t need = (p.n_tasks + wpc - 1) / wpc;
    const int64_t cap = static_cast<int64_t>(num_sms()) * occ;
    const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
    return launch_pdl(kernel, dim3(grid), dim3(BF16_THREADS), smem, s, p);
}

template <int R>
static cudaError_t launch_bf16_r(const Bf16Params &p, cudaStream_t s)
{
    const int nch = (p.n_groups + 31) / 32;
    if (nch <= 2) return launch_bf16_nch<R, 2>(p, s);
    if (nch <= 4) return launch_bf16_nch<R, 4>(p, s);
    if (nch <= 6) return launch_bf16_nch<R, 6>(p, s);
    if (nch <= 8) return launch_bf16_nch<R, 8>(p, s);
    if (nch <= 10) return launch_bf16_nch<R, 10>(p, s);
    return launch_bf16_nch<R, 8>(p, s);  // longer rows: several super-chunks
}

cudaError_t launch_gemv_bf16(const uint16_t *w, int64_t n_rows, int64_t k, const uint16_t *x,
                             const uint16_t *gamma, float eps, int epi, const float *residual, float *y,
                             cudaStream_t s)
{
    if (n_rows == 0) return cudaSuccess;
    Bf16Params p;
    p.w = w;
    p.x = x;
    p.gamma = gamma;
    p.residual = residual;
    p.y = y;
    p.n_rows = n_rows;
    p.half = n_rows / 2;
    p.n_out = (epi == QG_EPI_SILU_MUL_HALVES) ? n_rows / 2 : n_rows;
    p.k = static_cast<int>(k);
    p.n_groups = static_cast<int>(k / 8);
    p.inv_k = 1.0f / static_cast<float>(k);
    p.eps = eps;
    p.epi = epi;
    const bool silu = epi == QG_EPI_SILU_MUL_HALVES;
    const int64_t want_warps = static_cast<int64_t>(num_sms()) * 16;
    if (silu || n_rows / 2 >= want_warps) {
        p.n_tasks = silu ? p.half : (n_rows + 1) / 2;
        return launch_bf16_r<2>(p, s);
    }
    p.n_tasks = n_rows;
    return launch_bf16_r<1>(p, s);
}

}  // namespace qg
