// Activation quantization, RMSNorm + quantization, and Q8_0 weight packing.
//
// Q8_0 block ("Filling in the blanks: Inference using Phobos", Fast Decode):
// 32 int8 values sharing one scale.  Scale d = max|x|/127 in f32, code
// q = round half away from zero of x/d, stored scale binary16(d).
#include "qg_common.cuh"
#include "qg_norm.cuh"

namespace qg {

// x[rows][k] -> q[rows][k], d[rows][k/32].  Eight lanes per 32-value block,
// four values per lane (one 16-byte load of x and one store of codes per
// lane); a warp covers four blocks.  Lanes past the end take part in the
// shuffles with zeros and skip the stores.
__global__ void __launch_bounds__(256) quantize_act_kernel(const float *__restrict__ x, int64_t n_blocks,
                                                           int8_t *__restrict__ q, uint16_t *__restrict__ d)
{
    pdl_wait();
    pdl_trigger();
    const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
    const int sub = threadIdx.x & 7;
    const bool live = blk < n_blocks;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) v = *reinterpret_cast<const float4 *>(x + blk * QK + sub * 4);
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    if (!live) return;
    const float dd = div127(m);
    const float rd = q8_recip(dd);
    reinterpret_cast<uint32_t *>(q + blk * QK)[sub] = q8_pack4(v, dd, rd);
    if (sub == 0) d[blk] = f2h_rn(dd);
}

// The same quantization written as the operand tiles of the tensor-core prompt
// contraction: for each tile of 128 rows and each block j one record of
// ACT_TILE_RECORD bytes, the codes as binary16 values (exact: |q| <= 127) in
// four groups of eight, code 8g+e of tile row r at byte 2048 g + 16 r + 2 e,
// then the 128 binary16 scales.  Rows past the end of the last tile are zero.
// Eight lanes per (row, block) with the tile row fastest, so a warp's stores
// fill 64 contiguous bytes of each group.
__global__ void __launch_bounds__(256) quantize_act_tiles_kernel(const float *__restrict__ x, int64_t rows, int nb,
                                                                 int64_t n_groups, uint8_t *__restrict__ xt)
{
    pdl_wait();
    pdl_trigger();
    const int64_t gidx = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
    if (gidx >= n_groups) return;  // n_groups is a multiple of 128: whole warps leave together
    const int sub = threadIdx.x & 7;
    const int r = static_cast<int>(gidx & (ACT_TILE_ROWS - 1));
    const int64_t rec = gidx >> 7;  // tile * nb + block
    const int64_t tile = rec / nb;
    const int j = static_cast<int>(rec - tile * nb);
    const int64_t row = tile * ACT_TILE_ROWS + r;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < rows) v = *reinterpret_cast<const float4 *>(x + (row * nb + j) * QK + sub * 4);
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const float dd = div127(m);
    const float rd = q8_recip(dd);
    const uint32_t c0 = __half_as_ushort(__int2half_rn(q8_code(v.x, dd, rd)));
    const uint32_t c1 = __half_as_ushort(__int2half_rn(q8_code(v.y, dd, rd)));
    const uint32_t c2 = __half_as_ushort(__int2half_rn(q8_code(v.z, dd, rd)));
    const uint32_t c3 = __half_as_ushort(__int2half_rn(q8_code(v.w, dd, rd)));
    uint8_t *base = xt + rec * ACT_TILE_RECORD;
    *reinterpret_cast<uint2 *>(base + (sub >> 1) * 2048 + r * 16 + (sub & 1) * 8) =
        make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
    if (sub == 0) *reinterpret_cast<uint16_t *>(base + 8192 + r * 2) = f2h_rn(dd);
}

// One CTA per row.  r = 1/sqrt(mean(x^2) + eps) evaluated as in f64 and rounded
// once to f32 (compensated sum of exact squares, see qg_norm.cuh), then
// x_hat = (x * r) * gamma and Q8_0 quantization of x_hat ("One level down: #002
// the same compiler on a GPU", Emitting for a GPU: the normalization feeds the
// projection).
constexpr int NORM_THREADS = 256;

__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_quantize_kernel(
    const float *__restrict__ x, const float *__restrict__ gamma, int k, float inv_k, float eps,
    int8_t *__restrict__ q, uint16_t *__restrict__ d, float *__restrict__ inv_rms)
{
    __shared__ float scratch[2 * (NORM_THREADS / 32) + 1];
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x;
    const float *xr = x + static_cast<int64_t>(row) * k;
    f32pair acc = {0.0f, 0.0f};
    for (int i = threadIdx.x * 4; i < k; i += NORM_THREADS * 4) {
        const float4 v = *reinterpret_cast<const float4 *>(xr + i);
        pair_add_square(acc, v.x);
        pair_add_square(acc, v.y);
        pair_add_square(acc, v.z);
        pair_add_square(acc, v.w);
    }
    const float r = block_rms_inv(acc, k, inv_k, eps, scratch);
    if (threadIdx.x == 0 && inv_rms) inv_rms[row] = r;
    // quantize x_hat = (x * r) * gamma, eight lanes per block
    const int nb = k / QK;
    const int sub = threadIdx.x & 7;
    for (int b0 = 0; b0 < nb; b0 += NORM_THREADS / 8) {
        const int b = b0 + (threadIdx.x >> 3);
        const bool live = b < nb;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
            const float4 xv = *reinterpret_cast<const float4 *>(xr + b * QK + sub * 4);
            const float4 gv = *reinterpret_cast<const float4 *>(gamma + b * QK + sub * 4);
            v.x = __fmul_rn(__fmul_rn(xv.x, r), gv.x);
            v.y = __fmul_rn(__fmul_rn(xv.y, r), gv.y);
            v.z = __fmul_rn(__fmul_rn(xv.z, r), gv.z);
            v.w = __fmul_rn(__fmul_rn(xv.w, r), gv.w);
        }
        float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        if (live) {
            const float dd = div127(m);
            int8_t *qb = q + static_cast<int64_t>(row) * k + b * QK;
            reinterpret_cast<uint32_t *>(qb)[sub] = q8_pack4(v, dd, q8_recip(dd));
            if (sub == 0) d[static_cast<int64_t>(row) * nb + b] = f2h_rn(dd);
        }
    }
}

// Canonical 34-byte blocks -> planes.  One thread per block; byte loads (the
// source is only 2-byte aligned per block), two 16-byte stores of values.
// This kernel does not trigger its dependents early: a following GEMV may
// start streaming the weights only after the planes are complete.
__global__ void __launch_bounds__(256) pack_q8_0_kernel(const uint8_t *__restrict__ blocks, int64_t n_blocks,
                                                         int8_t *__restrict__ qs, uint16_t *__restrict__ d)
{
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n_blocks) return;
    const uint8_t *src = blocks + i * 34;
    d[i] = static_cast<uint16_t>(src[0] | (static_cast<uint16_t>(src[1]) << 8));
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        w[j] = static_cast<uint32_t>(src[2 + 4 * j]) | (static_cast<uint32_t>(src[3 + 4 * j]) << 8) |
               (static_cast<uint32_t>(src[4 + 4 * j]) << 16) | (static_cast<uint32_t>(src[5 + 4 * j]) << 24);
    uint4 *dst = reinterpret_cast<uint4 *>(qs + i * QK);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Row-major planes -> column-block-major planes: block b of row n moves to
// qs_cb[b][n][0..31], its scale to d_cb[b][n], so the n_rows blocks of one
// column block are contiguous.  One thread per block; like the pack above it
// does not trigger its dependents early.
__global__ void __launch_bounds__(256) column_blocks_kernel(const int8_t *__restrict__ qs,
                                                            const uint16_t *__restrict__ d, int64_t n_rows, int nb,
                                                            int8_t *__restrict__ qs_cb, uint16_t *__restrict__ d_cb)
{
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // n * nb + b
    if (i >= n_rows * nb) return;
    const int64_t n = i / nb;
    const int b = static_cast<int>(i - n * nb);
    const uint4 *src = reinterpret_cast<const uint4 *>(qs + i * QK);
    uint4 *dst = reinterpret_cast<uint4 *>(qs_cb + (static_cast<int64_t>(b) * n_rows + n) * QK);
    dst[0] = src[0];
    dst[1] = src[1];
    d_cb[static_cast<int64_t>(b) * n_rows + n] = d[i];
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
cudaError_t launch_quantize_act(const float *x, int64_t rows, int64_t k, int8_t *q, uint16_t *d,
                                cudaStream_t s)
{
    const int64_t n_blocks = rows * (k / QK);
    if (n_blocks == 0) return cudaSuccess;
    const int64_t threads = n_blocks * 8;
    const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
    return launch_pdl(quantize_act_kernel, dim3(grid), dim3(256), 0, s, x, n_blocks, q, d);
}

cudaError_t launch_quantize_act_tiles(const float *x, int64_t rows, int64_t k, void *xt, cudaStream_t s)
{
    const int nb = static_cast<int>(k / QK);
    const int64_t n_groups = act_tiles(rows) * nb * ACT_TILE_ROWS;
    if (n_groups == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((n_groups * 8 + 255) / 256);
    return launch_pdl(quantize_act_tiles_kernel, dim3(grid), dim3(256), 0, s, x, rows, nb, n_groups,
                      static_cast<uint8_t *>(xt));
}

cudaError_t launch_rmsnorm_quantize(const float *x, const float *gamma, int64_t rows, int64_t k, float eps,
                                    int8_t *q, uint16_t *d, float *inv_rms, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    return launch_pdl(rmsnorm_quantize_kernel, dim3(static_cast<unsigned>(rows)), dim3(NORM_THREADS), 0, s, x,
                      gamma, static_cast<int>(k), 1.0f / static_cast<float>(k), eps, q, d, inv_rms);
}

cudaError_t launch_pack_q8_0(const void *blocks, int64_t n_rows, int64_t k, int8_t *qs, uint16_t *d,
                             cudaStream_t s)
{
    const int64_t n_blocks = n_rows * (k / QK);
    if (n_blocks == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((n_blocks + 255) / 256);
    return launch_pdl(pack_q8_0_kernel, dim3(grid), dim3(256), 0, s, static_cast<const uint8_t *>(blocks),
                      n_blocks, qs, d);
}

cudaError_t launch_column_blocks(const int8_t *qs, const uint16_t *d, int64_t n_rows, int64_t k, int8_t *qs_cb,
                                 uint16_t *d_cb, cudaStream_t s)
{
    const int64_t n_blocks = n_rows * (k / QK);
    if (n_blocks == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((n_blocks + 255) / 256);
    return launch_pdl(column_blocks_kernel, dim3(grid), dim3(256), 0, s, qs, d, n_rows, static_cast<int>(k / QK), qs_cb,
                      d_cb);
}

}  // namespace qg
