// RMSNorm, then the order-128 Walsh-Hadamard rotation of the normalised row,
// then Q8_0 of the rotated values: the rotated activation computed once, for
// every projection that reads the same input.
//
// "Filling in the blanks: Inference using Phobos", PrismML Ternary-Bonsai-2-27B:
// the format rotates the activation with a Hadamard matrix over its block of
// 128, which spreads outliers over the block, and the rotated activation can be
// computed once and shared by every projection reading that input (the weights
// carry the inverse rotation, applied once at load time: W x = (W H^T / 128)(H x)).
//
// One CTA per row.  r as in rmsnorm_quantize (compensated sum of exact squares,
// one rounding; qg_norm.cuh), x_hat = (x r) gamma, then each warp rotates
// 128-value chunks: lane l holds chunk values 4l .. 4l+3, the butterflies of
// strides 1 and 2 run in registers and those of strides 4 .. 64 across lanes
// (a + b in the lane holding a, a - b in the lane holding b), all in f32 in that
// fixed order; each 32-value block of the result is then quantized by its eight
// lanes exactly as rmsnorm_quantize quantizes x_hat.
#include "qg_common.cuh"
#include "qg_norm.cuh"

namespace qg {

constexpr int ROT_THREADS = 256;

__device__ __forceinline__ void bfly(float &a, float &b)
{
    const float s = __fadd_rn(a, b), d = __fsub_rn(a, b);
    a = s;
    b = d;
}

__global__ void __launch_bounds__(ROT_THREADS) rmsnorm_hadamard_quantize_kernel(
    const float *__restrict__ x, const float *__restrict__ gamma, int k, float inv_k, float eps,
    int8_t *__restrict__ q, uint16_t *__restrict__ d, float *__restrict__ z_out, float *__restrict__ inv_rms)
{
    __shared__ float scratch[2 * (ROT_THREADS / 32) + 1];
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x;
    const float *xr = x + static_cast<int64_t>(row) * k;
    f32pair acc = {0.0f, 0.0f};
    for (int i = threadIdx.x * 4; i < k; i += ROT_THREADS * 4) {
        const float4 v = *reinterpret_cast<const float4 *>(xr + i);
        pair_add_square(acc, v.x);
        pair_add_square(acc, v.y);
        pair_add_square(acc, v.z);
        pair_add_square(acc, v.w);
    }
    const float r = block_rms_inv(acc, k, inv_k, eps, scratch);
    if (threadIdx.x == 0 && inv_rms) inv_rms[row] = r;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = k / QK;
    for (int c = warp; c < k / 128; c += ROT_THREADS / 32) {
        const int o = 128 * c + 4 * lane;
        const float4 xv = *reinterpret_cast<const float4 *>(xr + o);
        const float4 gv = *reinterpret_cast<const float4 *>(gamma + o);
        float v0 = __fmul_rn(__fmul_rn(xv.x, r), gv.x);
        float v1 = __fmul_rn(__fmul_rn(xv.y, r), gv.y);
        float v2 = __fmul_rn(__fmul_rn(xv.z, r), gv.z);
        float v3 = __fmul_rn(__fmul_rn(xv.w, r), gv.w);
        bfly(v0, v1);  // stride 1
        bfly(v2, v3);
        bfly(v0, v2);  // stride 2
        bfly(v1, v3);
#pragma unroll
        for (int m = 1; m <= 16; m <<= 1) {  // strides 4 m: partner lane l ^ m
            const bool hi = (lane & m) != 0;
            const float p0 = __shfl_xor_sync(0xffffffffu, v0, m), p1 = __shfl_xor_sync(0xffffffffu, v1, m);
            const float p2 = __shfl_xor_sync(0xffffffffu, v2, m), p3 = __shfl_xor_sync(0xffffffffu, v3, m);
            v0 = hi ? __fsub_rn(p0, v0) : __fadd_rn(v0, p0);
            v1 = hi ? __fsub_rn(p1, v1) : __fadd_rn(v1, p1);
            v2 = hi ? __fsub_rn(p2, v2) : __fadd_rn(v2, p2);
            v3 = hi ? __fsub_rn(p3, v3) : __fadd_rn(v3, p3);
        }
        const float4 zv = make_float4(v0, v1, v2, v3);
        if (z_out) *reinterpret_cast<float4 *>(z_out + static_cast<int64_t>(row) * k + o) = zv;
        // Q8_0 of the rotated block held by lanes 8 g .. 8 g + 7
        float mx = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        const float dd = div127(mx);
        *reinterpret_cast<uint32_t *>(q + static_cast<int64_t>(row) * k + o) = q8_pack4(zv, dd, q8_recip(dd));
        if ((lane & 7) == 0) d[static_cast<int64_t>(row) * nb + 4 * c + (lane >> 3)] = f2h_rn(dd);
    }
}

cudaError_t launch_rmsnorm_hadamard_quantize(const float *x, const float *gamma, int64_t rows, int64_t k, float eps,
                                             int8_t *q, uint16_t *d, float *z_out, float *inv_rms, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    return launch_pdl(rmsnorm_hadamard_quantize_kernel, dim3(static_cast<unsigned>(rows)), dim3(ROT_THREADS), 0, s, x,
                      gamma, static_cast<int>(k), 1.0f / static_cast<float>(k), eps, q, d, z_out, inv_rms);
}

}  // namespace qg
