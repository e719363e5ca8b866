// RMSNorm statistic on the GPU: r = 1 / sqrt(mean(x^2) + eps), evaluated as in
// f64 and rounded once to f32.
//
// GB300 runs f64 at a small fraction of its f32 rate, so a block-wide f64 sum
// would cost microseconds per CTA.  Instead each thread forms the exact square
// x*x = p + e (p = fl(x*x), e = fma(x, x, -p), Dekker's product) and adds both
// parts into a compensated pair (hi, lo) with Knuth's error-free two-sum; pairs
// are combined across the warp the same way and the per-warp pairs are added in
// f64 by one thread.  The sum carries about 48 significant bits, so r after the
// final f64 sqrt, division and rounding to f32 equals the f64-evaluated value
// except when that value lies within ~2^-40 (relative) of an f32 rounding
// boundary.
#pragma once

#include "qg_common.cuh"

namespace qg {

struct f32pair {
    float hi, lo;
};

// Knuth two-sum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void pair_add(f32pair &acc, float v)
{
    float s, e;
    two_sum(acc.hi, v, s, e);
    acc.hi = s;
    acc.lo = __fadd_rn(acc.lo, e);
}

// Add the exact square of x.
__device__ __forceinline__ void pair_add_square(f32pair &acc, float x)
{
    const float p = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -p);
    pair_add(acc, p);
    acc.lo = __fadd_rn(acc.lo, e);
}

__device__ __forceinline__ f32pair pair_merge(f32pair a, f32pair b)
{
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    f32pair r;
    r.hi = s;
    r.lo = __fadd_rn(__fadd_rn(a.lo, b.lo), e);
    return r;
}

__device__ __forceinline__ f32pair warp_pair_sum(f32pair v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        f32pair w;
        w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = pair_merge(v, w);
    }
    return v;
}

// Block-wide: every thread passes its pair; returns r to every thread.
// `scratch` holds 2 * (blockDim.x / 32) floats + 1; all threads must call.
__device__ __forceinline__ float block_rms_inv(f32pair v, int k, float eps, float *scratch)
{
    v = warp_pair_sum(v);
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        scratch[2 * warp] = v.hi;
        scratch[2 * warp + 1] = v.lo;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < nw; ++w) t += static_cast<double>(scratch[2 * w]);
        for (int w = 0; w < nw; ++w) t += static_cast<double>(scratch[2 * w + 1]);
        const double mean = t / static_cast<double>(k);
        scratch[2 * nw] = static_cast<float>(1.0 / sqrt(mean + static_cast<double>(eps)));
    }
    __syncthreads();
    return scratch[2 * nw];
}

}  // namespace qg
