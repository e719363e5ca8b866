// RMSNorm statistic on the GPU: r = 1 / sqrt(mean(x^2) + eps) rounded to f32,
// agreeing with an f64 evaluation of the same expression.
//
// GB300 runs f64 at a small fraction of its f32 rate (and f64 division and
// square root are long dependent chains), so everything here is f32 with
// error-free transformations:
//  * each thread forms the exact square x*x = p + e (p = fl(x*x),
//    e = fma(x, x, -p); Dekker's product) and adds both parts into a
//    compensated pair (hi, lo) with Knuth's two-sum; pairs are merged across the
//    warp and the block the same way;
//  * mean = s / k as a pair: m_hi = fl(s_hi * fl(1/k)) (any value within a few
//    ulp of s_hi / k will do), the remainder s_hi - m_hi k is exact through an
//    FMA, m_lo = (remainder + s_lo) / k to f32 accuracy; plus eps with a two-sum;
//  * y0 = rsqrtf(a), then one Newton-Taylor step r = y0 (1 + e/2 + 3e^2/8) with
//    the residual e = 1 - a y0^2 evaluated from exact products, and one final
//    f32 rounding.
// The result is within ~2^-46 (relative) of the real value before that final
// rounding, so it equals the f64-evaluated r except when the real value lies
// that close to a midpoint between two f32 numbers.
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

// r from the pair sum of squares; inv_k = fl(1 / k).
__device__ __forceinline__ float rms_inv_from_pair(f32pair s, int k, float inv_k, float eps)
{
    const float kf = static_cast<float>(k);  // exact: k < 2^24
    const float m_hi = __fmul_rn(s.hi, inv_k);
    const float rem = __fmaf_rn(-m_hi, kf, s.hi);  // s.hi - m_hi * k, exact
    const float m_lo = __fmul_rn(__fadd_rn(rem, s.lo), inv_k);
    float a_hi, a_e;
    two_sum(m_hi, eps, a_hi, a_e);
    float a_lo = __fadd_rn(a_e, m_lo);
    const float t = __fadd_rn(a_hi, a_lo);  // renormalise, |a_hi| >= |a_lo|
    a_lo = __fsub_rn(a_lo, __fsub_rn(t, a_hi));
    a_hi = t;
    if (a_hi == 0.0f) return __int_as_float(0x7f800000);  // 1/sqrt(0)
    if (isinf(a_hi)) return 0.0f;
    const float y0 = rsqrtf(a_hi);
    const float p = __fmul_rn(y0, y0);
    const float pe = __fmaf_rn(y0, y0, -p);        // y0^2 = p + pe
    const float th = __fmul_rn(a_hi, p);
    const float te = __fmaf_rn(a_hi, p, -th);      // a_hi p = th + te
    float e = __fsub_rn(1.0f, th);                 // exact: th is within [0.5, 2]
    e = __fsub_rn(e, te);
    e = __fmaf_rn(-a_hi, pe, e);
    e = __fmaf_rn(-a_lo, p, e);                    // e = 1 - a y0^2 (to ~2^-46)
    const float corr = __fmul_rn(y0, __fmul_rn(e, __fmaf_rn(0.375f, e, 0.5f)));
    return __fadd_rn(y0, corr);
}

// Block-wide: every thread passes its pair; returns r to every thread.
// `scratch` holds 2 * (blockDim.x / 32) + 1 floats; all threads must call.
__device__ __forceinline__ float block_rms_inv(f32pair v, int k, float inv_k, float eps, float *scratch)
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
        f32pair t = {scratch[0], scratch[1]};
        for (int w = 1; w < nw; ++w) t = pair_merge(t, f32pair{scratch[2 * w], scratch[2 * w + 1]});
        scratch[2 * nw] = rms_inv_from_pair(t, k, inv_k, eps);
    }
    __syncthreads();
    return scratch[2 * nw];
}

}  // namespace qg
