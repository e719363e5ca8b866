// Decode-step kernels whose whole weight slab is requested before they wait on
// the kernel that produces their input.
//
// "Filling in the blanks: Inference using Phobos", Fast Decode: decode is a
// pure weight stream; the activation is quantized once and shared, projections
// that read it are stacked, the residual add is folded into the matmul, and the
// pass is replayed as a graph.  "One level down: #002 the same compiler on a
// GPU", Emitting for a GPU: the normalization is fused with the projection that
// follows it and the activation with the projection before it.
//
// GB300 design.  A decode FFN layer moves 11.7 MB, about 1.7 us of HBM time,
// but it is a chain of dependent steps (norm -> gate|up -> down) each of which
// needs a full reduction of its predecessor's output.  Launched as separate
// grids, every step pays launch ramp-up plus one DRAM round trip before its
// weights arrive.  Here each kernel is a single wave whose CTAs copy their whole
// weight slab (values, scales, gain) into shared memory with bulk copies issued
// BEFORE griddepcontrol.wait (~30-85 KB per CTA).  Kernels further down the
// stream therefore become resident and stream their weights while their
// predecessors still compute; after the wait only on-chip work remains.
// (Plain loads into registers would not do: the compiler may legally sink
// read-only loads below the wait.)
//
// When each kernel releases its dependent launch is tuned for the decode layer
// (gate|up, then down, then the next layer's gate|up): the GEMV releases it on
// entry, so the next layer's gate|up stages its slab during this layer's whole
// chain, but the gate|up kernel releases the down GEMV only once its own wait
// has returned, so that the GEMV's CTAs are not resident on the SMs before the
// gate|up chain starts.  Measured over 24 layers on GB300: 102.5 us a step,
// against 117 with both releases on entry, 137 with both after the wait and 147
// with the gate|up release on entry and the GEMV's after its wait.
//
// Shared-memory reads are laid out so that every quarter-warp phase touches 32
// distinct banks: in the GEMV kernels lane j reads the 32-byte block j of a row
// as two 16-byte halves, half (j >> 2) & 1 first (activation words paired in the
// same order); ffn_up_kernel stages its rows 16 bytes apart (see there).
//
//  * ffn_up_kernel: RMSNorm + Q8_0 quantization of x (every CTA, from L2),
//    stacked gate|up block dots, SiLU(g)*u, and Q8_0 quantization of each
//    32-output block of h (a CTA owns whole blocks), so the down projection
//    reads codes directly.
//  * gemv_prefetch_kernel: batch-1 Q8_0 GEMV over pre-quantized input with the
//    NONE or RESIDUAL epilogue (the down projection, and small GEMVs).
//  * ffn_up_kernel<NBL, true>: the whole layer in one launch.  The down
//    projection is split along its reduction: the CTA that owns block b of h
//    also stages column block b of the down weights (hidden rows x 32 codes,
//    contiguous in the column-block layout of qg_q8_0_column_blocks) and, once
//    its h block is quantized, forms that block's Q8_0 term of every output.
//    The CTAs of a thread-block cluster (up to 8) add their terms through
//    distributed shared memory, each CTA one slice of the outputs, and every
//    cluster stores its partial output vector.  The layer's output is left
//    unreduced as (r, partials): the next layer (or qg_decode_layer_finish)
//    forms x = r + sum of the partials in a fixed order while it loads its
//    input anyway, so no float atomics and no extra pass are needed and the
//    result is the same on every run.

#include "qg_common.cuh"
#include "qg_norm.cuh"

namespace qg {

// ---------------------------------------------------------------------------
// shared pieces
// ---------------------------------------------------------------------------

// Waits on staged weight copies that gave up (the one-second limit) in the
// kernels of this file, on this GPU: a CTA (gate|up, one-launch layer) or a warp
// (down GEMV) counts one.  Read and cleared through copy_stalls.
static __device__ unsigned int g_copy_stalls;

__device__ __forceinline__ void count_copy_stall(bool counter_thread)
{
    if (counter_thread) atomicAdd(&g_copy_stalls, 1u);
}

// S * (d_w * d_x) accumulated the same way as the streaming GEMV kernels.
__device__ __forceinline__ float block_term(const u32x8 &w, const u32x8 &x, float dw, float dx, float acc)
{
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s = dp4a(w.v[i], x.v[i], s);
    return fmaf(small_int_to_float(s), dw * dx, acc);
}

// Order-128 Walsh-Hadamard transform (Sylvester order, unnormalised) of the 128
// values a warp holds, lane l holding values 4 l .. 4 l + 3: butterflies of
// strides 1 and 2 in registers, then strides 4 .. 64 across lanes (a + b in the
// lane holding a, a - b in the lane holding b), in f32, in that order (the order
// of rmsnorm_hadamard_quantize, so both give the same bits).
__device__ __forceinline__ float4 hadamard128_lane4(float4 v, int lane)
{
    auto bf = [](float &a, float &b) {
        const float s = __fadd_rn(a, b), d = __fsub_rn(a, b);
        a = s;
        b = d;
    };
    bf(v.x, v.y);
    bf(v.z, v.w);
    bf(v.x, v.z);
    bf(v.y, v.w);
#pragma unroll
    for (int m = 1; m <= 16; m <<= 1) {
        const bool hi = (lane & m) != 0;
        const float p0 = __shfl_xor_sync(0xffffffffu, v.x, m), p1 = __shfl_xor_sync(0xffffffffu, v.y, m);
        const float p2 = __shfl_xor_sync(0xffffffffu, v.z, m), p3 = __shfl_xor_sync(0xffffffffu, v.w, m);
        v.x = hi ? __fsub_rn(p0, v.x) : __fadd_rn(v.x, p0);
        v.y = hi ? __fsub_rn(p1, v.y) : __fadd_rn(v.y, p1);
        v.z = hi ? __fsub_rn(p2, v.z) : __fadd_rn(v.z, p2);
        v.w = hi ? __fsub_rn(p3, v.w) : __fadd_rn(v.w, p3);
    }
    return v;
}

__device__ __forceinline__ void zero(u32x8 &w)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) w.v[i] = 0u;
}

// 32-byte block at p (16-byte aligned), half c0 first.
__device__ __forceinline__ u32x8 ld_block_halves(const int8_t *p, int c0)
{
    const uint4 a = *reinterpret_cast<const uint4 *>(p + 16 * c0);
    const uint4 b = *reinterpret_cast<const uint4 *>(p + 16 * (c0 ^ 1));
    u32x8 r;
    r.v[0] = a.x; r.v[1] = a.y; r.v[2] = a.z; r.v[3] = a.w;
    r.v[4] = b.x; r.v[5] = b.y; r.v[6] = b.z; r.v[7] = b.w;
    return r;
}

__device__ __forceinline__ int lane_half(int lane) { return (lane >> 2) & 1; }


// ---------------------------------------------------------------------------
// gate|up with the norm in front and SiLU + quantization behind
// ---------------------------------------------------------------------------
constexpr int kMaxLayerPartials = 16;  // partial vectors a one-launch layer reads

struct FfnUpParams {
    const float *x;       // [k] input row (written by the previous kernel)
    const float *gamma;   // [k]
    const int8_t *w_qs;   // stacked [2F][k]
    const uint16_t *w_d;  // [2F][k/32]
    float *h;             // [F] silu(g) * u
    int8_t *hq;           // [F] Q8_0 codes of h
    uint16_t *hd;         // [F/32] binary16 scales of h
    int8_t *xq_out;       // optional [k]   (written by CTA 0)
    uint16_t *xd_out;     // optional [k/32]
    float *r_out;         // optional [1]
    int k;
    int nb;
    int64_t half;         // F
    float inv_k;          // fl(1 / k)
    float eps;
    // one-launch layer only (x above is r_in, the unreduced base of the input)
    const float *p_in;         // [n_in][k] partials of the input (x = r_in + sum over them)
    int n_in;
    float *r_next;             // [k] this layer's input, x (written by CTA 0)
    float *p_out;              // [F/32 / cluster][k] this layer's down partials, one per cluster
    const int8_t *wdn_qs;      // down values, column-block layout [F/32][k][32]
    const uint16_t *wdn_d;     // down scales, column-block layout [F/32][k]
    int cluster;               // CTAs per cluster (divides F/32)
};

__host__ __device__ constexpr size_t ffn_up_smem_bytes(int k, bool down = false)
{
    // values [64][k + 16] | scales [64][k/32] u16 | gamma [k] f32 | row partials [warps][64] f32
    // | warp partial pairs [2 * 16] f32
    // | (two-launch) the scales again, f32, in dot order [k/32][64]
    // | (one-launch layer) down column block [k][32] int8 | its scales [k] u16 | h codes [32]
    //   | h scale f32 (16 B); this CTA's terms of every output, [k] f32, reuse the values' space
    //   (dead once h is formed), so that two CTAs fit on an SM for k = 1024
    return static_cast<size_t>(64) * (k + 16) + 64 * (k / 32) * 2 + 4 * k +
           static_cast<size_t>(2048) * ((k + 1023) / 1024) + 4 * 32 +
           (down ? static_cast<size_t>(32) * k + 2 * k + 32 + 16 : static_cast<size_t>(8) * k);
}

// One CTA per 32-output block of h (rows o..o+31 of gate and of up).
// NBL = ceil(k / 1024); 8 NBL warps.  Warp w = wl + 8 wh (wl < 8) owns the four
// K blocks wl + 8 c + 32 wh (c < 4) of x and of all 64 stacked rows:
//  * thread (w, l) holds x values 4 (l % 8) .. +3 of block wl + 8 (l / 8) + 32 wh,
//    so the eight lanes of a block quantize it without leaving the warp, and the
//    same eight lanes then dot that block against rows l % 8 + 8 i (i < 8), the
//    block's codes passed around by shuffles;
//  * staged rows are k + 16 bytes apart, so the eight lanes of a quarter-warp
//    read eight different bank groups;
//  * the four lane groups are summed first (lane offsets 16 and 8: block index
//    bits 4 and 3), then the warps in shared memory (bits 2, 1, 0), which is the
//    order of the streaming GEMV's butterfly over 32 lanes: for k <= 1024, h has
//    the bits that rmsnorm_quantize -> qgemv_q8_0(SiLU) gives.
// Before the wait one CTA barrier agrees that the slab has landed; after it,
// while x is loaded, the weight scales are rewritten as f32 in dot order, and
// two barriers follow: the norm statistic's and the row partials'; warp 0 then
// forms h = SiLU(g) u and its Q8_0 block.
template <int NBL, bool DOWN, bool ROT = false>
__global__ void __launch_bounds__(256 * NBL) ffn_up_kernel(const FfnUpParams p)
{
    static_assert(!ROT || (NBL == 1 && !DOWN), "the rotated form serves k <= 1024, two-launch layers");
    constexpr int NW = 8 * NBL;  // warps per CTA
    extern __shared__ __align__(16) uint8_t smem[];
    const int K = p.k, nb = p.nb, KP = K + 16;
    int8_t *s_w = reinterpret_cast<int8_t *>(smem);
    uint16_t *s_wd = reinterpret_cast<uint16_t *>(smem + 64 * KP);
    float *s_gamma = reinterpret_cast<float *>(smem + 64 * KP + 128 * nb);
    float *s_red = s_gamma + K;       // [NW][64]
    float *s_part = s_red + NW * 64;  // [2 * NW]
    // (!DOWN) [nb][2][8][4]: scale of row g + 8 i, block b at ((2 b + i / 4) 8 + g) 4 + i % 4
    float *s_wdf = s_part + 32;
    int8_t *s_dn = reinterpret_cast<int8_t *>(s_part + 32);         // [K][32] (DOWN)
    uint16_t *s_dnd = reinterpret_cast<uint16_t *>(s_dn + 32 * K);  // [K]     (DOWN)
    int8_t *s_hq = reinterpret_cast<int8_t *>(s_dnd + K);           // [32]    (DOWN)
    float *s_hd = reinterpret_cast<float *>(s_hq + 32);             // [1]     (DOWN)
    float *s_out = reinterpret_cast<float *>(smem);                 // [K]     (DOWN, over the values)

    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int64_t ob = static_cast<int64_t>(blockIdx.x) * 32;

    __shared__ __align__(8) uint64_t s_bar;

    // ---- stage everything that does not depend on the previous kernel -------
    // Bulk copies issued by one thread are serviced one after another, so they
    // are spread over lanes: warp 0 copies the 64 rows (two per lane), warp 1
    // gamma, the two scale slabs and (one-launch layer) the down column block;
    // all complete on s_bar.
    if (t == 0) {
        mbar_init(&s_bar, 1);
        mbar_expect_tx(&s_bar, 4u * K + 128u * nb + 64u * K + (DOWN ? 34u * K : 0u));
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = lane + 32 * h;  // stacked: gate rows, then up rows
            const int64_t src = h == 0 ? ob + lane : p.half + ob + lane;
            bulk_copy_g2s(s_w + row * KP, p.w_qs + src * K, static_cast<uint32_t>(K), &s_bar, l2_evict_first_policy());
        }
    } else if (warp == 1) {
        if (DOWN && lane >= 3 && lane < 8) {
            // down column block b: four value pieces of K/4 rows x 32 bytes, then the K scales
            const int v = lane - 3;
            const int64_t cb = static_cast<int64_t>(blockIdx.x) * K;
            void *dst = v < 4 ? static_cast<void *>(s_dn + v * 8 * K) : static_cast<void *>(s_dnd);
            const void *src = v < 4 ? static_cast<const void *>(p.wdn_qs + (cb + v * (K / 4)) * QK)
                                    : static_cast<const void *>(p.wdn_d + cb);
            bulk_copy_g2s(dst, src, v < 4 ? 8u * K : 2u * K, &s_bar, l2_evict_first_policy());
        }
        if (lane < 3) {
            const int64_t srow = lane == 1 ? ob : p.half + ob;
            void *dst = lane == 0 ? static_cast<void *>(s_gamma) : static_cast<void *>(s_wd + (lane - 1) * 32 * nb);
            const void *src = lane == 0 ? static_cast<const void *>(p.gamma) : static_cast<const void *>(p.w_d + srow * nb);
            const uint32_t bytes = lane == 0 ? 4u * K : 64u * nb;
            bulk_copy_g2s(dst, src, bytes, &s_bar, lane == 0 ? l2_evict_last_policy() : l2_evict_first_policy());
        }
    }

    // Still before the wait, the threads see the slab land, asleep in the
    // barrier unit: a spin here would take issue slots from the kernel whose
    // chain runs on this SM (measured: 2 us a step).  A copy that has not landed
    // within the limit leaves NaN outputs for this block.
    const bool ok = mbar_wait_sleep_bounded(&s_bar, 0, kCopyWaitLimitNs);
    const bool staged = __syncthreads_and(ok);
    pdl_wait();
    pdl_trigger();  // the dependent (the layer's down GEMV) only now: see the top of the file

    const int wl = warp & 7, wh = warp >> 3;
    // block of this thread's four x values (and of its dots); the rotated form
    // gives warp w the blocks 4 w .. 4 w + 3, one 128-value block of the rotation,
    // lane l holding its values 4 l .. 4 l + 3
    const int xb = ROT ? 4 * wl + (lane >> 3) : wl + 8 * (lane >> 3) + 32 * wh;
    const int xo = 32 * xb + 4 * (lane & 7);        // their offset in x
    const bool live = xb < nb;
    const int rg = lane & 7;                        // this lane's rows: rg + 8 i

    float4 xv4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) xv4 = *reinterpret_cast<const float4 *>(p.x + xo);
    // While x is on its way from L2: the gate|up scales to f32 in the order the
    // dots read them, so a lane's eight scales are two 16-byte words and a
    // quarter-warp reads 128 contiguous bytes (published by the norm barrier).
    if (!DOWN && staged) {
        for (int e = t; e < 8 * nb; e += blockDim.x) {
            const int b = e >> 3, g = e & 7;
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = h2f(s_wd[(g + 8 * i) * nb + b]);
            *reinterpret_cast<float4 *>(s_wdf + (2 * b * 8 + g) * 4) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(s_wdf + ((2 * b + 1) * 8 + g) * 4) = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    if constexpr (DOWN) {
        // x = r + partials of the previous layer, all loads first, then the sum
        // in partial order (the order qg_decode_layer_finish uses)
        constexpr int MAXP = kMaxLayerPartials;
        float4 pv[MAXP];
#pragma unroll
        for (int c = 0; c < MAXP; ++c)
            if (c < p.n_in && live) pv[c] = *reinterpret_cast<const float4 *>(p.p_in + static_cast<int64_t>(c) * K + xo);
#pragma unroll
        for (int c = 0; c < MAXP; ++c) {
            if (c < p.n_in && live) {
                xv4.x += pv[c].x;
                xv4.y += pv[c].y;
                xv4.z += pv[c].z;
                xv4.w += pv[c].w;
            }
        }
        if (blockIdx.x == 0 && live) *reinterpret_cast<float4 *>(p.r_next + xo) = xv4;
    }

    // ---- RMSNorm statistic ---------------------------------------------------
    f32pair acc = {0.0f, 0.0f};
    if (live) {
        pair_add_square(acc, xv4.x);
        pair_add_square(acc, xv4.y);
        pair_add_square(acc, xv4.z);
        pair_add_square(acc, xv4.w);
    }
    acc = warp_pair_sum(acc);
    if (lane == 0) {
        s_part[2 * warp] = acc.hi;
        s_part[2 * warp + 1] = acc.lo;
    }
    __syncthreads();
    if (!staged) {
        count_copy_stall(t == 0);
        if (warp == 0) {
            p.h[ob + lane] = __int_as_float(0x7fc00000);
            p.hq[ob + lane] = 0;
            if (lane == 0) p.hd[blockIdx.x] = 0x7e00;
        }
        mbar_wait_bounded(&s_bar, 0, kCopyWaitLimitNs);
        // the one-launch layer still takes part in its cluster's reduction (NaN terms)
        if constexpr (!DOWN) return;
    }
    if (staged) {
    // every group of NW lanes merges the NW warp partials in one xor butterfly;
    // pair_merge is exactly commutative, so every lane ends with the same total
    f32pair tot = f32pair{s_part[2 * (lane % NW)], s_part[2 * (lane % NW) + 1]};
    float4 g4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) g4 = *reinterpret_cast<const float4 *>(s_gamma + xo);
#pragma unroll
    for (int off = NW / 2; off >= 1; off >>= 1) {
        f32pair o;
        o.hi = __shfl_xor_sync(0xffffffffu, tot.hi, off);
        o.lo = __shfl_xor_sync(0xffffffffu, tot.lo, off);
        tot = pair_merge(tot, o);
    }
    const float r = rms_inv_from_pair(tot, K, p.inv_k, p.eps);

    // ---- Q8_0 quantization of x_hat = (x * r) * gamma, eight threads per block
    uint32_t xc = 0u;  // this thread's four codes
    float xdf = 0.0f;  // its block's scale (binary16 value)
    {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
            v.x = __fmul_rn(__fmul_rn(xv4.x, r), g4.x);
            v.y = __fmul_rn(__fmul_rn(xv4.y, r), g4.y);
            v.z = __fmul_rn(__fmul_rn(xv4.z, r), g4.z);
            v.w = __fmul_rn(__fmul_rn(xv4.w, r), g4.w);
        }
        if constexpr (ROT) v = hadamard128_lane4(v, lane);
        float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        if (live) {
            const float dd = div127(m);
            xc = q8_pack4(v, dd, q8_recip(dd));
            const uint16_t dbits = f2h_rn(dd);
            xdf = h2f(dbits);
            if (blockIdx.x == 0) {
                if (p.xq_out) reinterpret_cast<uint32_t *>(p.xq_out)[xo / 4] = xc;
                if (p.xd_out && (lane & 7) == 0) p.xd_out[xb] = dbits;
            }
        }
        if (blockIdx.x == 0 && t == 0 && p.r_out) *p.r_out = r;
    }

    // ---- block dots: block xb of rows rg + 8 i ---------------------------------
    // word s of the block is held by lane 8 (lane / 8) + s
    u32x8 xw;
    const int src = lane & 24;
#pragma unroll
    for (int s = 0; s < 8; ++s) xw.v[s] = __shfl_sync(0xffffffffu, xc, src + s);
    const float xs = __shfl_sync(0xffffffffu, xdf, src);
    // the eight rows' blocks, then their dots
    float part[8];
    if (DOWN && live) {
        // (the one-launch layer keeps no f32 copy of the scales: shared memory)
        u32x8 wv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) wv[i] = ld_block_halves(s_w + (rg + 8 * i) * KP + xb * QK, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) part[i] = block_term(wv[i], xw, h2f(s_wd[(rg + 8 * i) * nb + xb]), xs, 0.0f);
    } else if (live) {
        const float4 sa = *reinterpret_cast<const float4 *>(s_wdf + ((2 * xb) * 8 + rg) * 4);
        const float4 sb = *reinterpret_cast<const float4 *>(s_wdf + ((2 * xb + 1) * 8 + rg) * 4);
        const float sc[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
        u32x8 wv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) wv[i] = ld_block_halves(s_w + (rg + 8 * i) * KP + xb * QK, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) part[i] = block_term(wv[i], xw, sc[i], xs, 0.0f);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) part[i] = 0.0f;
    }
    // the four lane groups of a row: offset 16 (block bit 4), then 8 (bit 3); a
    // lane keeps half of its values each time and ends with rows rg + 8 (2 (lane / 8) + k)
    float v4[4], v2[2];
    {
        const bool up = (lane & 16) != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float send = up ? part[k] : part[k + 4];
            const float keep = up ? part[k + 4] : part[k];
            v4[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    {
        const bool up = (lane & 8) != 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float send = up ? v4[k] : v4[k + 2];
            const float keep = up ? v4[k + 2] : v4[k];
            v2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) s_red[warp * 64 + rg + 8 * (2 * (lane >> 3) + k)] = v2[k];
    __syncthreads();

    // ---- warp 0: row totals over the warps (block bits 2, 1, 0: warp offsets 4,
    // 2, 1), SiLU(g) u, and the Q8_0 block of h ----------------------------------
    if (warp == 0) {
        auto row_total = [&](int row) {
            const float *c = s_red + row;
            float s = ((c[0] + c[4 * 64]) + (c[2 * 64] + c[6 * 64])) + ((c[64] + c[5 * 64]) + (c[3 * 64] + c[7 * 64]));
            if constexpr (NBL == 2) {
                c += 8 * 64;
                s += ((c[0] + c[4 * 64]) + (c[2 * 64] + c[6 * 64])) + ((c[64] + c[5 * 64]) + (c[3 * 64] + c[7 * 64]));
            }
            return s;
        };
        const float v = silu_mul(row_total(lane), row_total(32 + lane));
        p.h[ob + lane] = v;
        const float m = warp_max_abs(v);
        const float dd = div127(m);
        const int8_t code = static_cast<int8_t>(q8_code(v, dd, q8_recip(dd)));
        const uint16_t dbits = f2h_rn(dd);
        p.hq[ob + lane] = code;
        if (lane == 0) p.hd[blockIdx.x] = dbits;
        if constexpr (DOWN) {
            s_hq[lane] = code;
            if (lane == 0) *s_hd = h2f(dbits);
        }
    }
    }  // staged
    if constexpr (DOWN) {
        // ---- split-K down projection: block b's term of every output ---------
        __syncthreads();  // h codes
        constexpr int RPW_MAX = 128;  // rows per warp: K / (8 NBL) <= 128
        const int rpw = K / NW;
        const int c0 = lane_half(lane);
        const u32x8 hv = ld_block_halves(s_hq, c0);
        const float dh = *s_hd;
#pragma unroll
        for (int i = 0; i < RPW_MAX / 32; ++i) {
            if (32 * i + lane < rpw) {
                const int row = warp * rpw + 32 * i + lane;
                const u32x8 w = ld_block_halves(s_dn + row * QK, c0);
                s_out[row] = staged ? block_term(w, hv, h2f(s_dnd[row]), dh, 0.0f) : __int_as_float(0x7fc00000);
            }
        }
        // ---- cluster reduction through distributed shared memory ---------------
        // CTA rank r sums outputs [r K / C, (r + 1) K / C) over the C CTAs of its
        // cluster (loads first, then the sum in rank order) and stores the
        // cluster's partial.
        cluster_sync();  // every CTA's terms are complete
        const int C = p.cluster;
        const int slice = K / C;
        const int r0 = static_cast<int>(cluster_ctarank()) * slice;
        float *dst = p.p_out + static_cast<int64_t>(blockIdx.x / C) * K + r0;
        for (int j = t; j < slice; j += blockDim.x) {
            float v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                if (c < C) v[c] = ld_cluster_f32(s_out + r0 + j, static_cast<uint32_t>(c));
            float sum = v[0];
#pragma unroll
            for (int c = 1; c < 8; ++c)
                if (c < C) sum += v[c];
            dst[j] = sum;
        }
        cluster_sync();  // keep this CTA's terms alive until every reader is done
    }
}

// ---------------------------------------------------------------------------
// batch-1 GEMV with the whole weight slab staged before the wait
// ---------------------------------------------------------------------------
struct PrefetchParams {
    const int8_t *w_qs;
    const uint16_t *w_d;
    const int8_t *xq;
    const uint16_t *xd;
    const float *residual;  // RESIDUAL epilogue (may equal y)
    float *y;
    int64_t n_rows;
    int k;
    int nb;
    int epi;
    int rows_per_cta;
};

// CTA c owns rows [c * rows_per_cta, ...); warp w computes rows w, w + W, ...
template <int NBL>
__global__ void __launch_bounds__(256) gemv_prefetch_kernel(const PrefetchParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int K = p.k, nb = p.nb, R = p.rows_per_cta;
    int8_t *s_w = reinterpret_cast<int8_t *>(smem);
    uint16_t *s_wd = reinterpret_cast<uint16_t *>(smem + static_cast<size_t>(R) * K);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * R;
    const int nrow = static_cast<int>(p.n_rows - r0 < R ? p.n_rows - r0 : R);

    __shared__ __align__(8) uint64_t s_bar;
    pdl_trigger();
    if (threadIdx.x == 0) mbar_init(&s_bar, 1);
    __syncthreads();
    if (warp == 0) {
        // scales on lane 0, the value slab in up to four row pieces on lanes 1-4,
        // issued in one instruction (one lane's bulk copies are serviced in turn)
        const uint32_t vbytes = static_cast<uint32_t>(nrow) * K, sbytes = static_cast<uint32_t>(nrow) * 2 * nb;
        if (lane == 0) mbar_expect_tx(&s_bar, vbytes + sbytes);
        __syncwarp();
        const int pr = (nrow + 3) / 4;  // rows per value piece
        const int v0 = (lane - 1) * pr;
        const int vr = lane == 0 ? 0 : (nrow - v0 < pr ? nrow - v0 : pr);
        if (lane == 0 || (lane <= 4 && vr > 0)) {
            void *dst = lane == 0 ? static_cast<void *>(s_wd) : static_cast<void *>(s_w + static_cast<size_t>(v0) * K);
            const void *src = lane == 0 ? static_cast<const void *>(p.w_d + r0 * nb)
                                        : static_cast<const void *>(p.w_qs + (r0 + v0) * K);
            const uint32_t bytes = lane == 0 ? sbytes : static_cast<uint32_t>(vr) * K;
            bulk_copy_g2s(dst, src, bytes, &s_bar, l2_evict_first_policy());
        }
    }

    pdl_wait();

    // The activation and, for the residual epilogue, this lane's residual
    // value are all requested before any of them is used, so their L2 round
    // trips overlap: the loads are unconditional (a block past the row's end
    // reads the last block again) and nothing converts a loaded value until the
    // last request is out.  Blocks past the end are zeroed afterwards.
    const int c0 = lane_half(lane);
    u32x8 xv[NBL];
    uint16_t xdr[NBL];
#pragma unroll
    for (int j = 0; j < NBL; ++j) {
        const int blk = min(lane + 32 * j, nb - 1);
        xv[j] = ld_block_halves(p.xq + blk * QK, c0);
        xdr[j] = p.xd[blk];
    }
    // lane l of warp w holds the residual of row w + l * nw (rows of this CTA)
    float res = 0.0f;
    if (p.epi == QG_EPI_RESIDUAL_ADD && warp + lane * nw < nrow) res = p.residual[r0 + warp + lane * nw];
    // Every thread sees the staged slab land itself (normally long ago), so the
    // weight reads below overlap the activation's L2 round trip; a warp owns its
    // rows (and their residuals), so no CTA barrier is needed.  A copy that has
    // not landed within the limit leaves NaN outputs for this warp's rows.
    if (!mbar_wait_bounded(&s_bar, 0, kCopyWaitLimitNs)) {
        count_copy_stall(lane == 0);
        for (int rr = warp; rr < nrow; rr += nw)
            if (lane == 0) p.y[r0 + rr] = __int_as_float(0x7fc00000);
        mbar_wait_bounded(&s_bar, 0, kCopyWaitLimitNs);
        return;
    }
    float xs[NBL];
#pragma unroll
    for (int j = 0; j < NBL; ++j) {
        const bool in = lane + 32 * j < nb;
        xs[j] = in ? h2f(xdr[j]) : 0.0f;
        if (!in) zero(xv[j]);
    }

    for (int rr = warp, it = 0; rr < nrow; rr += nw, ++it) {
        // a block past the end: zero codes and zero scales, so its term adds +0
        u32x8 wr[NBL];
        uint16_t wsr[NBL];
#pragma unroll
        for (int j = 0; j < NBL; ++j) {
            const int blk = min(lane + 32 * j, nb - 1);
            wr[j] = ld_block_halves(s_w + rr * K + blk * QK, c0);
            wsr[j] = s_wd[rr * nb + blk];
        }
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < NBL; ++j)
            acc = block_term(wr[j], xv[j], lane + 32 * j < nb ? h2f(wsr[j]) : 0.0f, xs[j], acc);
        acc = warp_sum(acc);
        const float rv = __shfl_sync(0xffffffffu, res, it & 31);
        if (lane == 0) {
            const int64_t row = r0 + rr;
            float rres = rv;
            if (p.epi == QG_EPI_RESIDUAL_ADD && it >= 32) rres = p.residual[row];  // more than 32 rows per warp
            p.y[row] = (p.epi == QG_EPI_RESIDUAL_ADD) ? rres + acc : acc;
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr size_t kMaxSmem = 220 * 1024;

// The staged copies move 16-byte pieces of whole rows: rows of scales must be
// a multiple of 16 bytes, i.e. k a multiple of 256.
bool ffn_up_supported(int64_t k, int64_t half)
{
    return k % 256 == 0 && k <= 2048 && half % 32 == 0 && ffn_up_smem_bytes(static_cast<int>(k)) <= kMaxSmem;
}

// One-launch layer: as above, and the down column slab must fit too; the
// residual chunks of a CTA are at most four (k <= 128 * grid).
// CTAs per cluster: the largest of 8, 4, 2, 1 that divides the grid.
static unsigned layer_cluster(int64_t half)
{
    const int64_t grid = half / 32;
    for (unsigned c : {8u, 4u, 2u})
        if (grid % c == 0) return c;
    return 1u;
}

bool decode_layer_supported(int64_t k, int64_t half)
{
    return ffn_up_supported(k, half) && ffn_up_smem_bytes(static_cast<int>(k), true) <= kMaxSmem &&
           half / 32 / layer_cluster(half) <= kMaxLayerPartials;
}

template <int NBL, bool DOWN, bool ROT = false>
static cudaError_t ffn_up_attr()
{
    return opt_in_smem(reinterpret_cast<const void *>(ffn_up_kernel<NBL, DOWN, ROT>), static_cast<int>(kMaxSmem));
}

static FfnUpParams ffn_up_params(const float *x, const float *gamma, int64_t k, float eps, const int8_t *w_qs,
                                 const uint16_t *w_d, int64_t half, float *h, int8_t *hq, uint16_t *hd)
{
    FfnUpParams p = {};
    p.x = x;
    p.gamma = gamma;
    p.w_qs = w_qs;
    p.w_d = w_d;
    p.h = h;
    p.hq = hq;
    p.hd = hd;
    p.k = static_cast<int>(k);
    p.nb = static_cast<int>(k / QK);
    p.half = half;
    p.inv_k = 1.0f / static_cast<float>(k);
    p.eps = eps;
    return p;
}

template <bool DOWN>
static cudaError_t launch_ffn_up_impl(const FfnUpParams &p, cudaStream_t s)
{
    const dim3 grid(static_cast<unsigned>(p.half / 32));
    const size_t smem = ffn_up_smem_bytes(p.k, DOWN);
    const unsigned nbl = p.k <= 1024 ? 1 : 2;
    if (nbl == 1) {
        if (cudaError_t e = ffn_up_attr<1, DOWN>(); e != cudaSuccess) return e;
    } else {
        if (cudaError_t e = ffn_up_attr<2, DOWN>(); e != cudaSuccess) return e;
    }
    if constexpr (DOWN) {
        if (nbl == 1) return launch_pdl_cluster(ffn_up_kernel<1, true>, grid, dim3(256), smem, s, p.cluster, p);
        return launch_pdl_cluster(ffn_up_kernel<2, true>, grid, dim3(512), smem, s, p.cluster, p);
    }
    if (nbl == 1) return launch_pdl(ffn_up_kernel<1, DOWN>, grid, dim3(256), smem, s, p);
    return launch_pdl(ffn_up_kernel<2, DOWN>, grid, dim3(512), smem, s, p);
}

cudaError_t launch_ffn_up(const float *x, const float *gamma, int64_t k, float eps, const int8_t *w_qs,
                          const uint16_t *w_d, int64_t half, float *h, int8_t *hq, uint16_t *hd, int8_t *xq_out,
                          uint16_t *xd_out, float *r_out, cudaStream_t s)
{
    if (half == 0) return cudaSuccess;
    FfnUpParams p = ffn_up_params(x, gamma, k, eps, w_qs, w_d, half, h, hq, hd);
    p.xq_out = xq_out;
    p.xd_out = xd_out;
    p.r_out = r_out;
    return launch_ffn_up_impl<false>(p, s);
}

// The rotated form: hidden a multiple of 128 up to 1024 (one rotation block per
// warp), otherwise as ffn_up_supported.
bool ffn_up_rotated_supported(int64_t k, int64_t half)
{
    return k % 256 == 0 && k <= 1024 && ffn_up_supported(k, half);
}

cudaError_t launch_ffn_up_rotated(const float *x, const float *gamma, int64_t k, float eps, const int8_t *w_qs,
                                  const uint16_t *w_d, int64_t half, float *h, int8_t *hq, uint16_t *hd,
                                  int8_t *xq_out, uint16_t *xd_out, cudaStream_t s)
{
    if (half == 0) return cudaSuccess;
    FfnUpParams p = ffn_up_params(x, gamma, k, eps, w_qs, w_d, half, h, hq, hd);
    p.xq_out = xq_out;
    p.xd_out = xd_out;
    if (cudaError_t e = ffn_up_attr<1, false, true>(); e != cudaSuccess) return e;
    return launch_pdl(ffn_up_kernel<1, false, true>, dim3(static_cast<unsigned>(half / 32)), dim3(256),
                      ffn_up_smem_bytes(p.k, false), s, p);
}

int decode_layer_partials(int64_t half) { return static_cast<int>(half / 32 / layer_cluster(half)); }

cudaError_t copy_stalls(uint32_t *count, bool clear)
{
    unsigned int v = 0;
    if (cudaError_t e = cudaMemcpyFromSymbol(&v, g_copy_stalls, sizeof(v)); e != cudaSuccess) return e;
    *count = v;
    if (!clear || v == 0) return cudaSuccess;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_copy_stalls, &zero, sizeof(zero));
}

cudaError_t launch_decode_layer(const float *r_in, const float *p_in, int n_in, float *r_out, float *p_out,
                                const float *gamma, int64_t k, float eps, const int8_t *wgu_qs, const uint16_t *wgu_d,
                                const int8_t *wdn_qs, const uint16_t *wdn_d, int64_t half, float *h, int8_t *hq,
                                uint16_t *hd, cudaStream_t s)
{
    FfnUpParams p = ffn_up_params(r_in, gamma, k, eps, wgu_qs, wgu_d, half, h, hq, hd);
    p.p_in = p_in;
    p.n_in = n_in;
    p.r_next = r_out;
    p.p_out = p_out;
    p.wdn_qs = wdn_qs;
    p.wdn_d = wdn_d;
    p.cluster = static_cast<int>(layer_cluster(half));
    return launch_ffn_up_impl<true>(p, s);
}

// Rows per CTA when the rows are spread over one wave of num_sms CTAs.
static int64_t prefetch_rows_per_cta(int64_t n_rows)
{
    const int64_t sms = num_sms();
    return (n_rows + sms - 1) / sms;
}

bool prefetch_supported(int64_t n_rows, int64_t k)
{
    if (k % 256 != 0 || k > 4096 || n_rows <= 0) return false;
    const int64_t rpc = prefetch_rows_per_cta(n_rows);
    return static_cast<size_t>(rpc * (k + k / 16)) <= 160 * 1024;
}

template <int NBL>
static cudaError_t prefetch_attr()
{
    return opt_in_smem(reinterpret_cast<const void *>(gemv_prefetch_kernel<NBL>), static_cast<int>(kMaxSmem));
}

template <int NBL>
static cudaError_t launch_prefetch_nbl(PrefetchParams p, cudaStream_t s)
{
    if (cudaError_t e = prefetch_attr<NBL>(); e != cudaSuccess) return e;
    const int64_t rpc = prefetch_rows_per_cta(p.n_rows);
    p.rows_per_cta = static_cast<int>(rpc);
    const dim3 grid(static_cast<unsigned>((p.n_rows + rpc - 1) / rpc));
    const dim3 block(static_cast<unsigned>(32 * (rpc < 8 ? rpc : 8)));
    const size_t smem = static_cast<size_t>(rpc) * (p.k + 2 * p.nb);
    return launch_pdl(gemv_prefetch_kernel<NBL>, grid, block, smem, s, p);
}

cudaError_t launch_gemv_prefetch(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k,
                                 const int8_t *xq, const uint16_t *xd, int epi, const float *residual, float *y,
                                 cudaStream_t s)
{
    if (n_rows == 0) return cudaSuccess;
    PrefetchParams p;
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
    p.rows_per_cta = 0;
    switch ((p.nb + 31) / 32) {
    case 1: return launch_prefetch_nbl<1>(p, s);
    case 2: return launch_prefetch_nbl<2>(p, s);
    case 3: return launch_prefetch_nbl<3>(p, s);
    case 4: return launch_prefetch_nbl<4>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

// x = r + sum of the partials, in partial order (the order the next layer's
// prologue uses), for the output of a stack of one-launch layers.
__global__ void __launch_bounds__(256) layer_finish_kernel(const float *__restrict__ r, const float *__restrict__ part,
                                                           int n, int64_t k, float *__restrict__ x)
{
    pdl_wait();
    pdl_trigger();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= k) return;
    float v = r[i];
    for (int c = 0; c < n; ++c) v += part[static_cast<int64_t>(c) * k + i];
    x[i] = v;
}

cudaError_t launch_layer_finish(const float *r, const float *part, int n, int64_t k, float *x, cudaStream_t s)
{
    if (k == 0) return cudaSuccess;
    return launch_pdl(layer_finish_kernel, dim3(static_cast<unsigned>((k + 255) / 256)), dim3(256), 0, s, r, part, n,
                      k, x);
}

}  // namespace qg
