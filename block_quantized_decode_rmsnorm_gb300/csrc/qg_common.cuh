// Device helpers shared by the kernels of libqgemv.so (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/qgemv.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libqgemv targets Blackwell (sm_103a) only"
#endif

namespace qg {

constexpr int QK = 32;  // values per Q8_0 block

// Operand tiles of the tensor-core prompt contraction: activation rows in tiles
// of 128; per tile and block one record of 4 x 2048 bytes of binary16 codes and
// 128 binary16 scales.
constexpr int ACT_TILE_ROWS = 128;
constexpr int ACT_TILE_RECORD = 8192 + 256;
__host__ __device__ inline int64_t act_tiles(int64_t rows) { return (rows + ACT_TILE_ROWS - 1) / ACT_TILE_ROWS; }

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with the programmatic
// stream serialization attribute may begin before its predecessor ends; it
// must call pdl_wait() before it reads anything the predecessor writes or
// writes anything the predecessor reads.  pdl_trigger() lets the successor
// launch early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------
struct u32x8 {
    uint32_t v[8];
};

// 32 bytes of streamed, read-only data (weights): one 256-bit load, not kept in
// L1, with a 256-byte L2 prefetch hint.  p must be 32-byte aligned.
__device__ __forceinline__ u32x8 ld_stream_32B(const void *p)
{
    u32x8 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]),
                   "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p));
    return r;
}

// L2 policy for data read once per step (weights): evict first, so that the
// small activations, gains and scales of the step stay resident in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for small data read every step (gains): keep it resident.
__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// As ld_stream_32B, with an L2 cache policy.
__device__ __forceinline__ u32x8 ld_stream_32B(const void *p, uint64_t pol)
{
    u32x8 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]),
                   "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p), "l"(pol));
    return r;
}

// 16 bytes of streamed, read-only data (weights): not kept in L1, with a
// 256-byte L2 prefetch hint.  p must be 16-byte aligned.
__device__ __forceinline__ uint4 ld_stream_16B(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16 bytes through the read-only path.  p must be 16-byte aligned.
__device__ __forceinline__ uint4 ld_nc_16B(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const uint16_t *p)
{
    uint16_t r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// 16 bytes of data written by the previous kernel (coherent path, after pdl_wait).
__device__ __forceinline__ uint4 ld_16B(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

// binary16 bits -> f32 (exact)
__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// f32 -> binary16 bits, round to nearest even
__device__ __forceinline__ uint16_t f2h_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }

// 4-way int8 dot product accumulate (dp4a)
__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c)
{
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Exact int32 -> f32 for |s| < 2^22 without the conversion pipe: place s in
// the mantissa of 1.5 * 2^23 (integer add) and subtract that constant.
__device__ __forceinline__ float small_int_to_float(int s)
{
    return __int_as_float(s + 0x4B400000) - 12582912.0f;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum NV per-lane partials across the warp in one butterfly: at offset 16 a lane
// keeps half of its values and receives the partner's other half, and so on, so
// NV values need NV - 1 + (5 - log2 NV) shuffles instead of 5 NV.  Every value
// is summed over the same lane pairs, in the same order, as warp_sum does.
// Lane l ends with the total of value index l >> (5 - log2 NV) (NV a power of
// two, at most 32).
template <int NV>
__device__ __forceinline__ float warp_sum_many(float (&v)[NV], int lane)
{
    int n = NV;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (n > 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int k = 0; k < NV / 2; ++k) {
                if (k < n / 2) {
                    const float send = upper ? v[k] : v[k + n / 2];
                    const float keep = upper ? v[k + n / 2] : v[k];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            n /= 2;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
    return v[0];
}

// max |v| over the warp with fmaxf's treatment of NaN (ignored unless every lane
// holds one), in two warp reductions instead of five shuffles: the bit patterns
// of non-negative floats order as unsigned integers.
__device__ __forceinline__ float warp_max_abs(float v)
{
    const float a = fabsf(v);
    const bool nan = a != a;
    const uint32_t m = __reduce_max_sync(0xffffffffu, nan ? 0u : __float_as_uint(a));
    const uint32_t all_nan = __reduce_and_sync(0xffffffffu, nan ? 1u : 0u);
    return all_nan ? __uint_as_float(0x7fffffffu) : __uint_as_float(m);
}

// 1/d within one ulp (the hardware reciprocal approximation; a subnormal d
// gives infinity), for q8_code.
__device__ __forceinline__ float q8_recip(float d)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// Q8_0 code of one value given the block's f32 scale d and rd = q8_recip(d):
// round half away from zero of fl(v / d) (the IEEE-rounded quotient), clamped to
// [-127, 127]; 0 when d == 0.
//
// t = fl(v * rd) lies within 2^-22 |t| of fl(v / d) (rd's error below 2^-23,
// the product's and the quotient's roundings 2^-24 each), so the two round to
// the same integer unless a half-integer lies within 2^-20 |t| of t; only then,
// or when |t| is not below 2^22 (rd infinite: d subnormal), is the IEEE quotient
// computed and rounded.  Otherwise t is rounded by adding 1.5 * 2^23, which for
// |t| < 2^22 leaves the nearest integer in the sum's mantissa (t is not a tie,
// so nearest equals half away from zero) and needs neither a float rounding
// instruction nor a conversion.  Checked against the IEEE quotient on 1.2e8
// emulated cases, half of them within a few ulp of a tie, with rd at and one ulp
// either side of 1/d.
__device__ __forceinline__ int q8_code(float v, float d, float rd)
{
    if (d == 0.0f) return 0;
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const float t = __fmul_rn(v, rd);
    const float s = __fadd_rn(t, kMagic);
    const float off = fabsf(__fsub_rn(t, __fsub_rn(s, kMagic)));  // distance to the nearest integer, exact
    const float a = fabsf(t);
    int q;
    if (!(a < 4194304.0f) || !(fabsf(off - 0.5f) > a * 0x1p-20f))
        q = static_cast<int>(roundf(__fdiv_rn(v, d)));
    else
        q = __float_as_int(s) - 0x4B400000;
    return min(max(q, -127), 127);
}

// fl(m / 127) without a division: q0 = fl(m c), c = fl(1/127), then one FMA
// correction.  Equal to the IEEE quotient for every finite non-negative f32 m
// (checked exhaustively over all 2^31 - 2^23 such values against m / 127.0f).
__device__ __forceinline__ float div127(float m)
{
    constexpr float c = 1.0f / 127.0f;
    const float q0 = __fmul_rn(m, c);
    const float r = __fmaf_rn(-q0, 127.0f, m);
    return __fmaf_rn(r, c, q0);
}

// The four codes of v as one little-endian word.
__device__ __forceinline__ uint32_t q8_pack4(float4 v, float d, float rd)
{
    return (static_cast<uint32_t>(q8_code(v.x, d, rd)) & 0xffu) |
           ((static_cast<uint32_t>(q8_code(v.y, d, rd)) & 0xffu) << 8) |
           ((static_cast<uint32_t>(q8_code(v.z, d, rd)) & 0xffu) << 16) |
           ((static_cast<uint32_t>(q8_code(v.w, d, rd)) & 0xffu) << 24);
}

// SiLU(g) * u, silu(g) = g / (1 + e^-g), branch-free over the whole range with
// one fast exponential: t = e^(-|g|/2) lies in (0, 1], so with t^2 = e^-|g|
//   g >= 0:  silu = g / (1 + t^2),     g < 0:  silu = (g t) t / (1 + t^2),
// nothing overflows, and the tiny values of the negative tail come from IEEE
// products (the fast reciprocal only ever sees 1 + t^2 in [1, 2]).  The relative
// error is a few ulp near 0 and grows with |g| (the exponential's), far inside
// the tolerance, whose scale grows with |g| as well.
__device__ __forceinline__ float silu_mul(float g, float u)
{
    const float t = __expf(-0.5f * fabsf(g));
    const float num = g >= 0.0f ? g : (g * t) * t;
    return num * __fdividef(1.0f, __fmaf_rn(t, t, 1.0f)) * u;
}

// 16-byte asynchronous global -> shared copy (LDGSTS); src and dst 16-byte aligned.
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void *src, uint64_t pol)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// Bulk (TMA) copies global -> shared with mbarrier completion
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// One bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2; selp.u32 %0, 1, 0, q; }"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: while the phase is incomplete the thread
// sleeps in the barrier unit (until the phase completes or hint_ns pass)
// instead of spinning and taking issue slots from other warps on the SM.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2, %3; selp.u32 %0, 1, 0, q; }"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity`; false if it has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// The same with the thread asleep in the barrier unit between checks, for
// waits that may be long and overlap other kernels' work on the SM.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    constexpr uint32_t kHintNs = 1000000u;
    if (mbar_try_wait_sleep(bar, parity, kHintNs)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity, kHintNs))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// Limit for a wait on copies that were issued long before: one second.
constexpr uint64_t kCopyWaitLimitNs = 1000000000ull;

}  // namespace qg

// ---------------------------------------------------------------------------
// Host-side launch helpers (defined in qg_api.cu)
// ---------------------------------------------------------------------------
namespace qg {
int num_sms();
// Opt `func` in to `bytes` of dynamic shared memory on the current device.  The
// opt-in is an attribute of the kernel in each device's context, so it is made
// once per (device, kernel), and again only when a larger size is asked for.
cudaError_t opt_in_smem(const void *func, int bytes);
// Launch with programmatic stream serialization enabled.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launch with programmatic stream serialization and thread-block clusters of
// `cluster` CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               unsigned cluster, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- thread-block cluster helpers --------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster must call it (a hardware barrier:
// the CTAs of a cluster are resident together).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// f32 at the same shared-memory offset as `local`, in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const float *local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}
}  // namespace qg
