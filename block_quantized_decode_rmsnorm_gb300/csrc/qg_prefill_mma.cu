// Prompt-sized block-scaled Q8_0 contraction on the int8 tensor path (mma.sync).
//
// "Filling in the blanks: Inference using Phobos", Fast Decode: a 512-token
// prompt reuses every weight 512 times and wants the tensor cores; GPU
// Performance Heisenbugs: exact int8 values run straight on the integer tensor
// cores.
//
// Y[m][n] = sum_j f32(d_x[m][j]) * f32(d_w[n][j]) * S_j[m][n].  One
// m16n8k32 s8 MMA covers exactly one 32-value block, so its int32 result is the
// exact block sum S_j for a 16x8 tile; the block's scales are applied in
// registers right after each MMA.  CTA tile 128 (M) x 64 (N), eight warps of
// 32 x 32, cp.async multi-stage staging of the int8 tiles (16-byte chunks,
// XOR-swizzled so ldmatrix reads are conflict-free), all scales of the CTA's
// rows staged once as f32.

#include "qg_common.cuh"

namespace qg {

constexpr int PF_BM = 128;
constexpr int PF_BN = 64;
constexpr int PF_THREADS = 256;
constexpr int PF_STAGES = 4;
constexpr int PF_MAX_NB = 256;  // K <= 8192

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return smem_addr(p); }

// 16-byte async copy that zero-fills instead of reading when !valid (rows past the end).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8_16x8x32(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

// Byte offset of 16-byte chunk c (0 or 1) of tile row r: rows are 32 bytes,
// chunk index XOR-swizzled by bit 2 of the row.
__device__ __forceinline__ uint32_t tile_off(int r, int c) { return r * 32 + ((c ^ ((r >> 2) & 1)) << 4); }

struct PrefillParams {
    const int8_t *w_qs;
    const uint16_t *w_d;
    const int8_t *xq;
    const uint16_t *xd;
    float *y;
    int64_t m;
    int64_t n;
    int k;
    int nb;
};

__global__ void __launch_bounds__(PF_THREADS) prefill_mma_kernel(const PrefillParams p)
{
    extern __shared__ __align__(128) uint8_t sm[];
    uint8_t *tA = sm;                                   // [STAGES][BM][32]
    uint8_t *tB = tA + PF_STAGES * PF_BM * 32;          // [STAGES][BN][32]
    const int ss = p.nb + 1;  // padded row stride of the scale tables (bank spread)
    float *sx = reinterpret_cast<float *>(tB + PF_STAGES * PF_BN * 32);  // [BM][ss]
    float *sw = sx + PF_BM * ss;                        // [BN][ss]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int wm = warp & 3;  // warp row (32 rows each)
    const int wn = warp >> 2; // warp col (32 cols each)
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * PF_BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * PF_BN;

    // Weights (and their scales) are not produced by the preceding kernel.
    for (int i = tid; i < PF_BN * p.nb; i += PF_THREADS) {
        const int r = i / p.nb, j = i % p.nb;
        const int64_t n = n0 + r;
        sw[r * ss + j] = (n < p.n) ? h2f(p.w_d[n * p.nb + j]) : 0.0f;
    }
    auto load_B = [&](int stage, int blk) {
        // BN rows x 2 chunks = 128 chunks
        if (tid < PF_BN * 2) {
            const int r = tid >> 1, c = tid & 1;
            const int64_t n = n0 + r;
            const bool ok = n < p.n;
            const int8_t *src = p.w_qs + (ok ? n : 0) * p.k + blk * QK + c * 16;
            cp_async_16(smem_u32(tB + stage * PF_BN * 32 + tile_off(r, c)), src, ok);
        }
    };
    auto load_A = [&](int stage, int blk) {
        // BM rows x 2 chunks = 256 chunks, one per thread
        const int r = tid >> 1, c = tid & 1;
        const int64_t m = m0 + r;
        const bool ok = m < p.m;
        const int8_t *src = p.xq + (ok ? m : 0) * p.k + blk * QK + c * 16;
        cp_async_16(smem_u32(tA + stage * PF_BM * 32 + tile_off(r, c)), src, ok);
    };

    // Prologue: the weight tiles of the first stages, then wait for the
    // activation producer.
#pragma unroll
    for (int s = 0; s < PF_STAGES - 1; ++s)
        if (s < p.nb) load_B(s, s);
    pdl_trigger();
    pdl_wait();
    for (int i = tid; i < PF_BM * p.nb; i += PF_THREADS) {
        const int r = i / p.nb, j = i % p.nb;
        const int64_t m = m0 + r;
        sx[r * ss + j] = (m < p.m) ? h2f(p.xd[m * p.nb + j]) : 0.0f;
    }
#pragma unroll
    for (int s = 0; s < PF_STAGES - 1; ++s) {
        if (s < p.nb) load_A(s, s);
        cp_async_commit();
    }

    float acc[2][4][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.0f;

    const int g = lane >> 2;   // group id
    const int tg = lane & 3;   // thread in group
    // ldmatrix row/chunk each lane supplies
    const int lrow = lane & 7;
    const int lsel = lane >> 3;  // which of the 4 matrices

    for (int blk = 0; blk < p.nb; ++blk) {
        cp_async_wait<PF_STAGES - 2>();
        __syncthreads();
        {  // issue the stage STAGES-1 ahead
            const int nxt = blk + PF_STAGES - 1;
            if (nxt < p.nb) {
                load_B(nxt % PF_STAGES, nxt);
                load_A(nxt % PF_STAGES, nxt);
            }
            cp_async_commit();
        }
        const int st = blk % PF_STAGES;
        const uint8_t *A = tA + st * PF_BM * 32;
        const uint8_t *B = tB + st * PF_BN * 32;

        uint32_t af[2][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            // matrices: [rows 0-7, chunk 0], [rows 8-15, chunk 0], [rows 0-7, chunk 1], [rows 8-15, chunk 1]
            const int r = wm * 32 + mi * 16 + lrow + ((lsel & 1) << 3);
            const int c = lsel >> 1;
            ldmatrix_x4(smem_u32(A + tile_off(r, c)), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
        }
        uint32_t bf[4][2];
#pragma unroll
        for (int nj = 0; nj < 2; ++nj) {
            // matrices: [n 0-7, chunk 0], [n 0-7, chunk 1], [n 8-15, chunk 0], [n 8-15, chunk 1]
            const int r = wn * 32 + nj * 16 + lrow + ((lsel >> 1) << 3);
            const int c = lsel & 1;
            ldmatrix_x4(smem_u32(B + tile_off(r, c)), bf[2 * nj][0], bf[2 * nj][1], bf[2 * nj + 1][0],
                        bf[2 * nj + 1][1]);
        }
        // block scales for this thread's rows / columns
        float dxr[2][2], dwc[4][2];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            dxr[mi][0] = sx[(wm * 32 + mi * 16 + g) * ss + blk];
            dxr[mi][1] = sx[(wm * 32 + mi * 16 + g + 8) * ss + blk];
        }
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            dwc[ni][0] = sw[(wn * 32 + ni * 8 + 2 * tg) * ss + blk];
            dwc[ni][1] = sw[(wn * 32 + ni * 8 + 2 * tg + 1) * ss + blk];
        }
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                int s4[4];
                mma_s8_16x8x32(s4, af[mi], bf[ni][0], bf[ni][1]);
                acc[mi][ni][0] = fmaf(dxr[mi][0] * dwc[ni][0], small_int_to_float(s4[0]), acc[mi][ni][0]);
                acc[mi][ni][1] = fmaf(dxr[mi][0] * dwc[ni][1], small_int_to_float(s4[1]), acc[mi][ni][1]);
                acc[mi][ni][2] = fmaf(dxr[mi][1] * dwc[ni][0], small_int_to_float(s4[2]), acc[mi][ni][2]);
                acc[mi][ni][3] = fmaf(dxr[mi][1] * dwc[ni][1], small_int_to_float(s4[3]), acc[mi][ni][3]);
            }
    }
    cp_async_wait<0>();

    // store: c0,c1 at (row g, cols 2tg, 2tg+1); c2,c3 at row g+8
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int64_t m = m0 + wm * 32 + mi * 16 + g + half * 8;
            if (m >= p.m) continue;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int64_t n = n0 + wn * 32 + ni * 8 + 2 * tg;
                float *dst = p.y + m * p.n + n;
                const float v0 = acc[mi][ni][2 * half];
                const float v1 = acc[mi][ni][2 * half + 1];
                if (n + 1 < p.n && ((reinterpret_cast<uintptr_t>(dst) & 7) == 0)) {
                    *reinterpret_cast<float2 *>(dst) = make_float2(v0, v1);
                } else {
                    if (n < p.n) dst[0] = v0;
                    if (n + 1 < p.n) dst[1] = v1;
                }
            }
        }
}

cudaError_t launch_prefill_mma(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k, const int8_t *xq,
                               const uint16_t *xd, int64_t m, float *y, cudaStream_t s)
{
    if (m == 0 || n_rows == 0) return cudaSuccess;
    PrefillParams p;
    p.w_qs = w_qs;
    p.w_d = w_d;
    p.xq = xq;
    p.xd = xd;
    p.y = y;
    p.m = m;
    p.n = n_rows;
    p.k = static_cast<int>(k);
    p.nb = static_cast<int>(k / QK);
    if (p.nb > PF_MAX_NB) return cudaErrorInvalidValue;
    const size_t smem =
        PF_STAGES * (PF_BM + PF_BN) * 32 + static_cast<size_t>(PF_BM + PF_BN) * (p.nb + 1) * sizeof(float);
    if (cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(prefill_mma_kernel),
                                    static_cast<int>(PF_STAGES * (PF_BM + PF_BN) * 32 +
                                                     (PF_BM + PF_BN) * (PF_MAX_NB + 1) * sizeof(float)));
        e != cudaSuccess)
        return e;
    const dim3 grid(static_cast<unsigned>((n_rows + PF_BN - 1) / PF_BN), static_cast<unsigned>((m + PF_BM - 1) / PF_BM));
    return launch_pdl(prefill_mma_kernel, grid, dim3(PF_THREADS), smem, s, p);
}

// ---------------------------------------------------------------------------
// rate of the int8 mma.sync path, for the prompt contraction's second roofline
// ---------------------------------------------------------------------------
// Every warp runs `iters` rounds of eight independent m16n8k32 s8 MMAs (2 * 16 *
// 8 * 32 int-ops each) on register operands; nothing is loaded, so the time is
// the tensor pipe's.  The sums reach memory only through an impossible-looking
// test, which keeps the compiler from dropping the MMAs.
constexpr int MR_THREADS = 256;
__global__ void __launch_bounds__(MR_THREADS) mma_s8_rate_kernel(int iters, int *sink)
{
    uint32_t a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 0x01010101u * static_cast<uint32_t>((threadIdx.x + i) & 7);
    const uint32_t b0 = 0x01020304u ^ threadIdx.x, b1 = 0x05060708u ^ blockIdx.x;
    int c[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[j][i] = 0;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                         "{%0,%1,%2,%3};"
                         : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                         : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
        }
    }
    int t = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) t += c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
    if (t == 0x7fffffff) *sink = t;
}

cudaError_t launch_mma_s8_rate(int64_t iters, int *sink, int64_t *ops, cudaStream_t s)
{
    const int64_t grid = static_cast<int64_t>(num_sms()) * 4;
    *ops = grid * (MR_THREADS / 32) * iters * 8 * (2LL * 16 * 8 * 32);
    mma_s8_rate_kernel<<<static_cast<unsigned>(grid), MR_THREADS, 0, s>>>(static_cast<int>(iters), sink);
    return cudaGetLastError();
}

}  // namespace qg
