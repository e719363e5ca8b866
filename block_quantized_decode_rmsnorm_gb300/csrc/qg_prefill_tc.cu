// Prompt-sized block-scaled Q8_0 contraction on the 5th-generation tensor cores.
//
// "Filling in the blanks: Inference using Phobos", Fast Decode: prompt
// processing reuses every weight once per prompt row and belongs on the tensor
// cores; GPU Performance Heisenbugs: exact int8 values run straight on the
// integer tensor cores.
//
// GB300 has no integer tcgen05 kind on sm_103a, so the int8 codes run as f16
// values: every code is an integer in [-127, 127], exact in f16, and every
// partial sum of one 32-value block is an integer below 2^24, exact in the f32
// accumulator.  So the tensor core produces the exact block sums S_j and the
// block scales are applied afterwards:
//
//   Y[m][n] = sum_j f32(d_x[m][j]) * f32(d_w[n][j]) * S_j[m][n].
//
// Persistent kernel, one CTA per SM, output tiles of 128 (M) x BN (N) taken in
// turn; K is walked one 32-value block at a time and the block counter runs on
// across tiles, so the operand pipeline never drains between tiles.  Tiles are
// numbered M-fastest and each tile starts its K walk at a different multiple of
// eight blocks, so the SMs working at one time read many different activation
// records instead of all pulling the same lines out of L2.  Roles:
//   * warp 13 - copies, spread over lanes.  Per block: the activation record
//     (codes already f16 in the MMA's core-matrix order, written that way by
//     quantize_act_q8_0_tiles) as one 8 KB bulk copy, and the record's 128
//     row scales into the scale ring.  Per group of eight blocks: the weight
//     codes (two 2D TMA boxes of BN rows x 128 bytes, 128-byte swizzled) and
//     the weight scales (one box of BN rows x 8 binary16).
//   * warps 8-11 - convert the weight codes of each block (int8 -> f16, exact:
//     a byte permute against 0x64 and one f16x2 subtraction per two values)
//     into the no-swizzle K-major operand layout, and the block's weight
//     scales to f32 in the scale ring.
//   * warp 12, lane 0 - issues two tcgen05.mma kind::f16 (M=128, N=BN, K=16)
//     per block into one of four TMEM accumulators.
//   * warps 0-7 - epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (tile
//     rows) and columns (w / 4) BN/2 .. +BN/2, and accumulates
//     acc += (d_x d_w) S_j in registers with packed f32x2 multiply and FMA
//     (the same roundings as the scalar forms).
// Stages are tracked with mbarriers, arrived on once per warp (after
// __syncwarp) rather than once per thread: arrivals on one barrier serialise in
// shared memory.  Every wait is bounded by the global timer
// and a stalled pipeline aborts (NaN outputs for the tiles left) instead of
// hanging.
#include <cuda.h>

#include "qg_common.cuh"
#include "qg_tc.cuh"

namespace qg {

constexpr int TC_BM = ACT_TILE_ROWS;  // 128
constexpr int TC_GROUP = 8;           // K blocks per weight copy (256 codes of each row)
constexpr int TC_XB = 4;              // K blocks per activation copy (four whole records)
constexpr int TC_W_SLOTS = 3;         // converted-weight ring, batches
constexpr int TC_EPI_WARPS = 16;
constexpr int TC_CONV_WARPS = 4;
constexpr int TC_CONV_WARP0 = TC_EPI_WARPS;                 // 16
constexpr int TC_MMA_WARP = TC_CONV_WARP0 + TC_CONV_WARPS;  // 20
constexpr int TC_XCOPY_WARP0 = TC_MMA_WARP + 1;             // 21, 22
constexpr int TC_WCOPY_WARP = TC_XCOPY_WARP0 + 2;           // 23
constexpr int TC_THREADS = (TC_WCOPY_WARP + 1) * 32;        // 768

struct PrefillTcParams {
    const uint8_t *xt;  // activation records
    float *y;
    int64_t m;
    int64_t n;
    int nb;
    int64_t m_tiles;  // along M
    int64_t tiles;    // total; tile t covers rows 128 (t % m_tiles), columns BN (t / m_tiles)
};

// Shared-memory layout of one CTA (byte offsets from a 1024-byte aligned base).
// K blocks are handled in batches of B: every barrier wait, arrival, commit and
// proxy fence is paid once per batch, not once per block.
template <int BN>
struct TcLayout {
    static constexpr int B = BN == 64 ? 4 : 2;             // K blocks per batch
    static constexpr int TMEM_BATCH = B * BN;              // columns of one batch's block sums
    static constexpr int TMEM_COLS = 512;                  // two batches
    static constexpr int XS = 3;                           // activation stages of TC_XB records
    static constexpr int XSTAGE = TC_XB * ACT_TILE_RECORD; // 33792, a multiple of 1024
    static constexpr int W16 = BN * 64;                    // one block: BN rows x 32 f16, operand layout
    static constexpr int WSLOT = B * W16 + B * BN * 4;     // a batch of blocks, then f32 d_w[B][BN]
    static constexpr int WSLOT_AL = (WSLOT + 1023) / 1024 * 1024;
    static constexpr int W8_HALF = BN * 128;               // one swizzled box: BN rows x 4 blocks of codes
    static constexpr int W8 = 2 * W8_HALF;                 // one group of eight blocks
    static constexpr int DS = BN * 16;                     // [BN][8] binary16 weight scales of one group
    static constexpr int OFF_W16 = XS * XSTAGE;
    static constexpr int OFF_W8 = OFF_W16 + TC_W_SLOTS * WSLOT_AL;
    static constexpr int OFF_DS = OFF_W8 + 2 * W8;
    // BN = 64 only (the others leave no room): per epilogue warp a padded 32 x 17
    // f32 block through which its tile rows are turned into row-contiguous stores
    static constexpr bool XPOSE = BN == 64;
    static constexpr int OFF_XP = OFF_DS + 2 * DS;
    static constexpr int BYTES = OFF_XP + (XPOSE ? TC_EPI_WARPS * 32 * (BN / 4 + 1) * 4 : 0);
    static constexpr int CW = BN / 4;                      // columns per epilogue warp
    static_assert(BN % 32 == 0 && BN <= 128, "BN: a multiple of 32, at most 128");
    static_assert(2 * TMEM_BATCH <= TMEM_COLS, "two batches of block sums in TMEM");
    static_assert(TC_GROUP % B == 0 && TC_XB % B == 0, "batches never straddle copies");
    static_assert(XSTAGE % 1024 == 0 && W16 % 1024 == 0 && W8_HALF % 1024 == 0,
                  "swizzled boxes need 1024-byte alignment");
    static_assert(BYTES + 1024 <= 227 * 1024, "shared memory");
};

template <int BN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmd,
                      const PrefillTcParams p)
{
    using L = TcLayout<BN>;
    constexpr int CW = L::CW;
    constexpr int B = L::B;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t x_full[L::XS], x_empty[L::XS];
    __shared__ __align__(8) uint64_t w16_full[TC_W_SLOTS], w16_empty[TC_W_SLOTS];
    __shared__ __align__(8) uint64_t w8_full[2], w8_empty[2];
    __shared__ __align__(8) uint64_t tfull[2], tempty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int lane = t & 31;
    const int nb = p.nb;
    const int nbatch = nb / B;  // batches per tile

    if (t == 0) {
        abort_flag = 0;
        for (int i = 0; i < L::XS; ++i) {
            mbar_init(&x_full[i], 1);                 // the copy lane's expect_tx
            mbar_init(&x_empty[i], 1 + TC_EPI_WARPS); // MMA commit + every epilogue warp (it reads d_x there)
        }
        for (int i = 0; i < TC_W_SLOTS; ++i) {
            mbar_init(&w16_full[i], TC_CONV_WARPS);        // one arrival per converter warp
            mbar_init(&w16_empty[i], 1 + TC_EPI_WARPS);    // MMA commit + epilogue (it reads d_w there)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&w8_full[i], 1);
            mbar_init(&w8_empty[i], TC_CONV_WARPS);
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], TC_EPI_WARPS);
        }
    }
    if (warp == TC_MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                     "r"(L::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    pdl_wait();  // the activation records come from the previous kernel
    const uint32_t tmem = tmem_base;

    if (warp == TC_XCOPY_WARP0 || warp == TC_XCOPY_WARP0 + 1) {
        // ---------------- activation copies --------------------------------------
        // A warp's bulk copies are serviced one after another, so two warps take
        // alternate stages; each copy moves four whole records (codes and scales).
        if (lane == 0) {
            const uint32_t xw = warp - TC_XCOPY_WARP0;
            uint32_t xc = 0;  // activation stage counter
            int64_t last = -1;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
                const int64_t mt = tile % p.m_tiles, nt = tile / p.m_tiles;
                const uint8_t *rec = p.xt + mt * nb * static_cast<int64_t>(ACT_TILE_RECORD);
                const int rot = TC_GROUP * static_cast<int>(nt % (nb / TC_GROUP));
                for (int bi = 0; bi < nb; bi += TC_XB, ++xc) {
                    if ((xc & 1) != xw) continue;
                    const int blk = bi + rot < nb ? bi + rot : bi + rot - nb;
                    const uint32_t slot = xc % L::XS, use = xc / L::XS;
                    if (!(ok = tc_wait(&x_empty[slot], (use & 1) ^ 1, &abort_flag))) break;
                    mbar_expect_tx(&x_full[slot], L::XSTAGE);
                    bulk_load(smem + slot * L::XSTAGE, rec + blk * ACT_TILE_RECORD, L::XSTAGE, &x_full[slot]);
                    last = xc;
                }
            }
            // After an abort the last copy may still be landing: let it finish
            // (bounded) before the CTA's shared memory goes away.
            if (!ok && last >= 0) mbar_wait_bounded(&x_full[last % L::XS], (last / L::XS) & 1, kCopyWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == TC_WCOPY_WARP) {
        // ---------------- weight copies: lanes 0-2 issue one group's three boxes in
        // one instruction (codes half 0, codes half 1, scales) ---------------------
        if (lane < 3) {
            uint32_t g = 0;
            int64_t last = -1;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
                const int64_t nt = tile / p.m_tiles;
                const int n0 = static_cast<int>(nt * BN);
                const int rot = TC_GROUP * static_cast<int>(nt % (nb / TC_GROUP));
                for (int bi = 0; bi < nb; bi += TC_GROUP, ++g) {
                    const int blk = bi + rot < nb ? bi + rot : bi + rot - nb;
                    const uint32_t gs = g & 1, use = g >> 1;
                    bool mine = true;
                    if (lane == 0) mine = tc_wait(&w8_empty[gs], (use & 1) ^ 1, &abort_flag);
                    ok = __shfl_sync(0x7u, mine, 0);
                    if (!ok) break;
                    if (lane == 0) mbar_expect_tx(&w8_full[gs], L::W8 + L::DS);
                    __syncwarp(0x7u);
                    uint8_t *dst = lane < 2 ? smem + L::OFF_W8 + gs * L::W8 + lane * L::W8_HALF
                                            : smem + L::OFF_DS + gs * L::DS;
                    const CUtensorMap *map = lane < 2 ? &tmw : &tmd;
                    const int c0 = lane < 2 ? blk * QK + lane * 128 : blk;
                    tma_load_2d(dst, map, c0, n0, &w8_full[gs]);
                    last = g;
                }
            }
            if (!ok && last >= 0 && lane == 0)
                mbar_wait_bounded(&w8_full[last & 1], (last >> 1) & 1, kCopyWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= TC_CONV_WARP0 && warp < TC_MMA_WARP) {
        // ---------------- weight codes int8 -> f16 operand layout, weight scales --
        const int pt = t - TC_CONV_WARP0 * 32;  // 0..127
        uint32_t kb = 0;                         // batch counter
        bool ok = true;
        for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
            for (int bt = 0; bt < nbatch; ++bt, ++kb) {
                const int bsub0 = (bt * B) % TC_GROUP;  // first block of the batch within its group
                const uint32_t g = kb * B / TC_GROUP, gs = g & 1;
                if (bsub0 == 0 && !(ok = tc_wait(&w8_full[gs], (g >> 1) & 1, &abort_flag))) break;
                const uint32_t ws_i = kb % TC_W_SLOTS, wuse = kb / TC_W_SLOTS;
                if (!(ok = tc_wait(&w16_empty[ws_i], (wuse & 1) ^ 1, &abort_flag))) break;
                uint8_t *wslot = smem + L::OFF_W16 + ws_i * L::WSLOT_AL;
                const uint8_t *w8g = smem + L::OFF_W8 + gs * L::W8;
#pragma unroll
                for (int c0 = 0; c0 < 2 * BN * B; c0 += 128) {
                    const int c = c0 + pt;  // chunk: block i, half h, row r
                    if (c < 2 * BN * B) {
                        const int i = c / (2 * BN);
                        const int rem = c - i * 2 * BN;
                        const int h = rem >= BN ? 1 : 0;
                        const int r = rem - h * BN;
                        const int bsub = bsub0 + i;
                        // 16-byte chunk (bsub % 4) * 2 + h of row r, 128-byte swizzle: chunk ^ (r % 8)
                        const int chunk = ((bsub & 3) * 2 + h) ^ (r & 7);
                        const uint4 v =
                            *reinterpret_cast<const uint4 *>(w8g + (bsub >> 2) * L::W8_HALF + r * 128 + chunk * 16);
                        uint32_t f[8];
                        s8x4_to_f16x4(v.x, f[0], f[1]);
                        s8x4_to_f16x4(v.y, f[2], f[3]);
                        s8x4_to_f16x4(v.z, f[4], f[5]);
                        s8x4_to_f16x4(v.w, f[6], f[7]);
                        // K groups 2h and 2h+1 of row r: (r / 8) 128 + group (BN 16) + (r % 8) 16
                        uint8_t *d0 = wslot + i * L::W16 + (r >> 3) * 128 + (2 * h) * (BN * 16) + (r & 7) * 16;
                        *reinterpret_cast<uint4 *>(d0) = make_uint4(f[0], f[1], f[2], f[3]);
                        *reinterpret_cast<uint4 *>(d0 + BN * 16) = make_uint4(f[4], f[5], f[6], f[7]);
                    }
                }
                // f32 weight scales of the batch, [B][BN]
                const uint16_t *ds = reinterpret_cast<const uint16_t *>(smem + L::OFF_DS + gs * L::DS);
                float *dwf = reinterpret_cast<float *>(wslot + B * L::W16);
                for (int e = pt; e < B * BN; e += 128) {
                    const int i = e / BN, r = e - i * BN;
                    dwf[e] = h2f(ds[r * TC_GROUP + bsub0 + i]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&w16_full[ws_i]);
                    if (bsub0 + B == TC_GROUP) mbar_arrive(&w8_empty[gs]);
                }
            }
        }
    } else if (warp == TC_MMA_WARP) {
        // ---------------- MMA issuer -------------------------------------------
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(TC_BM >> 4) << 24);
            uint32_t kb = 0;
            int64_t last = -1;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
                for (int bt = 0; bt < nbatch; ++bt, ++kb) {
                    const uint32_t gb0 = kb * B;  // first block of the batch (global count)
                    const uint32_t xc = gb0 / TC_XB, xi0 = gb0 % TC_XB;
                    const uint32_t xs = xc % L::XS, xuse = xc / L::XS;
                    const uint32_t ws_i = kb % TC_W_SLOTS, wuse = kb / TC_W_SLOTS;
                    const uint32_t buf = kb & 1, tuse = kb >> 1;
                    if (xi0 == 0 && !(ok = tc_wait(&x_full[xs], xuse & 1, &abort_flag))) break;
                    if (!(ok = tc_wait(&w16_full[ws_i], wuse & 1, &abort_flag))) break;
                    if (!(ok = tc_wait(&tempty[buf], (tuse & 1) ^ 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint32_t wbase = smem_addr(smem + L::OFF_W16 + ws_i * L::WSLOT_AL);
#pragma unroll
                    for (int i = 0; i < B; ++i) {
                        const uint32_t xa = smem_addr(smem + xs * L::XSTAGE + (xi0 + i) * ACT_TILE_RECORD);
                        const uint32_t wa = wbase + i * L::W16;
                        const uint32_t d = tmem + buf * L::TMEM_BATCH + i * BN;
                        umma_f16(d, umma_desc(xa, 2048, 128), umma_desc(wa, BN * 16, 128), idesc, 0u);
                        umma_f16(d, umma_desc(xa + 2 * 2048, 2048, 128), umma_desc(wa + 2 * BN * 16, BN * 16, 128),
                                 idesc, 1u);
                    }
                    umma_commit(&tfull[buf]);
                    umma_commit(&w16_empty[ws_i]);
                    if (xi0 + B == TC_XB) umma_commit(&x_empty[xs]);
                    last = kb;
                }
            }
            // After an abort, wait (bounded) for the last issued MMAs before TMEM is freed.
            if (!ok && last >= 0) mbar_wait_bounded(&tfull[last & 1], (last >> 1) & 1, kCopyWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 0-15 ------------------------------------
        // warp w: TMEM lanes (tile rows) 32 (w % 4) .. +31, columns CW (w / 4) .. +CW
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int col0 = (warp >> 2) * CW;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint32_t kb = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
            const int64_t mt = tile % p.m_tiles;
            const int64_t n0 = tile / p.m_tiles * BN;
            uint64_t acc[CW / 2];
#pragma unroll
            for (int i = 0; i < CW / 2; ++i) acc[i] = 0;
            for (int bt = 0; ok && bt < nbatch; ++bt, ++kb) {
                const uint32_t gb0 = kb * B;
                const uint32_t xc = gb0 / TC_XB, xi0 = gb0 % TC_XB;
                const uint32_t xs = xc % L::XS, xuse = xc / L::XS;
                const uint32_t ws_i = kb % TC_W_SLOTS, wuse = kb / TC_W_SLOTS;
                const uint32_t buf = kb & 1, tuse = kb >> 1;
                // tcgen05.ld is warp-collective: the whole warp proceeds or stops
                ok = __all_sync(0xffffffffu, tc_wait(&tfull[buf], tuse & 1, &abort_flag) &&
                                                 tc_wait(&x_full[xs], xuse & 1, &abort_flag) &&
                                                 tc_wait(&w16_full[ws_i], wuse & 1, &abort_flag));
                if (!ok) break;
                tc_fence_after();
                const uint8_t *xrec = smem + xs * L::XSTAGE + xi0 * ACT_TILE_RECORD + 8192 + row * 2;
                const float *dwb = reinterpret_cast<const float *>(smem + L::OFF_W16 + ws_i * L::WSLOT_AL + B * L::W16);
#pragma unroll
                for (int i = 0; i < B; ++i) {
                    uint32_t sv[CW];
                    const uint32_t ta = tmem + lane_addr + buf * L::TMEM_BATCH + i * BN + col0;
#pragma unroll
                    for (int c = 0; c + 16 <= CW; c += 16) tmem_ld_16(ta + c, sv + c);
                    if constexpr (CW % 16 != 0) tmem_ld_8(ta + (CW / 16) * 16, sv + (CW / 16) * 16);
                    const float dx = h2f(*reinterpret_cast<const uint16_t *>(xrec + i * ACT_TILE_RECORD));
                    const uint64_t dx2 = pack2(dx, dx);
                    const float4 *dw4 = reinterpret_cast<const float4 *>(dwb + i * BN + col0);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < CW / 4; ++j) {
                        const float4 w = dw4[j];
                        const uint64_t c01 = mul2(dx2, pack2(w.x, w.y));
                        const uint64_t c23 = mul2(dx2, pack2(w.z, w.w));
                        acc[2 * j] = fma2(c01, pack2u(sv[4 * j], sv[4 * j + 1]), acc[2 * j]);
                        acc[2 * j + 1] = fma2(c23, pack2u(sv[4 * j + 2], sv[4 * j + 3]), acc[2 * j + 1]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&tempty[buf]);
                    mbar_arrive(&w16_empty[ws_i]);
                    if (xi0 + B == TC_XB) mbar_arrive(&x_empty[xs]);
                }
            }
            if (!ok) {
#pragma unroll
                for (int i = 0; i < CW / 2; ++i) acc[i] = pack2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
            }
            if constexpr (L::XPOSE) {
                // lane l holds row l of the warp's 32 x 16 block: through shared
                // memory, then each store writes 16 columns of two rows (64 bytes each)
                float *xp = reinterpret_cast<float *>(smem + L::OFF_XP) + warp * 32 * (CW + 1);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < CW / 2; ++i) {
                    const float2 a = unpack2(acc[i]);
                    xp[lane * (CW + 1) + 2 * i] = a.x;
                    xp[lane * (CW + 1) + 2 * i + 1] = a.y;
                }
                __syncwarp();
                const int hr = lane >> 4, col = lane & 15;
                const bool col_ok = n0 + col0 + col < p.n;
#pragma unroll 4
                for (int r2 = 0; r2 < 32; r2 += 2) {
                    const int64_t mr = mt * TC_BM + q * 32 + r2 + hr;
                    const float v = xp[(r2 + hr) * (CW + 1) + col];
                    if (mr < p.m && col_ok) p.y[mr * p.n + n0 + col0 + col] = v;
                }
                __syncwarp();  // the block is reused by the next tile
                continue;
            }
            const int64_t m = mt * TC_BM + row;
            if (m < p.m) {
                float *dst = p.y + m * p.n + n0 + col0;
                const bool full = (n0 + col0 + CW <= p.n) && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0);
                if (full) {
#pragma unroll
                    for (int i = 0; i < CW / 2; i += 2) {
                        const float2 a = unpack2(acc[i]), c = unpack2(acc[i + 1]);
                        *reinterpret_cast<float4 *>(dst + 2 * i) = make_float4(a.x, a.y, c.x, c.y);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < CW / 2; ++i) {
                        const float2 a = unpack2(acc[i]);
                        if (n0 + col0 + 2 * i < p.n) dst[2 * i] = a.x;
                        if (n0 + col0 + 2 * i + 1 < p.n) dst[2 * i + 1] = a.y;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == TC_MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Weight codes and scales are fetched eight blocks (256 codes of a row) at a
// time, so K must be a multiple of 256.
bool prefill_tc_supported(int64_t k) { return k > 0 && k % (QK * TC_GROUP) == 0; }

template <int BN>
static cudaError_t launch_prefill_tc_bn(EncodeTiledFn enc, const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows,
                                       int64_t k, const void *xt, int64_t m, float *y, cudaStream_t s)
{
    using L = TcLayout<BN>;
    const int64_t nb = k / QK;
    const cuuint32_t estride[2] = {1, 1};
    CUtensorMap wmap, dmap;
    const cuuint64_t wdim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(n_rows)};
    const cuuint64_t wstride[1] = {static_cast<cuuint64_t>(k)};
    const cuuint32_t wbox[2] = {128, BN};
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(w_qs), wdim, wstride, wbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const cuuint64_t ddim[2] = {static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(n_rows)};
    const cuuint64_t dstride[1] = {static_cast<cuuint64_t>(nb) * 2};
    const cuuint32_t dbox[2] = {TC_GROUP, BN};
    if (enc(&dmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(w_d), ddim, dstride, dbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    PrefillTcParams p;
    p.xt = static_cast<const uint8_t *>(xt);
    p.y = y;
    p.m = m;
    p.n = n_rows;
    p.nb = static_cast<int>(nb);
    p.m_tiles = act_tiles(m);
    p.tiles = p.m_tiles * ((n_rows + BN - 1) / BN);
    const size_t smem = L::BYTES + 1024;  // + alignment of the base to 1024 bytes
    if (cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(prefill_tc_kernel<BN>),
                                    static_cast<int>(TcLayout<BN>::BYTES + 1024));
        e != cudaSuccess)
        return e;
    const int64_t grid = p.tiles < num_sms() ? p.tiles : num_sms();
    return launch_pdl(prefill_tc_kernel<BN>, dim3(static_cast<unsigned>(grid)), dim3(TC_THREADS), smem, s, wmap, dmap,
                      p);
}

// Tile width: the one whose busiest SM covers the fewest output columns
// (tiles per SM x BN); on a tie the narrower tile, whose four-block batches
// amortise the pipeline's synchronisation best (measured on the 512 x 7168 x
// 1024 prompt contraction: 64 columns 30 us, 96 columns 33 us).
int prefill_tc_tile_n(int64_t n_rows, int64_t m)
{
    const int64_t sms = num_sms();
    int best = 64;
    int64_t best_cost = -1;
    for (int bn : {64, 96, 128}) {
        const int64_t tiles = act_tiles(m) * ((n_rows + bn - 1) / bn);
        const int64_t cost = (tiles + sms - 1) / sms * bn;
        if (best_cost < 0 || cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

cudaError_t launch_prefill_tc(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k, const void *xt,
                              int64_t m, float *y, int tile_n, cudaStream_t s)
{
    if (m == 0 || n_rows == 0) return cudaSuccess;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    if (tile_n == 0) tile_n = prefill_tc_tile_n(n_rows, m);
    switch (tile_n) {
        case 64: return launch_prefill_tc_bn<64>(enc, w_qs, w_d, n_rows, k, xt, m, y, s);
        case 96: return launch_prefill_tc_bn<96>(enc, w_qs, w_d, n_rows, k, xt, m, y, s);
        case 128: return launch_prefill_tc_bn<128>(enc, w_qs, w_d, n_rows, k, xt, m, y, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
