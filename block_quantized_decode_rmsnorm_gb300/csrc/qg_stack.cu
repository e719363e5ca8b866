// A whole stack of decode feed-forward blocks in one persistent launch.
//
// "Filling in the blanks: Inference using Phobos", Q4_K_M: fusing the whole MLP
// into one persistent kernel was worth a few percent on the pages' GPU; Fast
// Decode: the activation is quantized once and shared, the projections that
// read it are stacked, the residual add is folded into the matmul.  "One level
// down: #002 the same compiler on a GPU", Emitting for a GPU: the normalization
// is fused with the projection after it and the activation with the one before.
//
// GB300 design.  Each layer has two all-to-all dependencies: every gate|up CTA
// needs all of x (for the RMSNorm statistic), every down CTA needs all of h.
// Launched as separate kernels, each dependency costs a kernel boundary (about
// 1 us between the last CTA of one grid and the first wait return of the next).
// Here one cooperative grid (one CTA per SM, all resident together) runs every
// layer, and each dependency is a hand-off through 8-byte words that carry a
// 32-bit value and a 32-bit epoch, written with one store and read with one
// load, so a consumer that sees the epoch it expects has the value as well: no
// fence, no counter, no barrier.  Consumers poll their words; every poll is
// bounded by the global timer and by a shared status word, so a stalled
// producer turns into an error status and a normal return, never a hang.
//
// Per layer l and CTA c:
//  * phase A (CTAs c < ffn/32): block c of h.  Rows c*32.. of gate and of up
//    (64 rows, staged in shared memory long before) are dotted against the Q8_0
//    codes of RMSNorm(x)*gamma, which the CTA computes itself from x (polled);
//    warps 0-7 take the gate rows, warps 8-15 the up rows, each warp four K
//    blocks; then SiLU(g)*u and the block's Q8_0 codes and scale, published as
//    9 words.
//  * phase B (CTAs with output rows): rows c*rows_b.. of the down projection
//    with the residual, one warp per row, h's codes polled into shared memory;
//    x of the next layer published as one word per row (the last layer writes
//    x_out instead).
// Weight slabs are double-buffered by layer parity: layer l+1's down slab is
// requested after layer l's first barrier and layer l+2's gate|up slab after
// layer l's dots, so HBM streams the next layers while this one computes.
//
// Every sum is taken in the order of the two-launch layer (ffn_up_kernel, then
// gemv_prefetch_kernel), so the stack's output has the same bits as that path.
//
// Epochs: x of layer l (l >= 1) carries base + 2l, h of layer l base + 2l + 1,
// base = 256 * gen, where gen is a counter in the workspace that the last CTA
// of every launch increments.  A zero-filled workspace starts at gen 0 and its
// words at epoch 0, which no launch expects.
#include "qg_common.cuh"
#include "qg_norm.cuh"

namespace qg {

constexpr int kStackMaxLayers = 64;
// Every hand-off word is written to this many copies and each consumer CTA reads
// copy (CTA index mod kStackReplicas): with one copy, every CTA polling the same
// few kilobytes saturated the L2 slices that hold them (hand-offs of 1-2.5 us
// against 0.27-0.46 us for one CTA to another); a producer writes the copies
// with one store per lane.
constexpr int kStackReplicas = 16;
constexpr int kStackThreads = 512;
constexpr uint32_t kStackStall = 1u;      // status bit: a hand-off wait ran out (or saw another CTA's)
constexpr uint32_t kStackCopyStall = 2u;  // status bit: a weight slab did not land in time

struct StackLayer {
    const float *gamma;     // [k]
    const int8_t *wgu_qs;   // [2F][k]
    const uint16_t *wgu_d;  // [2F][k/32]
    const int8_t *wdn_qs;   // [k][F]
    const uint16_t *wdn_d;  // [k][F/32]
};

struct StackParams {
    const float *x_in;  // [k] layer 0's input (device or pinned host memory)
    float *x_out;       // [k] the last layer's output (device or pinned host memory)
    uint32_t *ctl;      // workspace: [0] status, [1] gen, [2] CTAs done
    uint64_t *xw;       // workspace: kStackReplicas copies, xstride words apart, of the k words of x
    uint64_t *hw;       // workspace: kStackReplicas copies, hstride words apart, of F/4 code words
                        // then F/32 scale words of h
    int xstride, hstride;
    float *h_last;      // optional [F]: the last layer's h
    int8_t *hq_last;    // optional [F]
    uint16_t *hd_last;  // optional [F/32]
    uint64_t wait_limit_ns;
    int n_layers;
    int k, nb;          // hidden size, its blocks
    int ffn, nbf;       // F, its blocks
    int units;          // F/32: CTAs with a block of h
    int rows_b;         // down rows per CTA
    int grid;
    float inv_k, eps;
    StackLayer layer[kStackMaxLayers];
};

// Shared-memory layout (byte offsets), the same on host and device.  Buffer b
// of a slab starts at its offset + b * its stride.
struct StackSmem {
    uint32_t a_w, a_d, a_g, a_stride;  // gate|up rows [64][k + 16], their scales [64][k/32], gamma [k] f32
    uint32_t b_w, b_d, b_stride;       // down rows [rows_b][F], their scales [rows_b][F/32]
    uint32_t red, part, x, res;        // row partials [2][8][32] f32, norm pairs [8][2] f32, x [k] f32, residuals [16] f32
    uint32_t hq, hd;                   // h codes [F], scales [F/32] f32
    uint32_t total;
};

__host__ __device__ inline uint32_t stack_round16(uint64_t bytes) { return static_cast<uint32_t>((bytes + 15) / 16 * 16); }

__host__ __device__ inline StackSmem stack_smem(int k, int ffn, int rows_b)
{
    StackSmem s;
    s.a_w = 0;
    s.a_d = stack_round16(static_cast<uint64_t>(64) * (k + 16));
    s.a_g = s.a_d + stack_round16(static_cast<uint64_t>(64) * (k / 32) * 2);
    s.a_stride = s.a_g + stack_round16(static_cast<uint64_t>(4) * k);
    s.b_w = 2 * s.a_stride;
    s.b_d = s.b_w + stack_round16(static_cast<uint64_t>(rows_b) * ffn);
    s.b_stride = s.b_d + stack_round16(static_cast<uint64_t>(rows_b) * (ffn / 32) * 2) - s.b_w;
    s.red = s.b_w + 2 * s.b_stride;
    s.part = s.red + 2 * 8 * 32 * 4;
    s.x = s.part + 16 * 4;
    s.res = s.x + stack_round16(static_cast<uint64_t>(4) * k);
    s.hq = s.res + 16 * 4;
    s.hd = s.hq + stack_round16(static_cast<uint64_t>(ffn));
    s.total = s.hd + stack_round16(static_cast<uint64_t>(ffn / 32) * 4);
    return s;
}

// ---- hand-off words ------------------------------------------------------------
__device__ __forceinline__ void st_word(uint64_t *p, uint32_t value, uint32_t epoch)
{
    const uint64_t v = (static_cast<uint64_t>(epoch) << 32) | value;
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_word(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Two consecutive words (16-byte aligned); each is read as one 8-byte access.
__device__ __forceinline__ void ld_word2(const uint64_t *p, uint64_t &a, uint64_t &b)
{
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ uint32_t ld_status(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t epoch_of(uint64_t w) { return static_cast<uint32_t>(w >> 32); }
__device__ __forceinline__ uint32_t value_of(uint64_t w) { return static_cast<uint32_t>(w); }

// A warp waits for the word pairs [p0, p1) (pair i = words 2i, 2i+1) to carry
// `epoch`: lane j reads pairs p0 + j + 32 m (m < kPollPerLane) with one 16-byte
// load each, all in flight together, hands every pair that is ready to
// sink(pair, value 2i, value 2i+1) and reads again only the pairs still missing,
// sleeping between rounds so that the consumers of a hand-off (every CTA reads
// the same few kilobytes) do not flood the L2 slices that hold them.  False,
// for the whole warp, once the wait has run longer than limit_ns or another CTA
// has set the status.
constexpr int kPollPerLane = 5;  // pairs per lane: up to 160 pairs per warp
constexpr int kPollWarps = 4;    // warps that read one hand-off

template <typename Sink>
__device__ __forceinline__ bool warp_poll(const uint64_t *w, int p0, int p1, uint32_t epoch, const uint32_t *status,
                                          uint64_t limit_ns, Sink sink)
{
    const int lane = threadIdx.x & 31;
    uint32_t pending = 0u;
#pragma unroll
    for (int m = 0; m < kPollPerLane; ++m)
        if (p0 + lane + 32 * m < p1) pending |= 1u << m;
    uint64_t t0 = 0;
    for (int round = 0;; ++round) {
        uint64_t a[kPollPerLane], b[kPollPerLane];
#pragma unroll
        for (int m = 0; m < kPollPerLane; ++m)
            if ((pending >> m) & 1u) ld_word2(w + 2 * (p0 + lane + 32 * m), a[m], b[m]);
#pragma unroll
        for (int m = 0; m < kPollPerLane; ++m) {
            if (((pending >> m) & 1u) && epoch_of(a[m]) == epoch && epoch_of(b[m]) == epoch) {
                sink(p0 + lane + 32 * m, value_of(a[m]), value_of(b[m]));
                pending &= ~(1u << m);
            }
        }
        if (__all_sync(0xffffffffu, pending == 0u)) return true;
        const uint64_t now = global_ns();
        if (round == 0) t0 = now;
        const bool give_up = now - t0 > limit_ns || ld_status(status) != 0u;
        if (__any_sync(0xffffffffu, give_up)) return false;
        __nanosleep(round < 2 ? 32u : 128u);
    }
}

// ---- shared pieces of the two phases (as in the two-launch layer) --------------
__device__ __forceinline__ float stack_block_term(const u32x8 &w, const u32x8 &x, float dw, float dx, float acc)
{
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s = dp4a(w.v[i], x.v[i], s);
    return fmaf(small_int_to_float(s), dw * dx, acc);
}

__device__ __forceinline__ u32x8 stack_ld_halves(const int8_t *p, int c0)
{
    const uint4 a = *reinterpret_cast<const uint4 *>(p + 16 * c0);
    const uint4 b = *reinterpret_cast<const uint4 *>(p + 16 * (c0 ^ 1));
    u32x8 r;
    r.v[0] = a.x; r.v[1] = a.y; r.v[2] = a.z; r.v[3] = a.w;
    r.v[4] = b.x; r.v[5] = b.y; r.v[6] = b.z; r.v[7] = b.w;
    return r;
}

// ---- slab copies ----------------------------------------------------------------
// Gate|up slab of unit c for layer l: 64 rows (two per lane of warp `wr`), the
// two scale slabs and gamma (lanes 0-2 of warp `wr + 1`).  One lane arms the
// barrier with the whole byte count; complete_tx before the arming arrival cannot
// finish the phase (its one arrival is still pending).
__device__ __forceinline__ void issue_a(const StackParams &p, const StackSmem &S, uint8_t *smem, uint64_t *bar,
                                       uint32_t *cnt, int l, int buf, int wr, int warp, int lane)
{
    const StackLayer &ly = p.layer[l];
    const int K = p.k, nb = p.nb, KP = K + 16;
    const int64_t ob = static_cast<int64_t>(blockIdx.x) * 32;
    if (warp == wr) {
        if (lane == 0) {
            mbar_expect_tx(bar, 64u * K + 128u * nb + 4u * K);
            ++*cnt;
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = lane + 32 * h;  // gate rows, then up rows
            const int64_t src = h == 0 ? ob + lane : p.ffn + ob + lane;
            bulk_copy_g2s(smem + S.a_w + buf * S.a_stride + row * KP, ly.wgu_qs + src * K, static_cast<uint32_t>(K), bar,
                          l2_evict_first_policy());
        }
    } else if (warp == wr + 1 && lane < 3) {
        void *dst = lane == 0 ? static_cast<void *>(smem + S.a_g + buf * S.a_stride)
                              : static_cast<void *>(smem + S.a_d + buf * S.a_stride + (lane - 1) * 64 * nb);
        const void *src = lane == 0 ? static_cast<const void *>(ly.gamma)
                                    : static_cast<const void *>(ly.wgu_d + (lane == 1 ? ob : p.ffn + ob) * nb);
        bulk_copy_g2s(dst, src, lane == 0 ? 4u * K : 64u * nb, bar,
                      lane == 0 ? l2_evict_last_policy() : l2_evict_first_policy());
    }
}

// Down slab of this CTA's rows for layer l: four value pieces and the scales on
// lanes 0-4 of warp `wr`, issued in one instruction.
__device__ __forceinline__ void issue_b(const StackParams &p, const StackSmem &S, uint8_t *smem, uint64_t *bar,
                                       uint32_t *cnt, int l, int buf, int nrow, int wr, int warp, int lane)
{
    if (warp != wr) return;
    const StackLayer &ly = p.layer[l];
    const int F = p.ffn, nbf = p.nbf;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * p.rows_b;
    const uint32_t vbytes = static_cast<uint32_t>(nrow) * F, sbytes = static_cast<uint32_t>(nrow) * 2 * nbf;
    if (lane == 0) {
        mbar_expect_tx(bar, vbytes + sbytes);
        ++*cnt;
    }
    __syncwarp();
    const int pr = (nrow + 3) / 4;  // rows per value piece
    const int v0 = (lane - 1) * pr;
    const int vr = lane == 0 ? 0 : (nrow - v0 < pr ? nrow - v0 : pr);
    if (lane == 0 || (lane <= 4 && vr > 0)) {
        void *dst = lane == 0 ? static_cast<void *>(smem + S.b_d + buf * S.b_stride)
                              : static_cast<void *>(smem + S.b_w + buf * S.b_stride + static_cast<size_t>(v0) * F);
        const void *src = lane == 0 ? static_cast<const void *>(ly.wdn_d + r0 * nbf)
                                    : static_cast<const void *>(ly.wdn_qs + (r0 + v0) * F);
        bulk_copy_g2s(dst, src, lane == 0 ? sbytes : static_cast<uint32_t>(vr) * F, bar, l2_evict_first_policy());
    }
}

// ---------------------------------------------------------------------------
// the kernel: 512 threads, one CTA per SM, launched cooperatively
// ---------------------------------------------------------------------------
template <int NBB>  // ceil(F / 32 / 32): h blocks per lane in the down rows
__global__ void __launch_bounds__(kStackThreads, 1) decode_stack_kernel(const __grid_constant__ StackParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_bar[4];  // gate|up slab 0, 1; down slab 0, 1
    __shared__ uint32_t s_cnt[4];               // phases armed on each barrier

    const StackSmem S = stack_smem(p.k, p.ffn, p.rows_b);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int K = p.k, nb = p.nb, KP = K + 16, F = p.ffn, nbf = p.nbf, L = p.n_layers;
    const bool has_a = static_cast<int>(blockIdx.x) < p.units;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * p.rows_b;
    const int nrow = static_cast<int>(K - r0 <= 0 ? 0 : (K - r0 < p.rows_b ? K - r0 : p.rows_b));
    const uint32_t *status = p.ctl;
    const uint32_t gen = p.ctl[1];  // written only by the previous launch
    const uint32_t base = gen * 256u;

    float *s_red = reinterpret_cast<float *>(smem + S.red);    // [2][8][32]
    float *s_part = reinterpret_cast<float *>(smem + S.part);  // [8][2]
    float *s_x = reinterpret_cast<float *>(smem + S.x);        // [K]
    float *s_res = reinterpret_cast<float *>(smem + S.res);    // [16]
    int8_t *s_hq = reinterpret_cast<int8_t *>(smem + S.hq);    // [F]
    float *s_hd = reinterpret_cast<float *>(smem + S.hd);      // [F/32]

    if (t == 0) {
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s_bar[i], 1);
            s_cnt[i] = 0;
        }
    }
    __syncthreads();
    // the slabs of layers 0 and 1
    for (int l = 0; l < 2 && l < L; ++l) {
        if (has_a) issue_a(p, S, smem, &s_bar[l], &s_cnt[l], l, l, 2 * l, warp, lane);
        if (nrow > 0) issue_b(p, S, smem, &s_bar[2 + l], &s_cnt[2 + l], l, l, nrow, 4 + l, warp, lane);
    }

    // phase-A thread roles: group g (0 gate, 1 up) of eight warps; warp wl of the
    // group owns K blocks wl + 8 q (q = lane / 8) and, in its lane group, rows
    // rg + 8 i (i < 4) of the group's 32 rows
    const int g = warp >> 3, wl = warp & 7;
    const int rg = lane & 7;
    const int xb = wl + 8 * (lane >> 3);
    const int xo = 32 * xb + 4 * rg;
    const bool live = xb < nb;
    const int64_t ob = static_cast<int64_t>(blockIdx.x) * 32;

    uint32_t stall = 0;
    for (int l = 0; l < L; ++l) {
        const int buf = l & 1;
        const uint32_t par = static_cast<uint32_t>(l >> 1) & 1u;
        if (has_a) {
            // ---- x of this layer (warps 0-3 read it into shared memory), the
            // norm statistic ---------------------------------------------------------
            bool ok = true;
            if (warp < kPollWarps) {
                const int np = K / 2, per = np / kPollWarps;  // K / 2 pairs, a quarter per warp
                const int p0 = warp * per, p1 = warp == kPollWarps - 1 ? np : p0 + per;
                if (l == 0) {
                    for (int pp = p0 + lane; pp < p1; pp += 32)
                        reinterpret_cast<float2 *>(s_x)[pp] = reinterpret_cast<const float2 *>(p.x_in)[pp];
                } else {
                    const uint64_t *xw = p.xw + static_cast<size_t>(blockIdx.x % kStackReplicas) * p.xstride;
                    ok = warp_poll(xw, p0, p1, base + 2u * l, status, p.wait_limit_ns,
                                   [&](int pp, uint32_t a, uint32_t b) {
                                       reinterpret_cast<float2 *>(s_x)[pp] = make_float2(__uint_as_float(a), __uint_as_float(b));
                                   });
                }
            }
            if (__syncthreads_or(!ok)) {  // x in shared memory
                stall = kStackStall;
                break;
            }
            float4 xv4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live) xv4 = *reinterpret_cast<const float4 *>(s_x + xo);
            f32pair acc = {0.0f, 0.0f};
            if (live) {
                pair_add_square(acc, xv4.x);
                pair_add_square(acc, xv4.y);
                pair_add_square(acc, xv4.z);
                pair_add_square(acc, xv4.w);
            }
            acc = warp_pair_sum(acc);
            if (g == 0 && lane == 0) {
                s_part[2 * wl] = acc.hi;
                s_part[2 * wl + 1] = acc.lo;
            }
            const bool staged = mbar_wait_bounded(&s_bar[buf], par, p.wait_limit_ns);
            if (__syncthreads_or(!staged)) {  // barrier 1
                stall = kStackCopyStall;
                break;
            }
            if (l >= 1 && l + 1 < L && nrow > 0)
                issue_b(p, S, smem, &s_bar[2 + (buf ^ 1)], &s_cnt[2 + (buf ^ 1)], l + 1, buf ^ 1, nrow, 3, warp, lane);

            f32pair tot = {0.0f, 0.0f};
            if (lane < 8) tot = f32pair{s_part[2 * lane], s_part[2 * lane + 1]};
#pragma unroll
            for (int off = 4; off >= 1; off >>= 1) {
                f32pair o;
                o.hi = __shfl_xor_sync(0xffffffffu, tot.hi, off);
                o.lo = __shfl_xor_sync(0xffffffffu, tot.lo, off);
                tot = pair_merge(tot, o);
            }
            tot.hi = __shfl_sync(0xffffffffu, tot.hi, 0);
            tot.lo = __shfl_sync(0xffffffffu, tot.lo, 0);
            const float r = rms_inv_from_pair(tot, K, p.inv_k, p.eps);

            // ---- Q8_0 of x_hat = (x r) gamma, eight threads per block ------------
            uint32_t xc = 0u;
            float xdf = 0.0f;
            {
                const float *s_g = reinterpret_cast<const float *>(smem + S.a_g + buf * S.a_stride);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (live) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(s_g + xo);
                    v.x = __fmul_rn(__fmul_rn(xv4.x, r), g4.x);
                    v.y = __fmul_rn(__fmul_rn(xv4.y, r), g4.y);
                    v.z = __fmul_rn(__fmul_rn(xv4.z, r), g4.z);
                    v.w = __fmul_rn(__fmul_rn(xv4.w, r), g4.w);
                }
                float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                if (live) {
                    const float dd = div127(m);
                    xc = q8_pack4(v, dd, q8_recip(dd));
                    xdf = h2f(f2h_rn(dd));
                }
            }

            // ---- block dots: block xb of rows 32 g + rg + 8 i ---------------------
            u32x8 xw;
            const int src = lane & 24;
#pragma unroll
            for (int s = 0; s < 8; ++s) xw.v[s] = __shfl_sync(0xffffffffu, xc, src + s);
            const float xs = __shfl_sync(0xffffffffu, xdf, src);
            const int8_t *s_w = reinterpret_cast<const int8_t *>(smem + S.a_w + buf * S.a_stride);
            const uint16_t *s_wd = reinterpret_cast<const uint16_t *>(smem + S.a_d + buf * S.a_stride);
            float part[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 32 * g + rg + 8 * i;
                part[i] = live ? stack_block_term(stack_ld_halves(s_w + row * KP + xb * QK, 0), xw,
                                                  h2f(s_wd[row * nb + xb]), xs, 0.0f)
                               : 0.0f;
            }
            // lane groups: offset 16 (block bit 4), then 8 (bit 3); lane l ends
            // with row 32 g + l
            float v2[2];
            {
                const bool up = (lane & 16) != 0;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float send = up ? part[k] : part[k + 2];
                    const float keep = up ? part[k + 2] : part[k];
                    v2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
            }
            float v1;
            {
                const bool up = (lane & 8) != 0;
                const float send = up ? v2[0] : v2[1];
                const float keep = up ? v2[1] : v2[0];
                v1 = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            s_red[(g * 8 + wl) * 32 + lane] = v1;
            __syncthreads();  // barrier 2: every warp is done with this layer's gate|up slab
            if (l + 2 < L) issue_a(p, S, smem, &s_bar[buf], &s_cnt[buf], l + 2, buf, 2, warp, lane);

            // ---- warp 0: row totals (block bits 2, 1, 0), SiLU(g) u, Q8_0 of h ----
            if (warp == 0) {
                auto row_total = [&](int grp) {
                    const float *c = s_red + grp * 8 * 32 + lane;
                    return ((c[0] + c[4 * 32]) + (c[2 * 32] + c[6 * 32])) +
                           ((c[32] + c[5 * 32]) + (c[3 * 32] + c[7 * 32]));
                };
                const float v = silu_mul(row_total(0), row_total(1));
                const float m = warp_max_abs(v);
                const float dd = div127(m);
                const uint32_t code = static_cast<uint32_t>(q8_code(v, dd, q8_recip(dd))) & 0xffu;
                const uint16_t dbits = f2h_rn(dd);
                // lane j holds code word j % 8 and writes it to copies j / 8 + 4 m;
                // lanes below kStackReplicas write the scale word's copies
                uint32_t word = 0u;
#pragma unroll
                for (int s = 0; s < 4; ++s) word |= __shfl_sync(0xffffffffu, code, 4 * (lane & 7) + s) << (8 * s);
                const uint32_t eh = base + 2u * l + 1u;
#pragma unroll
                for (int m = 0; m < kStackReplicas / 4; ++m)
                    st_word(p.hw + static_cast<size_t>((lane >> 3) + 4 * m) * p.hstride + ob / 4 + (lane & 7), word, eh);
                if (lane < kStackReplicas)
                    st_word(p.hw + static_cast<size_t>(lane) * p.hstride + F / 4 + blockIdx.x, dbits, eh);

                if (l == L - 1) {
                    if (p.h_last) p.h_last[ob + lane] = v;
                    if (p.hq_last) p.hq_last[ob + lane] = static_cast<int8_t>(code);
                    if (p.hd_last && lane == 0) p.hd_last[blockIdx.x] = dbits;
                }
            }
        } else if (l >= 1) {
            __syncthreads();  // every warp is done with layer l - 1's down slab
            if (l + 1 < L && nrow > 0)
                issue_b(p, S, smem, &s_bar[2 + (buf ^ 1)], &s_cnt[2 + (buf ^ 1)], l + 1, buf ^ 1, nrow, 3, warp, lane);
        }

        if (nrow > 0) {
            // ---- h codes and scales of this layer (warps 4-7 read them into
            // shared memory); layer 0's residual rows (warp 3) -------------------------
            bool ok = true;
            const uint32_t eh = base + 2u * l + 1u;
            if (warp >= 4 && warp < 4 + kPollWarps) {
                const int np = (F / 4 + nbf) / 2, per = (np + kPollWarps - 1) / kPollWarps;
                const int p0 = (warp - 4) * per, p1 = p0 + per < np ? p0 + per : np;
                const uint64_t *hw = p.hw + static_cast<size_t>(blockIdx.x % kStackReplicas) * p.hstride;
                ok = warp_poll(hw, p0, p1, eh, status, p.wait_limit_ns, [&](int pp, uint32_t a, uint32_t b) {
                    if (2 * pp < F / 4) {
                        reinterpret_cast<uint2 *>(s_hq)[pp] = make_uint2(a, b);
                    } else {
                        const int blk = 2 * pp - F / 4;
                        s_hd[blk] = h2f(static_cast<uint16_t>(a));
                        s_hd[blk + 1] = h2f(static_cast<uint16_t>(b));
                    }
                });
            } else if (warp == 3 && lane < nrow && l == 0) {
                s_res[lane] = p.x_in[r0 + lane];  // later layers: kept by the row's warp from the layer before
            }
            const bool staged = mbar_wait_bounded(&s_bar[2 + buf], par, p.wait_limit_ns);
            if (__syncthreads_or(!ok || !staged)) {  // barrier 3
                stall = __syncthreads_or(!staged) ? kStackCopyStall : kStackStall;
                break;
            }
            const float res = s_res[warp < 16 ? warp : 0];

            // ---- down rows: one warp per row -------------------------------------
            if (warp < nrow) {
                const int c0 = (lane >> 2) & 1;
                const int8_t *s_w = reinterpret_cast<const int8_t *>(smem + S.b_w + buf * S.b_stride) + static_cast<size_t>(warp) * F;
                const uint16_t *s_wd = reinterpret_cast<const uint16_t *>(smem + S.b_d + buf * S.b_stride) + warp * nbf;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < NBB; ++j) {
                    const int blk = lane + 32 * j;
                    u32x8 wv, hv;
                    float wsc = 0.0f, hs = 0.0f;
                    if (blk < nbf) {
                        wv = stack_ld_halves(s_w + blk * QK, c0);
                        hv = stack_ld_halves(s_hq + blk * QK, c0);
                        wsc = h2f(s_wd[blk]);
                        hs = s_hd[blk];
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) wv.v[i] = hv.v[i] = 0u;
                    }
                    acc = stack_block_term(wv, hv, wsc, hs, acc);
                }
                acc = warp_sum(acc);
                const float y = res + acc;  // every lane holds the row's total
                if (l == L - 1) {
                    if (lane == 0) p.x_out[r0 + warp] = y;
                } else {
                    if (lane < kStackReplicas)
                        st_word(p.xw + static_cast<size_t>(lane) * p.xstride + r0 + warp, __float_as_uint(y),
                                base + 2u * (l + 1));
                    if (lane == 0) s_res[warp] = y;  // the next layer's residual of this row
                }
            }
        }
    }

    // ---- exit: let every armed copy land, report, count this CTA out ----------
    __syncthreads();
    if (t == 0) {
        for (int i = 0; i < 4; ++i)
            if (s_cnt[i] > 0) mbar_wait_bounded(&s_bar[i], (s_cnt[i] - 1) & 1u, kCopyWaitLimitNs);
        if (stall) atomicOr(p.ctl, stall);
        __threadfence();
        if (atomicAdd(p.ctl + 2, 1u) == static_cast<uint32_t>(p.grid) - 1u) {
            p.ctl[2] = 0u;
            p.ctl[1] = gen + 1u;
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr size_t kStackMaxSmem = 227 * 1024 - 1024;

struct StackShape {
    int rows_b, grid;
    size_t smem;
};

// Shapes the stack serves: hidden a multiple of 256 up to 1024 (one K block per
// lane group), ffn a multiple of 256 up to 4096 with a CTA per h block, at most
// 16 down rows per CTA, and both layers' slabs in one CTA's shared memory.
bool stack_shape(int64_t k, int64_t ffn, StackShape *out)
{
    if (k <= 0 || k % 256 != 0 || k > 1024 || ffn <= 0 || ffn % 256 != 0 || ffn > 4096) return false;
    const int sms = num_sms();
    if (ffn / 32 > sms) return false;
    const int rows_b = static_cast<int>((k + sms - 1) / sms);
    if (rows_b > 16) return false;
    const int b_ctas = static_cast<int>((k + rows_b - 1) / rows_b);
    const int grid = static_cast<int>(ffn / 32) > b_ctas ? static_cast<int>(ffn / 32) : b_ctas;
    const size_t smem = stack_smem(static_cast<int>(k), static_cast<int>(ffn), rows_b).total;
    if (smem > kStackMaxSmem) return false;
    if (out) *out = StackShape{rows_b, grid, smem};
    return true;
}

// Copies of the hand-off words are a multiple of 4 KB plus 512 B apart, so that
// the copies of one word fall on different L2 lines and slices.
static size_t stack_stride_words(size_t words) { return (words + 511) / 512 * 512 + 64; }
static size_t stack_xstride(int64_t k) { return stack_stride_words(static_cast<size_t>(k)); }
static size_t stack_hstride(int64_t ffn)
{
    return stack_stride_words(static_cast<size_t>(ffn) / 4 + static_cast<size_t>(ffn) / 32);
}

// Workspace: control words (256 B), then the copies of the words of x, then
// those of h.
size_t stack_workspace_bytes(int64_t k, int64_t ffn)
{
    return 256 + static_cast<size_t>(kStackReplicas) * (stack_xstride(k) + stack_hstride(ffn)) * 8;
}

int stack_max_layers() { return kStackMaxLayers; }

template <int NBB>
static cudaError_t launch_stack_nbb(const StackParams &p, const StackShape &sh, cudaStream_t s)
{
    auto kern = decode_stack_kernel<NBB>;
    if (cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(kern), static_cast<int>(sh.smem)); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sh.grid));
    cfg.blockDim = dim3(kStackThreads);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once, or the launch fails
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_decode_stack(const float *x_in, float *x_out, int n_layers, const float *const *gamma,
                                const int8_t *const *wgu_qs, const uint16_t *const *wgu_d,
                                const int8_t *const *wdn_qs, const uint16_t *const *wdn_d, int64_t k, int64_t ffn,
                                float eps, void *workspace, float *h_last, int8_t *hq_last, uint16_t *hd_last,
                                uint64_t wait_limit_ns, cudaStream_t s)
{
    StackShape sh;
    if (!stack_shape(k, ffn, &sh) || n_layers <= 0 || n_layers > kStackMaxLayers) return cudaErrorInvalidValue;
    StackParams p = {};
    p.x_in = x_in;
    p.x_out = x_out;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.ctl = reinterpret_cast<uint32_t *>(ws);
    p.xstride = static_cast<int>(stack_xstride(k));
    p.hstride = static_cast<int>(stack_hstride(ffn));
    p.xw = reinterpret_cast<uint64_t *>(ws + 256);
    p.hw = p.xw + static_cast<size_t>(kStackReplicas) * p.xstride;
    p.h_last = h_last;
    p.hq_last = hq_last;
    p.hd_last = hd_last;
    p.wait_limit_ns = wait_limit_ns;
    p.n_layers = n_layers;
    p.k = static_cast<int>(k);
    p.nb = static_cast<int>(k / 32);
    p.ffn = static_cast<int>(ffn);
    p.nbf = static_cast<int>(ffn / 32);
    p.units = static_cast<int>(ffn / 32);
    p.rows_b = sh.rows_b;
    p.grid = sh.grid;
    p.inv_k = 1.0f / static_cast<float>(k);
    p.eps = eps;
    for (int l = 0; l < n_layers; ++l) p.layer[l] = StackLayer{gamma[l], wgu_qs[l], wgu_d[l], wdn_qs[l], wdn_d[l]};
    switch ((p.nbf + 31) / 32) {
    case 1: return launch_stack_nbb<1>(p, sh, s);
    case 2: return launch_stack_nbb<2>(p, sh, s);
    case 3: return launch_stack_nbb<3>(p, sh, s);
    case 4: return launch_stack_nbb<4>(p, sh, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
