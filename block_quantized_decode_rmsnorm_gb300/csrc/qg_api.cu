// extern "C" entry points of libqgemv.so: argument checks, then one launch.
// Declarations and the full contract are in include/qgemv.h.
#include <map>
#include <mutex>

#include "qg_common.cuh"

namespace qg {

cudaError_t launch_quantize_act(const float *, int64_t, int64_t, int8_t *, uint16_t *, cudaStream_t);
cudaError_t launch_rmsnorm_quantize(const float *, const float *, int64_t, int64_t, float, int8_t *, uint16_t *,
                                    float *, cudaStream_t);
cudaError_t launch_pack_q8_0(const void *, int64_t, int64_t, int8_t *, uint16_t *, cudaStream_t);
cudaError_t launch_rmsnorm_hadamard_quantize(const float *, const float *, int64_t, int64_t, float, int8_t *,
                                             uint16_t *, float *, float *, cudaStream_t);
cudaError_t launch_column_blocks(const int8_t *, const uint16_t *, int64_t, int64_t, int8_t *, uint16_t *,
                                 cudaStream_t);
cudaError_t launch_gemv_q8_0(const int8_t *, const uint16_t *, int64_t, int64_t, const int8_t *, const uint16_t *,
                             int64_t, int, const float *, float *, cudaStream_t);
cudaError_t launch_block_dots(const int8_t *, int64_t, int64_t, const int8_t *, int64_t, int32_t *, cudaStream_t);
cudaError_t launch_gemv_bf16(const uint16_t *, int64_t, int64_t, const uint16_t *, const uint16_t *, float, int,
                             const float *, float *, cudaStream_t);
cudaError_t launch_prefill_mma(const int8_t *, const uint16_t *, int64_t, int64_t, const int8_t *, const uint16_t *,
                               int64_t, float *, cudaStream_t);
bool ffn_up_supported(int64_t k, int64_t half);
cudaError_t launch_ffn_up(const float *, const float *, int64_t, float, const int8_t *, const uint16_t *, int64_t,
                          float *, int8_t *, uint16_t *, int8_t *, uint16_t *, float *, cudaStream_t);
bool prefetch_supported(int64_t n_rows, int64_t k);
bool ffn_up_rotated_supported(int64_t k, int64_t half);
cudaError_t launch_ffn_up_rotated(const float *, const float *, int64_t, float, const int8_t *, const uint16_t *,
                                  int64_t, float *, int8_t *, uint16_t *, int8_t *, uint16_t *, cudaStream_t);
bool decode_layer_supported(int64_t k, int64_t half);
int decode_layer_partials(int64_t half);
constexpr int kMaxLayerPartials = 16;
cudaError_t launch_decode_layer(const float *, const float *, int, float *, float *, const float *, int64_t, float,
                                const int8_t *, const uint16_t *, const int8_t *, const uint16_t *, int64_t, float *,
                                int8_t *, uint16_t *, cudaStream_t);
cudaError_t launch_layer_finish(const float *, const float *, int, int64_t, float *, cudaStream_t);
size_t layer_scratch_bytes(int64_t hidden, int64_t ffn, int partials);
size_t layer_scratch_capacity();
cudaError_t launch_decode_layers_noalloc(const float *, float *, int, const float *const *, const int8_t *const *,
                                         const uint16_t *const *, const int8_t *const *, const uint16_t *const *,
                                         int64_t, int64_t, float, cudaStream_t);
cudaError_t launch_quantize_act_tiles(const float *, int64_t, int64_t, void *, cudaStream_t);
bool prefill_tc_supported(int64_t k);
bool prefill_bf16_supported(int64_t k);
cudaError_t launch_mma_s8_rate(int64_t, int *, int64_t *, cudaStream_t);
int hbm_read_ctas();
cudaError_t launch_hbm_read(const void *, int64_t, uint32_t *, cudaStream_t);
cudaError_t launch_empty_chain(int, int, int, cudaStream_t);
cudaError_t launch_pack_q8_0_f16(const int8_t *, const uint16_t *, int64_t, int64_t, uint16_t *, float *, cudaStream_t);
cudaError_t launch_quantize_act_f16(const float *, int64_t, int64_t, uint16_t *, float *, cudaStream_t);
cudaError_t launch_prefill_tc2(const uint16_t *, const float *, int64_t, int64_t, const uint16_t *, const float *,
                               int64_t, float *, int, cudaStream_t);
cudaError_t launch_prefill_bf16(const uint16_t *, int64_t, int64_t, const uint16_t *, int64_t, const uint16_t *, float,
                                int, uint16_t *, float *, cudaStream_t);
cudaError_t launch_prefill_tc(const int8_t *, const uint16_t *, int64_t, int64_t, const void *, int64_t, float *, int,
                              cudaStream_t);
cudaError_t launch_gemv_prefetch(const int8_t *, const uint16_t *, int64_t, int64_t, const int8_t *, const uint16_t *,
                                 int, const float *, float *, cudaStream_t);
cudaError_t copy_stalls(uint32_t *count, bool clear);
struct StackShape {
    int rows_b, grid;
    size_t smem;
};
bool stack_shape(int64_t k, int64_t ffn, StackShape *out);
size_t stack_workspace_bytes(int64_t k, int64_t ffn);
int stack_max_layers();
cudaError_t launch_decode_stack(const float *, float *, int, const float *const *, const int8_t *const *,
                                const uint16_t *const *, const int8_t *const *, const uint16_t *const *, int64_t,
                                int64_t, float, void *, float *, int8_t *, uint16_t *, uint64_t, cudaStream_t);

// SM count of the current device, read once per device.
int num_sms()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

cudaError_t opt_in_smem(const void *func, int bytes)
{
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> done;  // (device, kernel) -> bytes opted in
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    int &have = done[{dev, func}];
    if (have >= bytes) return cudaSuccess;
    if (cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        e != cudaSuccess)
        return e;
    have = bytes;
    return cudaSuccess;
}

}  // namespace qg

namespace {

constexpr int64_t kMaxK = int64_t(1) << 20;       // longest supported reduction
constexpr int64_t kMaxRows = int64_t(1) << 31;    // rows per call

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [a, a + na) and [b, b + nb) share a byte
bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}
bool overlap(const void *a, const void *b, size_t bytes) { return overlap(a, bytes, b, bytes); }

qg_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status check_q8_k(int64_t k)
{
    if (k <= 0 || k % 32 != 0 || k > kMaxK) return QG_ERR_SHAPE;
    return QG_OK;
}

}  // namespace

extern "C" {

const char *qg_status_str(qg_status s)
{
    switch (s) {
    case QG_OK: return "ok";
    case QG_ERR_NULL: return "null pointer";
    case QG_ERR_ALIGN: return "misaligned pointer";
    case QG_ERR_SHAPE: return "bad shape";
    case QG_ERR_UNSUPPORTED: return "unsupported request";
    case QG_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int qg_abi_version(void) { return 1; }

qg_status qg_q8_0_pack(const void *blocks, int64_t n_rows, int64_t k, int8_t *qs, uint16_t *d, qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (n_rows == 0) return QG_OK;
    if (!blocks || !qs || !d) return QG_ERR_NULL;
    if (!aligned(qs, 32) || !aligned(d, 2)) return QG_ERR_ALIGN;
    return from_cuda(qg::launch_pack_q8_0(blocks, n_rows, k, qs, d, stream));
}

qg_status qg_q8_0_column_blocks(const int8_t *qs, const uint16_t *d, int64_t n_rows, int64_t k, int8_t *qs_cb,
                                uint16_t *d_cb, qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (n_rows == 0) return QG_OK;
    if (!qs || !d || !qs_cb || !d_cb) return QG_ERR_NULL;
    if (!aligned(qs, 32) || !aligned(qs_cb, 32) || !aligned(d, 2) || !aligned(d_cb, 2)) return QG_ERR_ALIGN;
    if (overlap(qs, qs_cb, static_cast<size_t>(n_rows) * k) || overlap(d, d_cb, static_cast<size_t>(n_rows) * (k / 32) * 2))
        return QG_ERR_SHAPE;
    return from_cuda(qg::launch_column_blocks(qs, d, n_rows, k, qs_cb, d_cb, stream));
}

qg_status quantize_act_q8_0(const float *x, int64_t rows, int64_t k, int8_t *q, uint16_t *d, qg_stream_t stream)
{
    if (rows < 0 || rows > kMaxRows) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (rows == 0) return QG_OK;
    if (!x || !q || !d) return QG_ERR_NULL;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(d, 2)) return QG_ERR_ALIGN;
    return from_cuda(qg::launch_quantize_act(x, rows, k, q, d, stream));
}

// Activation tiles: rows up to 2^24, and (tiles x blocks x 4) warps' worth of
// 8-lane groups must fit one launch grid.
static bool act_tiles_shape_ok(int64_t rows, int64_t k)
{
    if (rows < 0 || rows > (int64_t(1) << 24) || k <= 0 || k > kMaxK) return false;
    return qg::act_tiles(rows) * (k / qg::QK) * 4 < (int64_t(1) << 31);
}

int64_t qg_act_tiles_bytes(int64_t rows, int64_t k)
{
    if (k % qg::QK != 0 || !act_tiles_shape_ok(rows, k)) return -1;
    return qg::act_tiles(rows) * (k / qg::QK) * qg::ACT_TILE_RECORD;
}

qg_status quantize_act_q8_0_tiles(const float *x, int64_t rows, int64_t k, void *xt, qg_stream_t stream)
{
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (!act_tiles_shape_ok(rows, k)) return QG_ERR_SHAPE;
    if (rows == 0) return QG_OK;
    if (!x || !xt) return QG_ERR_NULL;
    if (!aligned(x, 16) || !aligned(xt, 16)) return QG_ERR_ALIGN;
    return from_cuda(qg::launch_quantize_act_tiles(x, rows, k, xt, stream));
}

qg_status rmsnorm_quantize(const float *x, const float *gamma, int64_t rows, int64_t k, float eps, int8_t *q,
                           uint16_t *d, float *inv_rms, qg_stream_t stream)
{
    if (rows < 0 || rows > (int64_t(1) << 31) - 1) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (k > 65536) return QG_ERR_SHAPE;
    if (!(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (rows == 0) return QG_OK;
    if (!x || !gamma || !q || !d) return QG_ERR_NULL;
    if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(q, 16) || !aligned(d, 2) || !aligned(inv_rms, 4))
        return QG_ERR_ALIGN;
    return from_cuda(qg::launch_rmsnorm_quantize(x, gamma, rows, k, eps, q, d, inv_rms, stream));
}

qg_status rmsnorm_hadamard_quantize(const float *x, const float *gamma, int64_t rows, int64_t k, float eps,
                                    int8_t *q, uint16_t *d, float *z, float *inv_rms, qg_stream_t stream)
{
    if (rows < 0 || rows > (int64_t(1) << 31) - 1) return QG_ERR_SHAPE;
    if (k <= 0 || k % 128 != 0 || k > 65536) return QG_ERR_SHAPE;
    if (!(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (rows == 0) return QG_OK;
    if (!x || !gamma || !q || !d) return QG_ERR_NULL;
    if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(q, 16) || !aligned(d, 2) || !aligned(z, 16) ||
        !aligned(inv_rms, 4))
        return QG_ERR_ALIGN;
    return from_cuda(qg::launch_rmsnorm_hadamard_quantize(x, gamma, rows, k, eps, q, d, z, inv_rms, stream));
}

qg_status qgemv_q8_0(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k, const int8_t *xq,
                     const uint16_t *xd, int64_t batch, int epilogue, const float *residual, float *y,
                     qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (batch < 1) return QG_ERR_SHAPE;
    if (batch > 8) return QG_ERR_UNSUPPORTED;
    if (epilogue != QG_EPI_NONE && epilogue != QG_EPI_SILU_MUL_HALVES && epilogue != QG_EPI_RESIDUAL_ADD)
        return QG_ERR_UNSUPPORTED;
    if (epilogue == QG_EPI_SILU_MUL_HALVES && (n_rows % 2) != 0) return QG_ERR_SHAPE;
    if (n_rows == 0) return QG_OK;
    if (!w_qs || !w_d || !xq || !xd || !y) return QG_ERR_NULL;
    if (epilogue == QG_EPI_RESIDUAL_ADD && !residual) return QG_ERR_NULL;
    if (!aligned(w_qs, 32) || !aligned(w_d, 2) || !aligned(xq, 16) || !aligned(xd, 2) || !aligned(y, 16))
        return QG_ERR_ALIGN;
    if (epilogue == QG_EPI_RESIDUAL_ADD && !aligned(residual, 16)) return QG_ERR_ALIGN;
    // Batch-1 products whose weights fit in one wave's registers take the
    // prefetching kernel; everything else streams.
    if (batch == 1 && epilogue != QG_EPI_SILU_MUL_HALVES && aligned(w_d, 16) &&
        qg::prefetch_supported(n_rows, k))
        return from_cuda(qg::launch_gemv_prefetch(w_qs, w_d, n_rows, k, xq, xd, epilogue, residual, y, stream));
    return from_cuda(qg::launch_gemv_q8_0(w_qs, w_d, n_rows, k, xq, xd, batch, epilogue, residual, y, stream));
}

qg_status qgemv_bf16(const uint16_t *w, int64_t n_rows, int64_t k, const uint16_t *x, const uint16_t *gamma,
                     float eps, int epilogue, const float *residual, float *y, qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows) return QG_ERR_SHAPE;
    if (k <= 0 || k % 8 != 0 || k > 16384) return QG_ERR_SHAPE;
    if (!(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (epilogue != QG_EPI_NONE && epilogue != QG_EPI_SILU_MUL_HALVES && epilogue != QG_EPI_RESIDUAL_ADD)
        return QG_ERR_UNSUPPORTED;
    if (epilogue == QG_EPI_SILU_MUL_HALVES && (n_rows % 2) != 0) return QG_ERR_SHAPE;
    if (n_rows == 0) return QG_OK;
    if (!w || !x || !y) return QG_ERR_NULL;
    if (epilogue == QG_EPI_RESIDUAL_ADD && !residual) return QG_ERR_NULL;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(gamma, 16) || !aligned(y, 16)) return QG_ERR_ALIGN;
    if (epilogue == QG_EPI_RESIDUAL_ADD && !aligned(residual, 16)) return QG_ERR_ALIGN;
    return from_cuda(qg::launch_gemv_bf16(w, n_rows, k, x, gamma, eps, epilogue, residual, y, stream));
}

qg_status qgemm_q8_0_prefill(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k, const int8_t *xq,
                             const uint16_t *xd, int64_t m, float *y, qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows || m < 0 || m > (int64_t(1) << 24)) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (k > 8192) return QG_ERR_UNSUPPORTED;
    if (n_rows == 0 || m == 0) return QG_OK;
    if (!w_qs || !w_d || !xq || !xd || !y) return QG_ERR_NULL;
    if (!aligned(w_qs, 32) || !aligned(w_d, 2) || !aligned(xq, 16) || !aligned(xd, 2) || !aligned(y, 16))
        return QG_ERR_ALIGN;
    return from_cuda(qg::launch_prefill_mma(w_qs, w_d, n_rows, k, xq, xd, m, y, stream));
}

qg_status qg_ffn_up_q8_0(const float *x, const float *gamma, int64_t hidden, float eps, const int8_t *w_qs,
                         const uint16_t *w_d, int64_t ffn, float *h, int8_t *hq, uint16_t *hd, int8_t *xq_out,
                         uint16_t *xd_out, float *inv_rms_out, qg_stream_t stream)
{
    if (hidden <= 0 || hidden % 32 != 0 || ffn < 0 || ffn % 32 != 0 || ffn > kMaxRows / 2) return QG_ERR_SHAPE;
    if (hq && !aligned(hq, 32)) return QG_ERR_ALIGN;
    if (!(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (!qg::ffn_up_supported(hidden, ffn)) return QG_ERR_UNSUPPORTED;
    if (ffn == 0) return QG_OK;
    if (!x || !gamma || !w_qs || !w_d || !h || !hq || !hd) return QG_ERR_NULL;
    if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(w_qs, 32) || !aligned(w_d, 16) || !aligned(h, 16) ||
        !aligned(hq, 16) || !aligned(hd, 2) || !aligned(xq_out, 16) || !aligned(xd_out, 2) || !aligned(inv_rms_out, 4))
        return QG_ERR_ALIGN;
    return from_cuda(qg::launch_ffn_up(x, gamma, hidden, eps, w_qs, w_d, ffn, h, hq, hd, xq_out, xd_out, inv_rms_out,
                                       stream));
}

qg_status qg_decode_ffn_q8_0_out(const float *x_in, float *x_out, const float *gamma, int64_t hidden, int64_t ffn,
                                 float eps, const int8_t *wgu_qs, const uint16_t *wgu_d, const int8_t *wdn_qs,
                                 const uint16_t *wdn_d, float *h, int8_t *hq, uint16_t *hd, qg_stream_t stream)
{
    if (hidden <= 0 || hidden % 32 != 0 || ffn <= 0 || ffn % 32 != 0 || ffn > kMaxRows / 2 || ffn > kMaxK)
        return QG_ERR_SHAPE;
    if (!(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (!qg::ffn_up_supported(hidden, ffn)) return QG_ERR_UNSUPPORTED;
    if (!x_in || !x_out || !gamma || !wgu_qs || !wgu_d || !wdn_qs || !wdn_d || !h || !hq || !hd) return QG_ERR_NULL;
    if (!aligned(x_in, 16) || !aligned(x_out, 16) || !aligned(gamma, 16) || !aligned(wgu_qs, 32) ||
        !aligned(wgu_d, 16) || !aligned(wdn_qs, 32) || !aligned(wdn_d, 16) || !aligned(h, 16) || !aligned(hq, 32) ||
        !aligned(hd, 2))
        return QG_ERR_ALIGN;
    // in place, or apart: a partial overlap would let the down projection read
    // residual rows that another CTA has already overwritten
    const size_t xb = static_cast<size_t>(hidden) * sizeof(float);
    if (x_in != x_out && overlap(x_in, xb, x_out, xb)) return QG_ERR_SHAPE;
    qg_status st = from_cuda(qg::launch_ffn_up(x_in, gamma, hidden, eps, wgu_qs, wgu_d, ffn, h, hq, hd, nullptr,
                                               nullptr, nullptr, stream));
    if (st != QG_OK) return st;
    if (qg::prefetch_supported(hidden, ffn) && aligned(wdn_d, 16))
        return from_cuda(qg::launch_gemv_prefetch(wdn_qs, wdn_d, hidden, ffn, hq, hd, QG_EPI_RESIDUAL_ADD, x_in,
                                                  x_out, stream));
    return from_cuda(
        qg::launch_gemv_q8_0(wdn_qs, wdn_d, hidden, ffn, hq, hd, 1, QG_EPI_RESIDUAL_ADD, x_in, x_out, stream));
}

qg_status qg_decode_ffn_q8_0_rotated(const float *x_in, float *x_out, const float *gamma, int64_t hidden,
                                     int64_t ffn, float eps, const int8_t *wgu_qs, const uint16_t *wgu_d,
                                     const int8_t *wdn_qs, const uint16_t *wdn_d, float *h, int8_t *hq, uint16_t *hd,
                                     int8_t *xq_out, uint16_t *xd_out, qg_stream_t stream)
{
    if (hidden <= 0 || hidden % 32 != 0 || ffn <= 0 || ffn % 32 != 0 || ffn > kMaxRows / 2 || ffn > kMaxK)
        return QG_ERR_SHAPE;
    if (!(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (!qg::ffn_up_rotated_supported(hidden, ffn) || !qg::prefetch_supported(hidden, ffn)) return QG_ERR_UNSUPPORTED;
    if (!x_in || !x_out || !gamma || !wgu_qs || !wgu_d || !wdn_qs || !wdn_d || !h || !hq || !hd) return QG_ERR_NULL;
    if (!aligned(x_in, 16) || !aligned(x_out, 16) || !aligned(gamma, 16) || !aligned(wgu_qs, 32) ||
        !aligned(wgu_d, 16) || !aligned(wdn_qs, 32) || !aligned(wdn_d, 16) || !aligned(h, 16) || !aligned(hq, 32) ||
        !aligned(hd, 2) || !aligned(xq_out, 16) || !aligned(xd_out, 2))
        return QG_ERR_ALIGN;
    const size_t xb = static_cast<size_t>(hidden) * sizeof(float);
    if (x_in != x_out && overlap(x_in, xb, x_out, xb)) return QG_ERR_SHAPE;
    qg_status st = from_cuda(qg::launch_ffn_up_rotated(x_in, gamma, hidden, eps, wgu_qs, wgu_d, ffn, h, hq, hd, xq_out,
                                                       xd_out, stream));
    if (st != QG_OK) return st;
    return from_cuda(
        qg::launch_gemv_prefetch(wdn_qs, wdn_d, hidden, ffn, hq, hd, QG_EPI_RESIDUAL_ADD, x_in, x_out, stream));
}

qg_status qg_decode_ffn_q8_0(float *x, const float *gamma, int64_t hidden, int64_t ffn, float eps,
                             const int8_t *wgu_qs, const uint16_t *wgu_d, const int8_t *wdn_qs,
                             const uint16_t *wdn_d, float *h, int8_t *hq, uint16_t *hd, qg_stream_t stream)
{
    return qg_decode_ffn_q8_0_out(x, x, gamma, hidden, ffn, eps, wgu_qs, wgu_d, wdn_qs, wdn_d, h, hq, hd, stream);
}

static bool layer_shape_ok(int64_t hidden, int64_t ffn)
{
    return hidden > 0 && hidden % 32 == 0 && ffn > 0 && ffn % 32 == 0 && ffn <= kMaxRows / 2 && ffn <= kMaxK;
}

int32_t qg_decode_layer_partials(int64_t hidden, int64_t ffn)
{
    if (!layer_shape_ok(hidden, ffn) || !qg::decode_layer_supported(hidden, ffn)) return -1;
    return qg::decode_layer_partials(ffn);
}

qg_status qg_decode_layer_q8_0(const float *r_in, const float *p_in, int32_t n_in, float *r_out, float *p_out,
                               const float *gamma, int64_t hidden, int64_t ffn, float eps, const int8_t *wgu_qs,
                               const uint16_t *wgu_d, const int8_t *wdn_qs, const uint16_t *wdn_d, float *h,
                               int8_t *hq, uint16_t *hd, qg_stream_t stream)
{
    if (!layer_shape_ok(hidden, ffn)) return QG_ERR_SHAPE;
    if (!(eps >= 0.0f) || n_in < 0 || n_in > qg::kMaxLayerPartials) return QG_ERR_SHAPE;
    if (!qg::decode_layer_supported(hidden, ffn)) return QG_ERR_UNSUPPORTED;
    if (!r_in || (n_in > 0 && !p_in) || !r_out || !p_out || !gamma || !wgu_qs || !wgu_d || !wdn_qs || !wdn_d || !h ||
        !hq || !hd)
        return QG_ERR_NULL;
    if (!aligned(r_in, 16) || !aligned(p_in, 16) || !aligned(r_out, 16) || !aligned(p_out, 16) ||
        !aligned(gamma, 16) || !aligned(wgu_qs, 32) || !aligned(wgu_d, 16) || !aligned(wdn_qs, 32) ||
        !aligned(wdn_d, 16) || !aligned(h, 16) || !aligned(hq, 32) || !aligned(hd, 2))
        return QG_ERR_ALIGN;
    const size_t xb = static_cast<size_t>(hidden) * 4;
    const size_t pin_b = xb * static_cast<size_t>(n_in);
    const size_t pout_b = xb * static_cast<size_t>(qg::decode_layer_partials(ffn));
    // the outputs are written while every CTA still reads the inputs
    if (overlap(r_out, xb, r_in, xb) || overlap(p_out, pout_b, r_in, xb) || overlap(r_out, xb, p_in, pin_b) ||
        overlap(p_out, pout_b, p_in, pin_b) || overlap(r_out, xb, p_out, pout_b))
        return QG_ERR_SHAPE;
    return from_cuda(qg::launch_decode_layer(r_in, p_in, n_in, r_out, p_out, gamma, hidden, eps, wgu_qs, wgu_d, wdn_qs,
                                             wdn_d, ffn, h, hq, hd, stream));
}

qg_status qg_decode_layer_finish(const float *r, const float *p, int32_t n, int64_t hidden, float *x,
                                 qg_stream_t stream)
{
    if (hidden < 0 || hidden > kMaxK || n < 0 || n > qg::kMaxLayerPartials) return QG_ERR_SHAPE;
    if (hidden == 0) return QG_OK;
    if (!r || (n > 0 && !p) || !x) return QG_ERR_NULL;
    if (!aligned(r, 4) || !aligned(p, 4) || !aligned(x, 4)) return QG_ERR_ALIGN;
    return from_cuda(qg::launch_layer_finish(r, p, n, hidden, x, stream));
}

qg_status qg_copy_stalls(uint32_t *count, int32_t clear)
{
    if (!count) return QG_ERR_NULL;
    return from_cuda(qg::copy_stalls(count, clear != 0));
}

qg_status qg_decode_layers_q8_0_noalloc(const float *x_in, float *x_out, int32_t n_layers, const float *const *gamma,
                                       const int8_t *const *wgu_qs, const uint16_t *const *wgu_d,
                                       const int8_t *const *wdn_qs, const uint16_t *const *wdn_d, int64_t hidden,
                                       int64_t ffn, float eps, qg_stream_t stream)
{
    if (!layer_shape_ok(hidden, ffn) || n_layers < 0 || n_layers > 65536 || !(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (!qg::decode_layer_supported(hidden, ffn)) return QG_ERR_UNSUPPORTED;
    if (qg::layer_scratch_bytes(hidden, ffn, qg::decode_layer_partials(ffn)) > qg::layer_scratch_capacity())
        return QG_ERR_UNSUPPORTED;  // the fixed scratch array is too small for this shape
    if (!x_in || !x_out) return QG_ERR_NULL;
    if (n_layers > 0 && (!gamma || !wgu_qs || !wgu_d || !wdn_qs || !wdn_d)) return QG_ERR_NULL;
    if (!aligned(x_in, 16) || !aligned(x_out, 4)) return QG_ERR_ALIGN;
    for (int32_t l = 0; l < n_layers; ++l) {
        if (!gamma[l] || !wgu_qs[l] || !wgu_d[l] || !wdn_qs[l] || !wdn_d[l]) return QG_ERR_NULL;
        if (!aligned(gamma[l], 16) || !aligned(wgu_qs[l], 32) || !aligned(wgu_d[l], 16) || !aligned(wdn_qs[l], 32) ||
            !aligned(wdn_d[l], 16))
            return QG_ERR_ALIGN;
    }
    return from_cuda(qg::launch_decode_layers_noalloc(x_in, x_out, n_layers, gamma, wgu_qs, wgu_d, wdn_qs, wdn_d,
                                                      hidden, ffn, eps, stream));
}

int64_t qg_decode_stack_workspace_bytes(int64_t hidden, int64_t ffn)
{
    if (!layer_shape_ok(hidden, ffn) || !qg::stack_shape(hidden, ffn, nullptr)) return -1;
    return static_cast<int64_t>(qg::stack_workspace_bytes(hidden, ffn));
}

int32_t qg_decode_stack_max_layers(void) { return qg::stack_max_layers(); }

qg_status qg_decode_stack_q8_0(const float *x_in, float *x_out, int32_t n_layers, const float *const *gamma,
                               const int8_t *const *wgu_qs, const uint16_t *const *wgu_d,
                               const int8_t *const *wdn_qs, const uint16_t *const *wdn_d, int64_t hidden,
                               int64_t ffn, float eps, void *workspace, float *h_last, int8_t *hq_last,
                               uint16_t *hd_last, int64_t wait_limit_ns, qg_stream_t stream)
{
    if (!layer_shape_ok(hidden, ffn) || n_layers < 1 || n_layers > qg::stack_max_layers() || !(eps >= 0.0f) ||
        wait_limit_ns < 0)
        return QG_ERR_SHAPE;
    if (!qg::stack_shape(hidden, ffn, nullptr)) return QG_ERR_UNSUPPORTED;
    if (!x_in || !x_out || !workspace || !gamma || !wgu_qs || !wgu_d || !wdn_qs || !wdn_d) return QG_ERR_NULL;
    if (!aligned(x_in, 16) || !aligned(x_out, 4) || !aligned(workspace, 256) || !aligned(h_last, 4) ||
        !aligned(hd_last, 2))
        return QG_ERR_ALIGN;
    for (int32_t l = 0; l < n_layers; ++l) {
        if (!gamma[l] || !wgu_qs[l] || !wgu_d[l] || !wdn_qs[l] || !wdn_d[l]) return QG_ERR_NULL;
        if (!aligned(gamma[l], 16) || !aligned(wgu_qs[l], 32) || !aligned(wgu_d[l], 16) || !aligned(wdn_qs[l], 32) ||
            !aligned(wdn_d[l], 16))
            return QG_ERR_ALIGN;
    }
    const size_t xb = static_cast<size_t>(hidden) * 4, wb = qg::stack_workspace_bytes(hidden, ffn);
    // in place or apart (each down row reads its residual before it writes the
    // row); nothing may overlap the workspace, which every CTA reads and writes
    if (x_in != x_out && overlap(x_in, xb, x_out, xb)) return QG_ERR_SHAPE;
    if (overlap(x_in, xb, workspace, wb) || overlap(x_out, xb, workspace, wb)) return QG_ERR_SHAPE;
    const size_t fb = static_cast<size_t>(ffn);
    if ((h_last && overlap(h_last, fb * 4, workspace, wb)) || (hq_last && overlap(hq_last, fb, workspace, wb)) ||
        (hd_last && overlap(hd_last, fb / 16, workspace, wb)))
        return QG_ERR_SHAPE;
    const uint64_t limit = wait_limit_ns == 0 ? qg::kCopyWaitLimitNs : static_cast<uint64_t>(wait_limit_ns);
    return from_cuda(qg::launch_decode_stack(x_in, x_out, n_layers, gamma, wgu_qs, wgu_d, wdn_qs, wdn_d, hidden, ffn,
                                             eps, workspace, h_last, hq_last, hd_last, limit, stream));
}

qg_status qgemm_q8_0_prefill_tc(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k, const void *xt,
                                int64_t m, float *y, int32_t tile_n, qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows || n_rows > UINT32_MAX / 2) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (!act_tiles_shape_ok(m, k)) return QG_ERR_SHAPE;
    if (!qg::prefill_tc_supported(k)) return QG_ERR_UNSUPPORTED;
    if (tile_n != 0 && tile_n != 64 && tile_n != 96 && tile_n != 128) return QG_ERR_UNSUPPORTED;
    if (n_rows == 0 || m == 0) return QG_OK;
    if (!w_qs || !w_d || !xt || !y) return QG_ERR_NULL;
    if (!aligned(w_qs, 32) || !aligned(w_d, 16) || !aligned(xt, 16) || !aligned(y, 16)) return QG_ERR_ALIGN;
    return from_cuda(qg::launch_prefill_tc(w_qs, w_d, n_rows, k, xt, m, y, tile_n, stream));
}

qg_status qgemm_bf16_prefill(const uint16_t *w, int64_t n_rows, int64_t k, const uint16_t *x, int64_t m,
                             const uint16_t *gamma, float eps, int epilogue, uint16_t *xhat, float *y,
                             qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows || n_rows > INT32_MAX) return QG_ERR_SHAPE;
    if (m < 0 || m > (int64_t(1) << 24)) return QG_ERR_SHAPE;
    if (k <= 0 || k > 16384 || !qg::prefill_bf16_supported(k)) return QG_ERR_SHAPE;
    if (!(eps >= 0.0f)) return QG_ERR_SHAPE;
    if (epilogue != QG_EPI_NONE && epilogue != QG_EPI_SILU_MUL_HALVES) return QG_ERR_UNSUPPORTED;
    if (epilogue == QG_EPI_SILU_MUL_HALVES && (n_rows % 2) != 0) return QG_ERR_SHAPE;
    if (n_rows == 0 || m == 0) return QG_OK;
    if (!w || !x || !y || (gamma && !xhat)) return QG_ERR_NULL;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(gamma, 16) || !aligned(xhat, 16) || !aligned(y, 16))
        return QG_ERR_ALIGN;
    // outputs (y, and xhat when written) must not overlap the inputs or each other
    const size_t xb = static_cast<size_t>(m) * k * 2, wb = static_cast<size_t>(n_rows) * k * 2;
    const size_t yb = static_cast<size_t>(m) * (epilogue == QG_EPI_SILU_MUL_HALVES ? n_rows / 2 : n_rows) * 4;
    if (overlap(y, yb, x, xb) || overlap(y, yb, w, wb) || (gamma && overlap(y, yb, gamma, static_cast<size_t>(k) * 2)))
        return QG_ERR_SHAPE;
    if (gamma && (overlap(xhat, xb, x, xb) || overlap(xhat, xb, w, wb) || overlap(xhat, xb, y, yb) ||
                  overlap(xhat, xb, gamma, static_cast<size_t>(k) * 2)))
        return QG_ERR_SHAPE;
    return from_cuda(qg::launch_prefill_bf16(w, n_rows, k, x, m, gamma, eps, epilogue, xhat, y, stream));
}

int64_t qg_scales_ld(int64_t rows) { return rows < 0 ? -1 : (rows + 3) & ~int64_t(3); }

qg_status qg_q8_0_pack_f16(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k, uint16_t *codes,
                           float *scales_t, qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (n_rows == 0) return QG_OK;
    if (!w_qs || !w_d || !codes || !scales_t) return QG_ERR_NULL;
    if (!aligned(w_qs, 8) || !aligned(w_d, 2) || !aligned(codes, 16) || !aligned(scales_t, 4)) return QG_ERR_ALIGN;
    const size_t nq = static_cast<size_t>(n_rows) * k, nd = static_cast<size_t>(n_rows) * (k / 32);
    const size_t ns = static_cast<size_t>(qg_scales_ld(n_rows)) * (k / 32);
    if (overlap(codes, nq * 2, w_qs, nq) || overlap(codes, nq * 2, w_d, nd * 2) || overlap(scales_t, ns * 4, w_qs, nq) ||
        overlap(scales_t, ns * 4, w_d, nd * 2) || overlap(codes, nq * 2, scales_t, ns * 4))
        return QG_ERR_SHAPE;
    return from_cuda(qg::launch_pack_q8_0_f16(w_qs, w_d, n_rows, k, codes, scales_t, stream));
}

qg_status quantize_act_q8_0_f16(const float *x, int64_t rows, int64_t k, uint16_t *codes, float *scales_t,
                                qg_stream_t stream)
{
    if (rows < 0 || rows > (int64_t(1) << 24)) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (rows == 0) return QG_OK;
    if (!x || !codes || !scales_t) return QG_ERR_NULL;
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales_t, 4)) return QG_ERR_ALIGN;
    const size_t n = static_cast<size_t>(rows) * k, ns = static_cast<size_t>(qg_scales_ld(rows)) * (k / 32);
    if (overlap(codes, n * 2, x, n * 4) || overlap(scales_t, ns * 4, x, n * 4) || overlap(codes, n * 2, scales_t, ns * 4))
        return QG_ERR_SHAPE;
    return from_cuda(qg::launch_quantize_act_f16(x, rows, k, codes, scales_t, stream));
}

qg_status qgemm_q8_0_prefill_tc2(const uint16_t *w_codes, const float *w_scales_t, int64_t n_rows, int64_t k,
                                 const uint16_t *x_codes, const float *x_scales_t, int64_t m, float *y, int32_t tile_n,
                                 qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows || n_rows > INT32_MAX) return QG_ERR_SHAPE;
    if (m < 0 || m > (int64_t(1) << 24)) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (tile_n != 0 && tile_n != 128 && tile_n != 192) return QG_ERR_UNSUPPORTED;
    if (n_rows == 0 || m == 0) return QG_OK;
    if (!w_codes || !w_scales_t || !x_codes || !x_scales_t || !y) return QG_ERR_NULL;
    if (!aligned(w_codes, 16) || !aligned(w_scales_t, 16) || !aligned(x_codes, 16) || !aligned(x_scales_t, 16) ||
        !aligned(y, 16))
        return QG_ERR_ALIGN;
    const size_t yb = static_cast<size_t>(m) * n_rows * 4;
    if (overlap(y, yb, w_codes, static_cast<size_t>(n_rows) * k * 2) ||
        overlap(y, yb, w_scales_t, static_cast<size_t>(qg_scales_ld(n_rows)) * (k / 32) * 4) ||
        overlap(y, yb, x_codes, static_cast<size_t>(m) * k * 2) ||
        overlap(y, yb, x_scales_t, static_cast<size_t>(qg_scales_ld(m)) * (k / 32) * 4))
        return QG_ERR_SHAPE;
    return from_cuda(
        qg::launch_prefill_tc2(w_codes, w_scales_t, n_rows, k, x_codes, x_scales_t, m, y, tile_n, stream));
}

qg_status qg_measure_mma_s8(int64_t iters, int32_t *sink, int64_t *ops, qg_stream_t stream)
{
    if (iters < 1 || iters > (int64_t(1) << 24)) return QG_ERR_SHAPE;
    if (!sink || !ops) return QG_ERR_NULL;
    return from_cuda(qg::launch_mma_s8_rate(iters, sink, ops, stream));
}

int32_t qg_measure_hbm_read_sink_len(void) { return qg::hbm_read_ctas(); }

qg_status qg_measure_hbm_read(const void *buf, int64_t bytes, uint32_t *sink, int32_t sink_len, qg_stream_t stream)
{
    if (bytes <= 0 || bytes % 32 != 0) return QG_ERR_SHAPE;
    if (!buf || !sink) return QG_ERR_NULL;
    if (!aligned(buf, 32) || !aligned(sink, 4)) return QG_ERR_ALIGN;
    if (sink_len < qg::hbm_read_ctas()) return QG_ERR_SHAPE;
    return from_cuda(qg::launch_hbm_read(buf, bytes, sink, stream));
}

qg_status qg_measure_launch_chain(int32_t n, int32_t grid, int32_t block, qg_stream_t stream)
{
    if (n < 0 || n > 65536 || grid < 1 || grid > 65535 || block < 1 || block > 1024 || block % 32 != 0)
        return QG_ERR_SHAPE;
    return from_cuda(qg::launch_empty_chain(n, grid, block, stream));
}

qg_status qg_debug_block_dots_q8_0(const int8_t *w_qs, int64_t n_rows, int64_t k, const int8_t *xq, int64_t batch,
                                   int32_t *s, qg_stream_t stream)
{
    if (n_rows < 0 || n_rows > kMaxRows) return QG_ERR_SHAPE;
    if (qg_status st = check_q8_k(k); st != QG_OK) return st;
    if (batch < 1 || batch > 8) return QG_ERR_SHAPE;
    if (n_rows == 0) return QG_OK;
    if (!w_qs || !xq || !s) return QG_ERR_NULL;
    if (!aligned(w_qs, 32) || !aligned(xq, 16) || !aligned(s, 4)) return QG_ERR_ALIGN;
    return from_cuda(qg::launch_block_dots(w_qs, n_rows, k, xq, batch, s, stream));
}

}  // extern "C"
