// A stack of one-launch decode layers for callers that cannot allocate device
// memory (or cannot pass work buffers through their own interface).
//
// qg_decode_layer_q8_0 keeps every intermediate of a layer in caller-owned
// buffers: the unreduced input and output (a base vector and one partial
// vector per thread-block cluster) and the layer's activation h with its Q8_0
// codes and scale.  Here those buffers live in one fixed device array,
// g_layer_scratch, compiled into the library: one copy per GPU, created when
// the library's code is loaded onto that GPU, never resized and never freed.
// The entry point looks its address up once per GPU (cudaGetSymbolAddress
// with that GPU current) and carves it into the buffers the layers need; a
// shape whose buffers do not fit is refused before anything is launched.
//
// Nothing in the array has to start at zero: layer 0 reads only x_in (no
// partials), every later layer reads buffers written by the layer before it,
// and the finish step reads only what the last layer wrote.
//
// Because there is one array per GPU, two calls on the same GPU must not run
// at the same time (issue them on one stream, or synchronise between them);
// calls on different GPUs are independent.  The address lookup happens on the
// first call on each GPU, so make that first call before capturing the entry
// point into a CUDA graph; later calls, captured or not, only launch kernels.
#include <mutex>

#include "qg_common.cuh"

namespace qg {

cudaError_t launch_decode_layer(const float *, const float *, int, float *, float *, const float *, int64_t, float,
                                const int8_t *, const uint16_t *, const int8_t *, const uint16_t *, int64_t, float *,
                                int8_t *, uint16_t *, cudaStream_t);
cudaError_t launch_layer_finish(const float *, const float *, int, int64_t, float *, cudaStream_t);
int decode_layer_partials(int64_t half);

// 256 KB: enough for every ffn the one-launch layer serves at hidden 1024 (up
// to 4096, i.e. 16 partial vectors from clusters of 8: 160,000 B; the 0.8B
// shape, hidden 1024 / ffn 3584, takes 141,056 B); the largest shapes it serves
// (hidden 1792 with 16 partials: 264,448 B) do not fit and are refused.
constexpr size_t kLayerScratchBytes = 256 * 1024;
static __device__ __align__(256) uint8_t g_layer_scratch[kLayerScratchBytes];

// Bytes of scratch a stack of layers of this shape needs (buffers 256-byte aligned).
size_t layer_scratch_bytes(int64_t hidden, int64_t ffn, int partials)
{
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t x = al(static_cast<size_t>(hidden) * 4);
    const size_t part = al(static_cast<size_t>(partials) * hidden * 4);
    return 2 * x + 2 * part + al(static_cast<size_t>(ffn) * 4) + al(static_cast<size_t>(ffn)) +
           al(static_cast<size_t>(ffn / 32) * 2);
}

size_t layer_scratch_capacity() { return kLayerScratchBytes; }

// Address of this GPU's copy of the array, looked up once per GPU with that GPU
// current.
static cudaError_t layer_scratch(uint8_t **out)
{
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaError_t e = cudaGetSymbolAddress(&p, g_layer_scratch); e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = static_cast<uint8_t *>(addr[dev]);
    return cudaSuccess;
}

cudaError_t launch_decode_layers_noalloc(const float *x_in, float *x_out, int n_layers, const float *const *gamma,
                                         const int8_t *const *wgu_qs, const uint16_t *const *wgu_d,
                                         const int8_t *const *wdn_qs, const uint16_t *const *wdn_d, int64_t hidden,
                                         int64_t ffn, float eps, cudaStream_t s)
{
    uint8_t *base = nullptr;
    if (cudaError_t e = layer_scratch(&base); e != cudaSuccess) return e;
    const int np = decode_layer_partials(ffn);
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t xb = al(static_cast<size_t>(hidden) * 4), pb = al(static_cast<size_t>(np) * hidden * 4);
    float *r[2] = {reinterpret_cast<float *>(base), reinterpret_cast<float *>(base + xb)};
    float *p[2] = {reinterpret_cast<float *>(base + 2 * xb), reinterpret_cast<float *>(base + 2 * xb + pb)};
    uint8_t *rest = base + 2 * xb + 2 * pb;
    float *h = reinterpret_cast<float *>(rest);
    int8_t *hq = reinterpret_cast<int8_t *>(rest + al(static_cast<size_t>(ffn) * 4));
    uint16_t *hd = reinterpret_cast<uint16_t *>(rest + al(static_cast<size_t>(ffn) * 4) + al(static_cast<size_t>(ffn)));
    // layer l reads (r, p)[l % 2] (layer 0 reads x_in alone) and writes (r, p)[(l + 1) % 2]
    for (int l = 0; l < n_layers; ++l) {
        const float *r_in = l == 0 ? x_in : r[l % 2];
        const float *p_in = l == 0 ? nullptr : p[l % 2];
        if (cudaError_t e = launch_decode_layer(r_in, p_in, l == 0 ? 0 : np, r[(l + 1) % 2], p[(l + 1) % 2], gamma[l],
                                                hidden, eps, wgu_qs[l], wgu_d[l], wdn_qs[l], wdn_d[l], ffn, h, hq, hd,
                                                s);
            e != cudaSuccess)
            return e;
    }
    if (n_layers == 0) return cudaMemcpyAsync(x_out, x_in, static_cast<size_t>(hidden) * 4, cudaMemcpyDeviceToDevice, s);
    return launch_layer_finish(r[n_layers % 2], p[n_layers % 2], np, hidden, x_out, s);
}

}  // namespace qg
