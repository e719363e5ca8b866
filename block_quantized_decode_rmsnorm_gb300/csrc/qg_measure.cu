// Measurement aids: the floors that the decode kernels are judged against.
//
// "One level down: #002 the same compiler on a GPU", Decode: memory decides:
// a decode matrix-vector product is judged against what a pure read of the
// same memory achieves on the same machine, not against the data sheet.  The
// read probe here streams a buffer once with the loads the GEMV kernels use
// (32-byte, not kept in L1) from every SM; the launch chain measures what a
// kernel boundary alone costs when kernels follow each other with programmatic
// dependent launch, the floor of a GEMV too small to be bound by its bytes.
#include "qg_common.cuh"

namespace qg {

// Every thread folds four 32-byte pieces per step (all four in flight) into an
// XOR; one word per CTA is written so the loads cannot be dropped.
__global__ void __launch_bounds__(512) hbm_read_kernel(const uint8_t *__restrict__ buf, int64_t n32,
                                                       uint32_t *__restrict__ sink)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint32_t acc = 0u;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n32; i += 4 * stride) {
        u32x8 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ld_stream_32B(buf + 32 * (i + u * stride));
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int w = 0; w < 8; ++w) acc ^= v[u].v[w];
    }
    for (; i < n32; i += stride) {
        const u32x8 v = ld_stream_32B(buf + 32 * i);
#pragma unroll
        for (int w = 0; w < 8; ++w) acc ^= v.v[w];
    }
    acc = __reduce_xor_sync(0xffffffffu, acc);
    __shared__ uint32_t s_acc[16];
    if ((threadIdx.x & 31) == 0) s_acc[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t a = 0u;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) a ^= s_acc[w];
        sink[blockIdx.x] = a;
    }
}

int hbm_read_ctas() { return 4 * num_sms(); }

cudaError_t launch_hbm_read(const void *buf, int64_t bytes, uint32_t *sink, cudaStream_t s)
{
    hbm_read_kernel<<<hbm_read_ctas(), 512, 0, s>>>(static_cast<const uint8_t *>(buf), bytes / 32, sink);
    return cudaGetLastError();
}

// An empty kernel that waits for its predecessor and lets its successor launch,
// as every kernel of the library does.
__global__ void empty_pdl_kernel()
{
    pdl_wait();
    pdl_trigger();
}

cudaError_t launch_empty_chain(int n, int grid, int block, cudaStream_t s)
{
    for (int i = 0; i < n; ++i)
        if (cudaError_t e = launch_pdl(empty_pdl_kernel, dim3(grid), dim3(block), 0, s); e != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace qg
