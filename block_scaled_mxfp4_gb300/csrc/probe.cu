// Measurement hook: a plain streaming read of a device buffer, the floor a
// single pass over that many bytes reaches (what the GEMM's HBM-bound shapes
// are compared with).  Every thread keeps eight independent 16-byte loads in
// flight; the words are folded into one value so the loads are not removed.
#include "internal.h"

namespace mxfp4 {

__global__ void __launch_bounds__(256) stream_read_kernel(const uint4 *__restrict__ p, size_t n,
                                                          unsigned *__restrict__ sink)
{
    unsigned acc = 0;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += 8 * stride) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const size_t k = i + j * stride;
            if (k < n)
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v[j].x), "=r"(v[j].y), "=r"(v[j].z), "=r"(v[j].w)
                             : "l"(p + k));
            else
                v[j] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
    }
    if (acc == 0x9E3779B9u)   // practically never; keeps the loads live
        *sink = acc;
}

cudaError_t launch_stream_read(const void *src, size_t bytes, unsigned *sink, int sms,
                               cudaStream_t stream)
{
    const size_t n = bytes / 16;
    const int blocks = (sms > 0 ? sms : 152) * 4;
    stream_read_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(src), n, sink);
    return cudaGetLastError();
}

}  // namespace mxfp4
