// Measurement helper for the benchmark, not part of the GEMM library: one
// streaming read of a device buffer, the floor that a single pass over that
// many bytes reaches on this GPU (what the GEMM's bandwidth-bound shapes are
// compared with).  Every thread keeps eight independent 16-byte loads in
// flight; the words are folded into one value so the loads are not removed.
// mode 0: a plain launch.  mode 1: a programmatic dependent of the previous
// launch that lets the next one start at once and waits for the previous one
// before reading -- the launch form of mxfp4_gemm, so back-to-back reads over
// rotating buffers time the same way.  mode 2: as 1 without the wait, so the
// reads overlap the previous launch (as the weight prefetch of
// MXFP4_FLAG_B_STATIC does; valid here because nothing is written).
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__global__ void __launch_bounds__(256) stream_read_kernel(const uint4 *__restrict__ p, size_t n,
                                                          unsigned *__restrict__ sink, int wait)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (wait)
        asm volatile("griddepcontrol.wait;" ::: "memory");
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

}  // namespace

// Reads `bytes` (rounded down to a multiple of 16) of `src` (16-byte
// aligned) once from every SM; `sink` is a device word the kernel may write.
// Returns 0, -1 for bad arguments, or the CUDA error code of the launch.
extern "C" int mxfp4_probe_stream_read(const void *src, size_t bytes, void *sink, int mode,
                                       void *stream)
{
    if (!src || !sink || bytes < 16 || (reinterpret_cast<uintptr_t>(src) % 16) != 0)
        return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms * 4));
    cfg.blockDim = dim3(256);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = mode != 0 ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, stream_read_kernel, static_cast<const uint4 *>(src),
                                             bytes / 16, static_cast<unsigned *>(sink),
                                             mode == 2 ? 0 : 1);
    return e == cudaSuccess ? 0 : static_cast<int>(e);
}
