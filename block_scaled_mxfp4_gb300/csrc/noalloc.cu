// mxfp4_gemm_noalloc: the GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// under an allocator they do not control (a framework's caching allocator
// they may not call into, a plugin host that forbids allocation after
// start-up), or code where a cudaMalloc would synchronise the device at the
// wrong time.  For them this entry point takes only inputs and outputs and
// keeps its scratch (relaid scales and split-K partial sums) in a fixed-size
// array that is part of the library image on the device.
//
// The array is MXFP4_NOALLOC_SCRATCH_BYTES bytes; every GPU that loads the
// library holds it until the process exits.  All calls share it, so calls
// whose work overlaps on the GPU (different streams, or different host
// threads on the same device) race on it and must be serialised by the
// caller.  Nothing carried over from the previous call needs clearing: each
// call writes its relaid scales and split-K partials before reading them, and
// the split-K tile counters carry a per-call tag, so a counter left behind by
// an earlier call reads as zero.
#include <mutex>

#include "../../include/mxfp4_gemm.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MXFP4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (the name is only a host-side stand-in for the array, so the
// address has to come from the runtime).  Returns nullptr on failure.
void *scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int mxfp4_gemm_noalloc(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A,
                                  int64_t lda, const void *B, int64_t ldb, const void *scaleA,
                                  int64_t ld_sa, const void *scaleB, int64_t ld_sb, float alpha,
                                  float beta, int M, int N, int K, int split_k, void *stream)
{
    mxfp4_plan plan;
    const int st = mxfp4_plan_gemm(M, N, K, split_k, 0, &plan);
    if (st != MXFP4_OK)
        return st;
    const size_t need = mxfp4_gemm_workspace_size(M, N, K, split_k);
    if (need > static_cast<size_t>(MXFP4_NOALLOC_SCRATCH_BYTES))
        return MXFP4_ERR_WORKSPACE;   // this shape needs more scratch than the fixed array
    // The array's address is per device: the stream must run on the device
    // whose copy is passed to the kernels.
    int cur = -1, sdev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess ||
        cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
        cudaGetLastError();
        return MXFP4_ERR_CUDA;
    }
    if (sdev != cur)
        return MXFP4_ERR_INVALID_ARG;
    void *scratch = scratch_on_current_device();
    if (!scratch)
        return MXFP4_ERR_CUDA;
    return mxfp4_gemm(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha, beta,
                      M, N, K, split_k, scratch, static_cast<size_t>(MXFP4_NOALLOC_SCRATCH_BYTES),
                      stream);
}
