// Scale-factor relayout kernel.
#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

// ------------------------------------------------------- scale relayout --
//
// Row-major E8M0 scales [rows, K/32] (one per 32 K elements; page "asm_f4gemm
// -- driving aiter's gfx950 MXFP4 GEMM code objects", section "Data layouts",
// "A_scale / B_scale", which also pads with 0x7F = 1.0) -> 512-byte atoms of
// 128 rows x 4 blocks.  Atom (rb, g) sits at (rb * groups + g) * 512; inside
// it, row 32j + i and block b sit at byte 16i + 4j + b, so that one 16-byte
// line holds rows i, i+32, i+64, i+96: the four 32-bit tensor-memory columns
// lane i of every lane group holds (column j <-> row 32j + i), which the
// GEMM's scale writers store with one tcgen05.st per lane.
//
// One CTA of 256 threads handles one 128-row block (of either operand when
// both are relaid in one launch) and up to kGroupsPerCta
// atoms along K: it reads the 128 x (4*kGroupsPerCta) scale bytes with
// consecutive threads on consecutive words of a row, stages them in shared
// memory (rows padded to an odd word count, so the column reads below hit 32
// different banks), and writes the atoms as 16-byte lines, consecutive
// threads on consecutive lines.
// NVFP4 scales (one UE4M3 byte per 16 K) take the same path with a block of
// 16 in place of 32: an atom then spans 64 K, and padding is 0x38 (UE4M3 1.0).
//
// 8 groups (32 scale bytes of each of 128 rows) per CTA: measured fastest for
// 8192 x 8192 scales (6.5 us for both operands, against 7.5 at 16, 10.8 at 32
// and 8.2 at 4 groups): enough CTAs to keep DRAM busy, 4 words per thread.
constexpr int kGroupsPerCta = 8;
constexpr int kRelayoutThreads = 256;

// One or two operands per launch: row blocks [0, rblocks0) of grid x belong to
// operand 0, the rest to operand 1 (both have the same K).
struct RelayoutJob {
    uint8_t *dst[2];
    const uint8_t *src[2];
    int rows[2];
    int64_t ld[2];
    int64_t rblocks0;
    int vec4[2];
    uint32_t pad;           // padding byte, replicated into the four bytes of a word
};

__global__ void __launch_bounds__(kRelayoutThreads)
    scale_relayout_kernel(const RelayoutJob job, int kblocks, int64_t groups)
{
    __shared__ uint32_t tile[128][kGroupsPerCta + 1];
    const int t = threadIdx.x;
    // Launched as a programmatic dependent of the preceding work on the
    // stream: the scales may be that work's output, so wait for it first.
    // Only then let the GEMM that follows launch: it reads A and B before its
    // own wait (on this grid), which is safe once the work before this grid
    // has finished.
    pdl_wait_prerequisites();
    if (t == 0)
        pdl_launch_dependents();
    const int op = static_cast<int64_t>(blockIdx.x) < job.rblocks0 ? 0 : 1;
    const int64_t rb = static_cast<int64_t>(blockIdx.x) - (op ? job.rblocks0 : 0);
    const uint8_t *src = job.src[op];
    const int rows = job.rows[op];
    const int64_t ld = job.ld[op];
    const int vec4 = job.vec4[op];
    const int64_t g0 = static_cast<int64_t>(blockIdx.y) * kGroupsPerCta;
    const int ng = static_cast<int>(groups - g0 < kGroupsPerCta ? groups - g0 : kGroupsPerCta);

    // All of a thread's loads are issued before any is stored, so each thread
    // keeps its 8 words in flight at once (the scales come cold from DRAM).
    constexpr int kPerThread = 128 * kGroupsPerCta / kRelayoutThreads;
    uint32_t words[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int e = t + k * kRelayoutThreads;
        const int r = e / kGroupsPerCta;
        const int w = e % kGroupsPerCta;
        const int64_t row = rb * 128 + r;
        const int64_t kb = (g0 + w) * 4;
        uint32_t word = job.pad;
        if (row < rows && w < ng) {
            const uint8_t *p = src + row * ld + kb;
            if (vec4 && kb + 4 <= kblocks) {
                word = __ldg(reinterpret_cast<const uint32_t *>(p));
            } else {
                word = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    word |= (kb + b < kblocks ? static_cast<uint32_t>(p[b]) : (job.pad & 0xFFu)) << (8 * b);
            }
        }
        words[k] = word;
    }
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int e = t + k * kRelayoutThreads;
        tile[e / kGroupsPerCta][e % kGroupsPerCta] = words[k];
    }
    __syncthreads();
    uint8_t *out = job.dst[op] + (rb * groups + g0) * kSfAtomBytes;
    for (int e = t; e < ng * 32; e += kRelayoutThreads) {
        const int atom = e / 32;
        const int i = e % 32;
        reinterpret_cast<uint4 *>(out + atom * kSfAtomBytes)[i] =
            make_uint4(tile[i][atom], tile[i + 32][atom], tile[i + 64][atom], tile[i + 96][atom]);
    }
}

// kblocks: scale bytes per row (K / 32, or K / 16 for NVFP4); groups: atoms
// per 128-row block.
static cudaError_t launch_relayout_job(RelayoutJob &job, int nops, int kblocks, int64_t groups,
                                       cudaStream_t stream)
{
    int64_t total = 0;
    for (int i = 0; i < nops; ++i) {
        job.vec4[i] = (reinterpret_cast<uintptr_t>(job.src[i]) % 4 == 0) && (job.ld[i] % 4 == 0);
        total += sf_row_blocks(job.rows[i]);
    }
    job.rblocks0 = sf_row_blocks(job.rows[0]);
    if (nops == 1) {
        job.dst[1] = job.dst[0];
        job.src[1] = job.src[0];
        job.rows[1] = job.rows[0];
        job.ld[1] = job.ld[0];
        job.vec4[1] = job.vec4[0];
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(total),
                       static_cast<unsigned>((groups + kGroupsPerCta - 1) / kGroupsPerCta));
    cfg.blockDim = dim3(kRelayoutThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scale_relayout_kernel, job, kblocks, groups);
}

cudaError_t launch_scale_relayout(uint8_t *dst, const uint8_t *src, int rows, int K, int64_t ld,
                                  cudaStream_t stream)
{
    RelayoutJob job{};
    job.dst[0] = dst;
    job.src[0] = src;
    job.rows[0] = rows;
    job.ld[0] = ld;
    job.pad = 0x7F7F7F7Fu;
    return launch_relayout_job(job, 1, K / 32, sf_groups(K), stream);
}

cudaError_t launch_scale_relayout2(uint8_t *dst0, const uint8_t *src0, int rows0, int64_t ld0,
                                   uint8_t *dst1, const uint8_t *src1, int rows1, int64_t ld1,
                                   int K, cudaStream_t stream)
{
    RelayoutJob job{};
    job.dst[0] = dst0;
    job.src[0] = src0;
    job.rows[0] = rows0;
    job.ld[0] = ld0;
    job.dst[1] = dst1;
    job.src[1] = src1;
    job.rows[1] = rows1;
    job.ld[1] = ld1;
    job.pad = 0x7F7F7F7Fu;
    return launch_relayout_job(job, 2, K / 32, sf_groups(K), stream);
}

cudaError_t launch_scale_relayout2_nv(uint8_t *dst0, const uint8_t *src0, int rows0, int64_t ld0,
                                      uint8_t *dst1, const uint8_t *src1, int rows1, int64_t ld1,
                                      int K, cudaStream_t stream)
{
    RelayoutJob job{};
    job.dst[0] = dst0;
    job.src[0] = src0;
    job.rows[0] = rows0;
    job.ld[0] = ld0;
    job.dst[1] = dst1;
    job.src[1] = src1;
    job.rows[1] = rows1;
    job.ld[1] = ld1;
    job.pad = 0x38383838u;
    return launch_relayout_job(job, 2, K / 16, sf_groups_nv(K), stream);
}

}  // namespace mxfp4
