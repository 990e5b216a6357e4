// Internal launchers shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxfp4 {

constexpr int kTileM = 128;        // MMA M (rows of the MMA-A operand per tile)
constexpr int kTileK = 256;        // K elements per pipeline stage = 128 bytes per row
constexpr int kSfAtomBytes = 512;  // 128 rows x 4 scale blocks of the tcgen05 layout
constexpr int kSfRowBlock = 128;

// Relaid scale buffer geometry (see mxfp4_scale_relayout): 128-row blocks
// (the count rounded up to an even number so a 256-row tile never reads past
// the end) times 2*ceil(K/256) atoms of 512 bytes.
__host__ __device__ inline int64_t sf_groups(int K) { return 2 * ((static_cast<int64_t>(K) + kTileK - 1) / kTileK); }
__host__ __device__ inline int64_t sf_row_blocks(int rows) { return 2 * ((static_cast<int64_t>(rows) + 255) / 256); }
inline size_t sf_relaid_bytes(int rows, int K)
{
    return static_cast<size_t>(sf_row_blocks(rows) * sf_groups(K) * kSfAtomBytes);
}
// NVFP4 (one UE4M3 scale per 16 K): the same atoms, each holding 4 blocks of
// 16 (64 K), four per 256-K stage.
__host__ __device__ inline int64_t sf_groups_nv(int K) { return 4 * ((static_cast<int64_t>(K) + kTileK - 1) / kTileK); }
inline size_t sf_relaid_bytes_nv(int rows, int K)
{
    return static_cast<size_t>(sf_row_blocks(rows) * sf_groups_nv(K) * kSfAtomBytes);
}

// Arguments of one GEMM launch.  "P" is the operand whose rows feed the MMA's
// M side (A, or B when swapped), "Q" the operand on the MMA's N side.
struct GemmArgs {
    const uint8_t *sfP;     // scales of P: relaid atoms, or row-major if sf_rowmajor
    const uint8_t *sfQ;     // scales of Q, same form
    int64_t sf_rb_stride;   // relaid: bytes per 128-row block of atoms
    int sf_rowmajor;        // 1: scales are row-major E8M0 [rows, ld] (atoms built in-kernel)
    int sf_vec8;            // row-major scales allow aligned 8-byte loads per stage
    int sf_async;           // row-major scales allow 4-byte cp.async (aligned rows)
    int sf_tma;             // row-major scales come by 2-D TMA (16-byte aligned rows)
    int q_box_rows;         // rows of a Q tile copied per stage (Q's rows rounded up to 8,
                            // at most tile_n; rows past them are never stored)
    int64_t ldsP, ldsQ;     // row-major: row strides in bytes
    int rowsP, rowsQ;       // rows of P and Q
    int M, N, K;
    int kt_total;           // stages of 128 bytes per row: ceil(K / 256) fp4, ceil(K / 128) fp8
    int kt_per_split;
    int split_k;
    float alpha, beta;
    const uint16_t *C;      // bf16 bits
    int64_t ldc;
    uint16_t *D;            // bf16 bits
    int64_t ldd;
    // Split-K (split_k > 1): each CTA parks its fp32 partial tile in slot
    // (tile, z) of `partials` (128 rows x part_cols floats, row-major by tile
    // row); the CTA that completes a tile's count sums the slots in z order.
    float *partials;
    unsigned long long *tile_count;   // [tiles]: (epoch << 32) | CTAs of the tile done
    int part_cols;          // columns per partial row: min(tile_n, rows of Q)
    uint32_t epoch;         // this call's counter tag (never 0)
    int cluster_reduce;     // 1: the split_k CTAs of a tile form one thread-block
                            // cluster and sum their partials through distributed
                            // shared memory (no partials, counters or workspace)
    int vec_ok;             // D (and C) allow aligned 16-byte row accesses
    int vec32_ok;           // D allows aligned 32-byte row stores
    int stream_p;           // P is read once: hint L2 evict-first
    int p_is_b;             // P holds B's rows (swap-AB)
    int b_early;            // B and its scales may be read before the preceding grid ends
    int ab_early;           // pair kernel: A and B may be read before the preceding grid
                            // ends (it is this library's relayout, which waited first)
    long long wait_limit;   // SM cycles before a wait gives up
    uint32_t idesc8;        // fp8: kind::mxf8f6f4 instruction descriptor (set at launch)
    int fmt_p, fmt_q;       // fp8: element types of P and Q (kind::mxf8f6f4 codes)
};

struct GemmShape {
    int tile_n;
    int stages;
    int swap;
    int ctas_per_sm;        // resident CTAs per SM the plan assumed
    int pair;               // 1: CTA-pair kernel (256 x 256 tiles, cta_group::2)
    int pair_ctas;          // pair kernel: grid size (upper bound; 2 x pairs)
    int fp8;                // 1: 8-bit elements (one-tile kernel, kind::mxf8f6f4)
    int nv;                 // 1: NVFP4 (kind::mxf4nvf4, UE4M3 per 16 K; one-tile: swap-AB
                            //    with row-major scales by TMA only)
};

// Dynamic shared memory one GEMM configuration needs (0 if unsupported).
size_t gemm_smem_bytes(const GemmShape &s);

// Whether (tile_n, stages, swap) is one of the compiled configurations.
bool gemm_config_exists(const GemmShape &s);

// One-tile kernel, launched as a programmatic dependent of the preceding work
// on `stream`: it waits in-kernel for that work before touching memory the
// work may write (everything but B and its scales when a.b_early).
// tmSP / tmSQ: row-major scale maps (used when a.sf_tma).
cudaError_t launch_gemm(const GemmArgs &a, const CUtensorMap &tmP, const CUtensorMap &tmQ,
                        const CUtensorMap &tmSP, const CUtensorMap &tmSQ, const GemmShape &s,
                        dim3 grid, cudaStream_t stream);

// CTA-pair kernel (relaid scales): grid of up to `ctas` CTAs in clusters of
// two (clamped to the clusters the GPU holds at once), persistent over 256 x
// 256 tiles, launched as a programmatic dependent of the preceding work.
// a.ab_early: that work is this library's scale relayout, so only the scale
// loads and the epilogue wait for it.
size_t gemm_pair_smem_bytes();
// nv: NVFP4 operands (UE4M3 scales per 16 K, relaid with sf_groups_nv).
cudaError_t launch_gemm_pair(const GemmArgs &a, int tiles_p, int tiles_q, int ctas,
                             const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const CUtensorMap &tmSA, const CUtensorMap &tmSB, bool nv,
                             cudaStream_t stream);

cudaError_t launch_scale_relayout(uint8_t *dst, const uint8_t *src, int rows, int K, int64_t ld,
                                  cudaStream_t stream);
// Both operands' scales (same K) in one launch, as a programmatic dependent
// of the preceding work on the stream (it waits for that work before reading).
cudaError_t launch_scale_relayout2(uint8_t *dst0, const uint8_t *src0, int rows0, int64_t ld0,
                                   uint8_t *dst1, const uint8_t *src1, int rows1, int64_t ld1,
                                   int K, cudaStream_t stream);

// NVFP4 scales: row-major UE4M3 [rows, ld] (one per 16 K) -> atoms of
// 128 rows x 4 blocks of 16, sf_groups_nv(K) per 128-row block, padded with
// 0x38 (UE4M3 1.0; the E8M0 pad 0x7F would be NaN here).
cudaError_t launch_scale_relayout2_nv(uint8_t *dst0, const uint8_t *src0, int rows0, int64_t ld0,
                                      uint8_t *dst1, const uint8_t *src1, int rows1, int64_t ld1,
                                      int K, cudaStream_t stream);

cudaError_t launch_wait_probe(long long limit, cudaStream_t stream);

// MXFP4 quantiser (quantize.cu): X bf16 [rows, ldx] -> Q [rows, ldq_bytes],
// S [rows, lds]; K % 32 == 0, X rows and Q rows 16-byte aligned.
// MXFP8 quantiser: bf16 [rows, K] -> codes [rows, ldq bytes] (fmt 0 E4M3,
// 1 E5M2) + E8M0 scales.
cudaError_t launch_quantize8(uint8_t *Q, int64_t ldq, uint8_t *S, int64_t lds, const uint16_t *X,
                             int64_t ldx, int rows, int K, int fmt, int sms, cudaStream_t stream);
cudaError_t launch_quantize(uint8_t *Q, int64_t ldq_bytes, uint8_t *S, int64_t lds,
                            const uint16_t *X, int64_t ldx, int rows, int K, int sms,
                            cudaStream_t stream);

cudaError_t read_device_status(int *status, int reset);

}  // namespace mxfp4
