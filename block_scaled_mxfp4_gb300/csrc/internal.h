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

// Arguments of one GEMM launch.  "P" is the operand whose rows feed the MMA's
// M side (A, or B when swapped), "Q" the operand on the MMA's N side.
struct GemmArgs {
    const uint8_t *sfP;     // scales of P: relaid atoms, or row-major if sf_rowmajor
    const uint8_t *sfQ;     // scales of Q, same form
    int64_t sf_rb_stride;   // relaid: bytes per 128-row block of atoms
    int sf_rowmajor;        // 1: scales are row-major E8M0 [rows, ld] (atoms built in-kernel)
    int sf_vec8;            // row-major scales allow aligned 8-byte loads per stage
    int sf_async;           // row-major scales allow 4-byte cp.async (aligned rows)
    int sf_tma;             // row-major scales allow 2-D TMA (16-byte aligned rows)
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
    float *ws;              // fp32 partials [split_k][M][N] (split_k > 1)
    int vec_ok;             // D (and C) allow aligned 16-byte row accesses
    int vec32_ok;           // D allows aligned 32-byte row stores
    int stream_p;           // P is read once: hint L2 evict-first
    long long wait_limit;   // SM cycles before a wait gives up
    uint32_t idesc8;        // fp8: kind::mxf8f6f4 instruction descriptor (set at launch)
    int fmt_p, fmt_q;       // fp8: element types of P and Q (0 = E4M3, 1 = E5M2)
    int cluster_split;      // > 1: the split_k CTAs of a tile form one cluster and reduce
                            // their partials through distributed shared memory (no ws)
};

struct GemmShape {
    int tile_n;
    int stages;
    int swap;
    int persistent;         // 1: stream-K persistent kernel (gemm_mxf4_persistent)
    int nacc;               // persistent: TMEM accumulator buffers (1 or 2)
    int ctas_per_sm;        // resident CTAs per SM the plan assumed
    int pair;               // 1: CTA-pair kernel (256 x 256 tiles, cta_group::2)
    int pair_ctas;          // pair kernel: grid size (upper bound; 2 x pairs)
    int pair_cluster;       // pair kernel: pairs per cluster (1 or 2)
    int pair_kc;            // pair kernel: 256-K chunks per pipeline stage (1 or 2)
    int gemv;               // 1: GEMV kernel for M <= 2 (gemv.cu)
    int fp8;                // 1: 8-bit elements (one-tile kernel, kind::mxf8f6f4)
    int split_cluster;      // 1: split-K reduced inside each tile's cluster (no partials)
};

// Work schedule of the persistent stream-K kernel.  Tile t (raster below)
// covers rows [128p, 128p+128) of P and [tile_n q, ...) of Q.  CTA c first
// takes whole tiles c, c+G, ... (dp_waves of them), then the K-stage units
// [c*S/G, (c+1)*S/G) of the remaining tiles (S = sk_units), in order.
struct Sched {
    int tiles_p, tiles_q;   // output tiles along P and Q
    int kt;                 // K stages per tile
    int ctas;               // G
    int dp_waves;           // whole tiles per CTA before the stream-K part
    int sk_tile0;           // first stream-K tile (= dp_waves * G)
    long long sk_units;     // (tiles - sk_tile0) * kt
    int group;              // raster: groups of `group` tile rows along P
    int *flags;             // [G] per-CTA partial-ready flags
    float *partials;        // [G][pcols][128] fp32 partial tiles
    int pcols;              // columns per partial slot: tile_n, or Q's rows if fewer
    int epoch;              // this call's flag value (never 0)
};

// Every workspace layout starts with this many bytes reserved for the
// stream-K flags (nothing else is ever written there), so flags left by one
// call can only hold an earlier call's epoch.
constexpr size_t kFlagBytes = 4096;
constexpr int kMaxPersistentCtas = static_cast<int>(kFlagBytes / sizeof(int));

// Dynamic shared memory one GEMM configuration needs (0 if unsupported).
size_t gemm_smem_bytes(const GemmShape &s);

// Whether (tile_n, stages, swap) is one of the compiled configurations.
bool gemm_config_exists(const GemmShape &s);

cudaError_t launch_gemm(const GemmArgs &a, const CUtensorMap &tmP, const CUtensorMap &tmQ,
                        const GemmShape &s, dim3 grid, cudaStream_t stream);

cudaError_t launch_gemm_persistent(const GemmArgs &a, const Sched &sched, const CUtensorMap &tmP,
                                   const CUtensorMap &tmQ, const CUtensorMap &tmSP,
                                   const CUtensorMap &tmSQ, const GemmShape &s,
                                   cudaStream_t stream);

// CTA-pair kernel (relaid scales): grid of up to `ctas` CTAs in clusters of
// cluster_pairs pairs (clamped to the clusters the GPU holds at once), tiles
// of 256 x tile_n (256: one accumulator, 1 or 2 pairs per cluster, stages
// of 256 or 512 K; 192: two accumulators, 1 pair, 256-K stages).  after_relayout: launched right after this
// library's scale relayout on the same stream (programmatic dependent launch;
// only the scale loads wait).
size_t gemm_pair_smem_bytes(int tile_n, int k_chunks);
cudaError_t launch_gemm_pair(const GemmArgs &a, int tile_n, int cluster_pairs, int k_chunks, int tiles_p,
                             int tiles_q, int ctas, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const CUtensorMap &tmSA, const CUtensorMap &tmSB, bool after_relayout,
                             cudaStream_t stream);

// Persistent configuration: dynamic smem (0 if not compiled) and resident
// CTAs per SM the occupancy calculator allows (0 on error).
size_t gemm_persistent_smem_bytes(const GemmShape &s);
int gemm_persistent_occupancy(const GemmShape &s);

// GEMV form for M <= 2 (gemv.cu).  Scales row-major ([rows, ld] bytes) or,
// with sf_relaid, the relaid atoms of mxfp4_scale_relayout.
struct GemvArgs {
    const uint8_t *A, *B, *SA, *SB;
    int64_t lda_bytes, ldb_bytes;   // row strides of the packed operands (bytes)
    int64_t ld_sa, ld_sb;           // row-major scales: row strides (bytes)
    int sf_relaid;
    int M, N, K;
    float alpha, beta;
    const uint16_t *C;
    int64_t ldc;
    uint16_t *D;
    int64_t ldd;
};
constexpr int kGemvMaxM = 2;
void gemv_launch_shape(int N, int sms, int *ctas, int *threads);
cudaError_t launch_gemv(const GemvArgs &g, int sms, cudaStream_t stream);

cudaError_t launch_scale_relayout(uint8_t *dst, const uint8_t *src, int rows, int K, int64_t ld,
                                  cudaStream_t stream);
// Both operands' scales (same K) in one launch.
cudaError_t launch_scale_relayout2(uint8_t *dst0, const uint8_t *src0, int rows0, int64_t ld0,
                                   uint8_t *dst1, const uint8_t *src1, int rows1, int64_t ld1,
                                   int K, cudaStream_t stream);

cudaError_t launch_splitk_reduce(const float *ws, int split, int M, int N, float alpha, float beta,
                                 const uint16_t *C, int64_t ldc, uint16_t *D, int64_t ldd,
                                 int sms, cudaStream_t stream);

cudaError_t launch_wait_probe(long long limit, cudaStream_t stream);

cudaError_t launch_stream_read(const void *src, size_t bytes, unsigned *sink, int sms,
                               cudaStream_t stream);

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
