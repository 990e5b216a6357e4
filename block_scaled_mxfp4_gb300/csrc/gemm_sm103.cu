// Block-scaled MXFP4 GEMM on sm_103a tensor cores (tcgen05 kind::mxf4).
//
//   D[M,N] = alpha * A[M,K] . B[N,K]^T + beta * C[M,N]          (page "asm_f4gemm
//   -- driving aiter's gfx950 MXFP4 GEMM code objects", formula and section
//   "Data layouts"; each E8M0 scale multiplies its 32 inputs before they are
//   accumulated, page "CDNA4 dense MFMA builtins", section "Mixed-precision
//   with scaling").
//
// One CTA computes one 128 x BN output tile over a range of K (a split):
//   producers  per 256-K stage, one 128x128-byte tile of P and one Q tile
//           (128-byte swizzle) into an S-stage shared-memory ring guarded by
//           full/empty mbarriers.  Scales come one of three ways: relaid
//           atoms by 1-D bulk copy (warps 4, 6, 7 issue P, Q and the atoms);
//           row-major scales by 2-D TMA as the aligned 16-byte window of
//           each row that holds the stage's bytes (warp 4 issues P and P's
//           window, warp 6 Q and Q's); or, when the scale rows are not
//           16-byte aligned, gathered by warp 4 with cp.async or plain loads.
//           Each issuing thread waits out its own copy instructions (a few
//           hundred cycles apiece), hence one thread per copy stream;
//   warps 0-3  scale writers during the main loop: each lane takes its line
//           of the stage's scales from shared memory and writes it with
//           tcgen05.st into its own TMEM lane (warp w owns lanes 32w..32w+31,
//           so the four warps lay down the four replicas), then the warp
//           arrives on the stage's sf_full barrier;
//   warp 5  allocates tensor memory; one thread waits for a stage's scales
//           (whose barrier the scale writers complete only after the stage's
//           operands landed) and issues four block-scaled MMAs into an fp32
//           TMEM accumulator, then commits the stage back to the producers;
//   warps 0-3  then the epilogue: tcgen05.ld the accumulator (warp w owns TMEM
//           lanes 32w..32w+31 = tile rows), apply alpha/beta with C, round to
//           bf16 and store.  With split-K the splits of a tile sum their fp32
//           partials in split order 0, 1, ... inside the launch: up to 8
//           splits form one thread-block cluster and reduce over distributed
//           shared memory; more park their partials in the workspace and the
//           CTA that completes the tile's epoch-tagged counter reduces them.
//           Either way the result does not depend on which split finished
//           last, and alpha/beta and the bf16 rounding come once, at the end.
// The kernel is launched as a programmatic dependent of the preceding work on
// the stream: it starts while that work drains and waits for it in-kernel
// (griddepcontrol.wait) before the first read of A, C or the scales and
// before any write.  With b_early, the thread that loads B's tiles and B's
// scales starts filling the ring without that wait: callers whose weights the
// preceding work does not write let the weight stream of one GEMM start
// before the kernel ahead of it has finished.
// With swap (skinny M), P = B and Q = A, so the tile holds D^T: TMEM lane = n,
// column = m, and a warp's 32 lanes write 32 consecutive n of one row of D.
//
// Scale-factor placement in TMEM (one 32-bit column word per lane holds the
// scales of 4 consecutive 32-K blocks; lane i, column c <-> row 32c + i of a
// 128-row block, replicated in the four lane groups).  A K=64 instruction uses
// two consecutive bytes of those words, chosen by the scale-factor id (0 or 2).
// Every stage has its own TMEM scale slot.  A slot is rewritten only after the
// stage's full barrier completed again, which needs the producers to have
// seen the stage's previous MMAs commit, so no write overtakes a read.
#include <atomic>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

__device__ int g_device_status = 0;

// G = scale words (4 scale bytes each) per row and stage of 128 bytes per
// row: 2 for fp4 elements with E8M0 per 32 (256 K per stage), 1 for 8-bit
// elements (128 K per stage), 4 for NVFP4 (UE4M3 per 16, 256 K per stage).
// RAW_ONLY: scales only ever come as row-major 16-byte windows (the shared
// memory of a stage is sized for those, not for relaid atoms).
template <int BN, int STAGES, int G = 2, bool RAW_ONLY = false>
struct Cfg {
    static constexpr int BM = kTileM;
    static constexpr int BN_COLS = BN;
    static constexpr int STAGE_COUNT = STAGES;
    static constexpr int GROUPS = G;
    static constexpr int P_BYTES = BM * 128;
    static constexpr int Q_BYTES = BN * 128;
    static constexpr int NQ = BN >= 128 ? BN / 128 : 1;      // 128-row scale blocks of Q
    static constexpr int SFP_BYTES = G * kSfAtomBytes;       // G atoms per stage
    static constexpr int SFQ_BYTES = NQ * G * kSfAtomBytes;
    // Row-major scales copied by TMA: 16 bytes of each row (the aligned
    // 16-byte window holding the stage's 4G scale bytes).
    static constexpr int SFRP_BYTES = BM * 16;
    static constexpr int SFRQ_BYTES = BN * 16;
    static constexpr bool RAW = RAW_ONLY;
    static constexpr int SF_AREA = (!RAW_ONLY && (SFP_BYTES + SFQ_BYTES) > (SFRP_BYTES + SFRQ_BYTES))
                                       ? (SFP_BYTES + SFQ_BYTES) : (SFRP_BYTES + SFRQ_BYTES);
    // Stages start on 1024-byte boundaries (128-byte swizzle atoms).
    static constexpr int STAGE_BYTES = (P_BYTES + Q_BYTES + SF_AREA + 1023) / 1024 * 1024;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static constexpr int SF_COLS_P = 4 * G;                  // G groups x 4 columns
    static constexpr int SF_COLS_Q = 4 * G * NQ;
    static constexpr int SF_COLS = SF_COLS_P + SF_COLS_Q;
    static constexpr int TMEM_USED = BN + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static_assert(TMEM_USED <= 512, "tensor memory budget");
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile N");
    static_assert(G == 1 || G == 2 || G == 4, "scale words per stage");
};

// The configuration of element format FMT (0 MXFP4, 1 byte formats, 2 NVFP4).
template <int BN, int STAGES, int FMT>
using CfgFor = Cfg<BN, STAGES, FMT == 0 ? 2 : FMT == 1 ? 1 : 4, FMT == 2>;

constexpr int kGemmThreadsC = 256;     // threads of the one-tile kernel

// Row stride (floats) of a partial parked in shared memory for the cluster
// reduction: the columns rounded up to 4, plus 4 against bank conflicts.
__host__ __device__ inline int cluster_part_stride(int part_cols) { return (part_cols + 3) / 4 * 4 + 4; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// D[m][n0 .. n0+31] = bf16(alpha * v + beta * C), vector stores when the
// whole chunk is inside the row and the pointers allow it.
__device__ __forceinline__ void store_d_row(const GemmArgs &a, int m, int n0, float (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] *= a.alpha;
    const bool full = n0 + 32 <= a.N;
    if (a.beta != 0.0f) {
        const uint16_t *c = a.C + static_cast<int64_t>(m) * a.ldc + n0;
        if (a.vec_ok && full) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                uint4 w = *reinterpret_cast<const uint4 *>(c + i);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[i + 2 * j] = fmaf(a.beta, bf16_bits_to_float(ww[j] & 0xFFFF), v[i + 2 * j]);
                    v[i + 2 * j + 1] = fmaf(a.beta, bf16_bits_to_float(ww[j] >> 16), v[i + 2 * j + 1]);
                }
            }
        } else {
            for (int i = 0; i < 32 && n0 + i < a.N; ++i)
                v[i] = fmaf(a.beta, bf16_bits_to_float(c[i]), v[i]);
        }
    }
    uint16_t *d = a.D + static_cast<int64_t>(m) * a.ldd + n0;
    if (a.vec32_ok && full) {
        // 32-byte stores: half the store instructions of 16-byte ones.  D is
        // written once and not read back: evict-first, so it does not push
        // the operand panels that other tiles still load out of L2.
        const uint64_t pol = l2_policy_evict_first();
#pragma unroll
        for (int i = 0; i < 32; i += 16)
            st_global_v8_hint(d + i, pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                              pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]),
                              pack_bf16x2(v[i + 8], v[i + 9]), pack_bf16x2(v[i + 10], v[i + 11]),
                              pack_bf16x2(v[i + 12], v[i + 13]), pack_bf16x2(v[i + 14], v[i + 15]),
                              pol);
    } else if (a.vec_ok && full) {
#pragma unroll
        for (int i = 0; i < 32; i += 8)
            *reinterpret_cast<uint4 *>(d + i) =
                make_uint4(pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                           pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]));
    } else {
        for (int i = 0; i < 32 && n0 + i < a.N; ++i) {
            __nv_bfloat16 b = __float2bfloat16_rn(v[i]);
            d[i] = *reinterpret_cast<uint16_t *>(&b);
        }
    }
}

// D[m0 + i][n] = bf16(alpha * v[i] + beta * C) for the valid i (swap: one n
// per lane, consecutive across the warp).  All of C is loaded before the
// first store: C may alias D, so a load after a store could not be issued
// early, and 32 dependent DRAM round trips would follow.
__device__ __forceinline__ void store_d_col(const GemmArgs &a, int m0, int n, const float (&v)[32])
{
    if (n >= a.N)
        return;
    const int mcount = min(32, a.M - m0);
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        x[i] = a.alpha * v[i];
    if (a.beta != 0.0f) {
        uint16_t c[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            c[i] = i < mcount ? a.C[(static_cast<int64_t>(m0) + i) * a.ldc + n] : uint16_t(0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            x[i] = fmaf(a.beta, bf16_bits_to_float(c[i]), x[i]);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (i < mcount) {
            __nv_bfloat16 b = __float2bfloat16_rn(x[i]);
            a.D[(static_cast<int64_t>(m0) + i) * a.ldd + n] = *reinterpret_cast<uint16_t *>(&b);
        }
    }
}

// One-tile kernel epilogue of one 32-column chunk of one row (no swap): r[i]
// is the fp32 accumulator of D[m][n0 + i].
__device__ __forceinline__ void store_row_chunk(const GemmArgs &a, int m, int n0, const uint32_t (&r)[32])
{
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
    store_d_row(a, m, n0, v);
}

// Same with swap: r[i] is the accumulator of D[m0 + i][n].
__device__ __forceinline__ void store_col_chunk(const GemmArgs &a, int m0, int n, const uint32_t (&r)[32])
{
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
    store_d_col(a, m0, n, v);
}

// Split-K: slot (tile, z) of the partials holds the tile's fp32 partial as
// chunks of 4 columns, rows contiguous inside a chunk: value (row r, column
// c) at float ((c / 4) * 128 + r) * 4 + c % 4.  A warp (32 consecutive rows)
// then stores or loads one chunk as 512 contiguous bytes.
__device__ __forceinline__ float *partial_slot(const GemmArgs &a, int64_t tile, int z)
{
    return a.partials + (tile * a.split_k + z) * static_cast<int64_t>(kTileM * 4 * ((a.part_cols + 3) / 4));
}

// Row `row` of this CTA's partial, accumulator columns [c0, c0 + 32) (the
// chunks below part_cols).
__device__ __forceinline__ void park_partial_chunk(const GemmArgs &a, float *slot, int row, int c0,
                                                   const uint32_t (&r)[32])
{
    const int nch = (a.part_cols + 3) / 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int ch = c0 / 4 + i;
        if (ch < nch)
            __stcg(reinterpret_cast<float4 *>(slot + (static_cast<int64_t>(ch) * kTileM + row) * 4),
                   make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                               __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
    }
}

// Count this CTA into its tile and report whether it completed the count.
// The word holds (epoch << 32) | done; a word tagged with another call's
// epoch (never written, or left by a call that stopped on a timeout) counts
// as zero, so the workspace needs no clearing.  The CTA that completes the
// count resets the word to 0, so a replay of a captured call, which repeats
// the tag, starts from zero too.  Lock-free: each failed exchange means
// another CTA of the tile got its increment in.
__device__ __forceinline__ bool tile_count_done(unsigned long long *word, uint32_t epoch, int split)
{
    unsigned long long cur = atomicAdd(word, 0ull);
    for (;;) {
        const unsigned long long next = (static_cast<uint32_t>(cur >> 32) == epoch)
                                            ? cur + 1ull
                                            : ((static_cast<unsigned long long>(epoch) << 32) | 1ull);
        const unsigned long long prev = atomicCAS(word, cur, next);
        if (prev == cur)
            return static_cast<int>(next & 0xFFFFFFFFull) == split;
        cur = prev;
    }
}

// The CTA that completed a tile's count: thread t sums row (t & 127), one
// half of the columns (t >> 7), over the tile's split partials in the fixed
// order z = 0, 1, ..., split-1, then applies alpha / beta with C and rounds
// once to bf16 (swap: the row is n, the columns are m).
template <bool SWAP>
__device__ __forceinline__ void reduce_tile(const GemmArgs &a, int64_t tile, int p0, int q0, int t)
{
    const int row = t & (kTileM - 1);
    const int prows = SWAP ? a.N : a.M;
    if (p0 + row >= prows)
        return;
    const int qvalid = min(a.part_cols, (SWAP ? a.M : a.N) - q0);
    // Halves on 32-column boundaries: a chunk's stores (bounded by M and N
    // only) never reach the other half's columns.
    const int half = ((a.part_cols + 63) / 64) * 32;
    const int c_begin = (t >> 7) * half;
    const int c_end = min(qvalid, c_begin + half);
    const int64_t zstride = static_cast<int64_t>(kTileM) * 4 * ((a.part_cols + 3) / 4);
    const float *base = partial_slot(a, tile, 0) + static_cast<int64_t>(row) * 4;
    for (int cg = c_begin; cg < c_end; cg += 32) {
        const int cn = min(32, c_end - cg);
        const int nv = (cn + 3) / 4;                 // 4-column chunks of this group
        float acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            acc[i] = 0.0f;
        // Two splits' loads in flight per step; each column adds its splits
        // in the order z = 0, 1, ..., split-1.
        for (int z = 0; z < a.split_k; z += 2) {
            const bool two = z + 1 < a.split_k;
            const float *s0 = base + z * zstride + static_cast<int64_t>(cg / 4) * kTileM * 4;
            const float *s1 = s0 + zstride;
            float4 x[8], y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = i < nv ? __ldcg(reinterpret_cast<const float4 *>(s0 + i * kTileM * 4))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                y[i] = (two && i < nv) ? __ldcg(reinterpret_cast<const float4 *>(s1 + i * kTileM * 4))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[4 * i] += x[i].x;
                acc[4 * i + 1] += x[i].y;
                acc[4 * i + 2] += x[i].z;
                acc[4 * i + 3] += x[i].w;
            }
            if (two) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[4 * i] += y[i].x;
                    acc[4 * i + 1] += y[i].y;
                    acc[4 * i + 2] += y[i].z;
                    acc[4 * i + 3] += y[i].w;
                }
            }
        }
        if (!SWAP)
            store_d_row(a, p0 + row, q0 + cg, acc);
        else
            store_d_col(a, q0 + cg, p0 + row, acc);
    }
}

// Split-K inside a cluster: every CTA of the tile has parked its fp32
// partial in its own shared memory (row r at float r * stride, columns
// contiguous), and cluster rank z holds split z.  Rank r sums the rows
// [r * R, (r + 1) * R), R = ceil(128 / split), over ranks 0, 1, ..., split-1
// in that order, four columns per item, then applies alpha / beta with C
// and rounds once (swap: the rows are n, the columns m).  Consecutive
// threads take consecutive 4-column chunks of a row, so a warp reads whole
// runs of each peer's partial row (distributed shared memory serves scattered
// 16-byte reads of many rows far more slowly).
template <bool SWAP>
__device__ __forceinline__ void reduce_tile_cluster(const GemmArgs &a, uint32_t part_smem, int stride,
                                                    int p0, int q0, int t)
{
    const int S = a.split_k;
    const int rank = static_cast<int>(cluster_ctarank());
    const int R = (kTileM + S - 1) / S;
    const int r0 = rank * R;
    const int prows = SWAP ? a.N : a.M;
    const int nrows = max(0, min(min(kTileM, r0 + R), prows - p0) - r0);
    const int qvalid = min(a.part_cols, (SWAP ? a.M : a.N) - q0);
    const int nch = (qvalid + 3) / 4;
    const int items = nrows * nch;
    // Two items per thread per step: all their shared-memory and C loads are
    // in flight before either is summed.
    for (int base = t; base < items; base += 2 * kGemmThreadsC) {
        float4 v[2][8];
        uint16_t c[2][4];
        int64_t m[2][4], n[2][4];
        int cnt[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int it = base + u * kGemmThreadsC;
            cnt[u] = 0;
            if (it >= items)
                continue;
            const int k = it / nch;
            const int ch = it % nch;
            const int row = r0 + k;
            cnt[u] = min(4, qvalid - 4 * ch);
            const uint32_t off = part_smem + static_cast<uint32_t>((row * stride + 4 * ch) * 4);
#pragma unroll
            for (int z = 0; z < 8; ++z)
                if (z < S)
                    v[u][z] = ld_dsmem_v4(map_to_rank(off, static_cast<uint32_t>(z)));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                m[u][j] = SWAP ? q0 + 4 * ch + j : p0 + row;
                n[u][j] = SWAP ? p0 + row : q0 + 4 * ch + j;
                c[u][j] = (a.beta != 0.0f && j < cnt[u]) ? a.C[m[u][j] * a.ldc + n[u][j]] : uint16_t(0);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (cnt[u] == 0)
                continue;
            float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
            for (int z = 0; z < 8; ++z) {
                if (z < S) {
                    x0 += v[u][z].x;
                    x1 += v[u][z].y;
                    x2 += v[u][z].z;
                    x3 += v[u][z].w;
                }
            }
            const float xs[4] = {x0, x1, x2, x3};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < cnt[u]) {
                    float y = a.alpha * xs[j];
                    if (a.beta != 0.0f)
                        y = fmaf(a.beta, bf16_bits_to_float(c[u][j]), y);
                    __nv_bfloat16 b = __float2bfloat16_rn(y);
                    a.D[m[u][j] * a.ldd + n[u][j]] = *reinterpret_cast<uint16_t *>(&b);
                }
            }
        }
    }
}

// Bring the lines of C that this CTA's share of the cluster reduction reads
// into L2 (called while the CTA waits for its peers).
template <bool SWAP>
__device__ __forceinline__ void prefetch_c_share(const GemmArgs &a, int p0, int q0, int t)
{
    const int S = a.split_k;
    const int R = (kTileM + S - 1) / S;
    const int r0 = static_cast<int>(cluster_ctarank()) * R;
    const int prows = SWAP ? a.N : a.M;
    const int nrows = max(0, min(min(kTileM, r0 + R), prows - p0) - r0);
    const int qvalid = min(a.part_cols, (SWAP ? a.M : a.N) - q0);
    if (nrows <= 0 || qvalid <= 0)
        return;
    if (SWAP) {
        // Row m of C: n = p0 + r0 .. + nrows (2 bytes each).
        for (int i = t; i < qvalid; i += kGemmThreadsC) {
            const uint16_t *row = a.C + static_cast<int64_t>(q0 + i) * a.ldc + p0 + r0;
            prefetch_l2(row);
            prefetch_l2(row + nrows - 1);
        }
    } else {
        for (int i = t; i < nrows; i += kGemmThreadsC) {
            const uint16_t *row = a.C + static_cast<int64_t>(p0 + r0 + i) * a.ldc + q0;
            for (int c = 0; c < qvalid; c += 64)
                prefetch_l2(row + c);
            prefetch_l2(row + qvalid - 1);
        }
    }
}

// Row-major scales -> one lane's share of a 128-row block for stage kt: rows
// row0 + lane + 32j (j = 0..3), K blocks 4G kt .. 4G kt + 4G - 1 as G 4-byte
// words (byte b of word g = block 4G kt + 4g + b).  Missing rows / blocks
// read 0x7F.
template <int G>
__device__ __forceinline__ void load_sf_rows(const uint8_t *S, int64_t ld, int rows, int kblocks,
                                             int row0, int kt, int vec8, int lane,
                                             uint32_t (&w)[4][G])
{
    const int kb0 = kt * 4 * G;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = row0 + lane + 32 * j;
        if (r < rows) {
            const uint8_t *p = S + static_cast<int64_t>(r) * ld + kb0;
            if (vec8 && kb0 + 4 * G <= kblocks) {
                if constexpr (G == 2) {
                    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
                    w[j][0] = v.x;
                    w[j][1] = v.y;
                } else {
                    w[j][0] = __ldg(reinterpret_cast<const uint32_t *>(p));
                }
            } else {
                uint32_t x[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    x[g] = 0u;
#pragma unroll
                for (int b = 0; b < 4 * G; ++b) {
                    const uint32_t v = (kb0 + b < kblocks) ? static_cast<uint32_t>(p[b]) : 0x7Fu;
                    x[b >> 2] |= v << (8 * (b & 3));
                }
#pragma unroll
                for (int g = 0; g < G; ++g)
                    w[j][g] = x[g];
            }
        } else {
#pragma unroll
            for (int g = 0; g < G; ++g)
                w[j][g] = 0x7F7F7F7Fu;
        }
    }
}

// Asynchronous form of load_sf_rows + store_sf_lines: each 4-byte scale word
// goes straight from global memory to its place in the atom (row lane + 32j,
// word g -> atom g, line lane, word j).  Missing rows / blocks are zero-filled
// (their operand data is zero-filled by TMA too, so the product is 0).
template <int G = 2>
__device__ __forceinline__ void copy_sf_rows_async(uint8_t *atoms, const uint8_t *S, int64_t ld,
                                                   int rows, int kblocks, int row0, int kt,
                                                   int lane)
{
    const int kb0 = kt * 4 * G;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = row0 + lane + 32 * j;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int have = kblocks - (kb0 + 4 * g);
            const uint32_t bytes = (r < rows && have > 0) ? static_cast<uint32_t>(min(have, 4)) : 0u;
            const uint8_t *src = bytes ? S + static_cast<int64_t>(r) * ld + kb0 + 4 * g : S;
            cp_async_4(atoms + g * kSfAtomBytes + 16 * lane + 4 * j, src, bytes);
        }
    }
}

// Line `lane` of the G atoms of a stage: 16 bytes = rows lane, lane+32,
// lane+64, lane+96, four K blocks each.
template <int G>
__device__ __forceinline__ void store_sf_lines(uint8_t *atoms, const uint32_t (&w)[4][G], int lane)
{
#pragma unroll
    for (int g = 0; g < G; ++g)
        *reinterpret_cast<uint4 *>(atoms + g * kSfAtomBytes + 16 * lane) =
            make_uint4(w[0][g], w[1][g], w[2][g], w[3][g]);
}

// Scale writers (warps 0-3): for each stage of the ring, once its copies have
// landed, lane i of warp w reads line i of the stage's atoms (16 bytes = rows
// i, i+32, i+64, i+96 of a 128-row block, four K blocks each) and writes it to
// TMEM lane 32w + i of the stage's scale slot: P's two atoms to columns
// [0, 8), Q's atoms (K group g, row block r) to columns 8 + (g*NQ + r)*4.
// t_lane = TMEM base address with this warp's lane quarter in its lane field.
// raw: the stage holds row-major scales (16 bytes per row, the stage's 4G
// bytes at offset (4G kt) % 16 of each row, P's 128 rows then Q's BN rows),
// gathered here into the same lines.
template <class Cf>
__device__ __forceinline__ void write_stage_scales(uint8_t *smem, uint64_t *full, uint64_t *sf_full,
                                                   uint32_t t_lane, int nkt, int kt0, bool raw,
                                                   int lane, volatile int *abort_flag,
                                                   long long limit)
{
    constexpr int STAGES = Cf::STAGE_COUNT;
    const uint32_t t_sf = t_lane + Cf::BN_COLS;
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < nkt; ++i) {
        bool ok = mbar_wait(&full[stage], phase, abort_flag, limit, &g_device_status);
        if (!__all_sync(0xffffffffu, ok))
            return;
        constexpr int G = Cf::GROUPS;
        const uint8_t *sf_s = smem + stage * Cf::STAGE_BYTES + Cf::P_BYTES + Cf::Q_BYTES;
        uint32_t wp[4 * G];
        uint32_t wq[4 * G * Cf::NQ];
        if (raw) {
            const int off = ((kt0 + i) * 4 * G) & 15;
            const uint8_t *rp = sf_s + off;
            const uint8_t *rq = sf_s + Cf::SFRP_BYTES + off;
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    wp[4 * g + j] = *reinterpret_cast<const uint32_t *>(rp + (lane + 32 * j) * 16 + 4 * g);
#pragma unroll
                for (int r = 0; r < Cf::NQ; ++r)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = 128 * r + 32 * j + lane;
                        wq[(g * Cf::NQ + r) * 4 + j] =
                            row < Cf::BN_COLS ? *reinterpret_cast<const uint32_t *>(rq + row * 16 + 4 * g) : 0u;
                    }
            }
        } else if constexpr (!Cf::RAW) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 v = *reinterpret_cast<const uint4 *>(sf_s + g * kSfAtomBytes + 16 * lane);
            wp[4 * g] = v.x;
            wp[4 * g + 1] = v.y;
            wp[4 * g + 2] = v.z;
            wp[4 * g + 3] = v.w;
#pragma unroll
            for (int r = 0; r < Cf::NQ; ++r) {
                const uint4 u = *reinterpret_cast<const uint4 *>(
                    sf_s + Cf::SFP_BYTES + r * G * kSfAtomBytes + g * kSfAtomBytes + 16 * lane);
                const int o = (g * Cf::NQ + r) * 4;
                wq[o] = u.x;
                wq[o + 1] = u.y;
                wq[o + 2] = u.z;
                wq[o + 3] = u.w;
            }
        }
        }
        const uint32_t slot = t_sf + stage * Cf::SF_COLS;
        if constexpr (G == 4)
            tmem_st_32x32b_x16(slot, wp);
        else if constexpr (G == 2)
            tmem_st_32x32b_x8(slot, wp);
        else
            tmem_st_32x32b_x4(slot, wp);
        if constexpr (4 * G * Cf::NQ == 32)
            tmem_st_32x32b_x32(slot + Cf::SF_COLS_P, wq);
        else if constexpr (4 * G * Cf::NQ == 16)
            tmem_st_32x32b_x16(slot + Cf::SF_COLS_P, wq);
        else if constexpr (4 * G * Cf::NQ == 8)
            tmem_st_32x32b_x8(slot + Cf::SF_COLS_P, wq);
        else
            tmem_st_32x32b_x4(slot + Cf::SF_COLS_P, wq);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sf_full[stage]);
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

constexpr int kGemmThreads = kGemmThreadsC;

// FMT 0: fp4 (E2M1) elements, kind::mxf4; FMT 1: one byte per element
// (E4M3 / E5M2 / padded E2M3, E3M2, E2M1), kind::mxf8f6f4 with the element
// types in a.idesc8.  MINB: CTAs per SM the configuration is planned for.
template <int BN, int STAGES, bool SWAP, int FMT, int MINB>
__global__ void __launch_bounds__(kGemmThreads, MINB)
    gemm_mxf4_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap tmP,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmSP,
                     const __grid_constant__ CUtensorMap tmSQ)
{
    using Cf = CfgFor<BN, STAGES, FMT>;
    constexpr int G = Cf::GROUPS;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment of the ring (128-byte swizzle atoms).
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cf::STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *sf_full = empty + STAGES;
    uint64_t *acc_full = sf_full + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Tile of this CTA.  Launch order runs x fastest; consecutive CTAs walk a
    // band of up to 8 tile columns (Q) before the next tile row (P), so the
    // CTAs resident at once share a few P and Q panels in L2 instead of
    // sweeping all of P for every column.
    const int tp = static_cast<int>(gridDim.x), tq = static_cast<int>(gridDim.y);
    int pt, qt;
    {
        const int lin = static_cast<int>(blockIdx.y) * tp + static_cast<int>(blockIdx.x);
        const int band = tq < 8 ? tq : 8;
        const int b = lin / (band * tp);
        const int within = lin - b * band * tp;
        const int bw = min(band, tq - b * band);
        pt = within / bw;
        qt = b * band + within % bw;
    }
    const int64_t tile = static_cast<int64_t>(pt) * tq + qt;
    const int p0 = pt * kTileM;
    const int q0 = qt * BN;
    const int z = blockIdx.z;
    const int kt0 = z * a.kt_per_split;
    const int nkt = min(a.kt_per_split, a.kt_total - kt0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], !a.sf_rowmajor ? 3 : a.sf_tma ? 2 : a.sf_async ? 33 : 2);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 4);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, Cf::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tensormap(&tmP);
        prefetch_tensormap(&tmQ);
        if (a.sf_tma) {
            prefetch_tensormap(&tmSP);
            prefetch_tensormap(&tmSQ);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The next kernel on the stream may launch now; it waits in-kernel for
    // this grid before it touches anything this grid writes.
    if (threadIdx.x == 0)
        pdl_launch_dependents();

    if (warp == 4 || warp >= 6) {
        // ------------------------------------------------------ producer --
        // Loads may read the preceding work's output, so they wait for it --
        // except, with b_early, those of the thread that loads only B and its
        // scales (P with swap, else Q): the caller guarantees the preceding
        // work does not write them.
        const bool b_role = a.b_early && (a.sf_tma || !a.sf_rowmajor) &&
                            warp == (a.p_is_b ? 4 : 6);
        if (!b_role)
            pdl_wait_prerequisites();
        if (a.sf_rowmajor && a.sf_tma && nkt > 0) {
            // Two issuing threads: warp 4 the P tile and P's row-major scales,
            // warp 6 the Q tile (a.q_box_rows rows) and Q's; each scale box
            // is the aligned 16-byte window of 128 (or q_box_rows) rows that
            // holds the stage's 4G bytes.  Each thread arrives on the stage's
            // full barrier with its bytes.
            if (lane == 0 && (warp == 4 || warp == 6)) {
                const bool is_p = warp == 4;
                const uint64_t pol = (is_p && a.stream_p) ? l2_policy_evict_first() : l2_policy_evict_last();
                const uint32_t bytes = is_p ? static_cast<uint32_t>(Cf::P_BYTES + Cf::SFRP_BYTES)
                                            : static_cast<uint32_t>(a.q_box_rows * (128 + 16));
                int stage = 0;
                uint32_t phase = 0;
                int issued = 0;
                for (int i = 0; i < nkt; ++i) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_limit,
                                   &g_device_status))
                        break;
                    uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                    const int kt = kt0 + i;
                    const int sx = (kt * 4 * G) & ~15;
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    if (is_p) {
                        tma_load_2d(st, &tmP, &full[stage], kt * 128, p0, pol);
                        tma_load_2d(st + Cf::P_BYTES + Cf::Q_BYTES, &tmSP, &full[stage], sx, p0, pol);
                    } else {
                        tma_load_2d(st + Cf::P_BYTES, &tmQ, &full[stage], kt * 128, q0, pol);
                        tma_load_2d(st + Cf::P_BYTES + Cf::Q_BYTES + Cf::SFRP_BYTES, &tmSQ, &full[stage],
                                    sx, q0, pol);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (*abort_flag) {
                    for (int i = max(0, issued - STAGES); i < issued; ++i)
                        mbar_wait_drain(&full[i % STAGES], (i / STAGES) & 1u, a.wait_limit);
                }
            }
        } else if constexpr (FMT != 2) {
        // (NVFP4 takes row-major scales by TMA only; these paths are not built for it.)
        if (a.sf_rowmajor && a.sf_async && nkt > 0 && warp == 4) {
            // Whole warp: lane 0 issues the operand TMAs; every lane copies its
            // lines of the stage's scale atoms with 4-byte cp.async straight
            // from the row-major scales, and the stage's full barrier counts
            // one arrival per lane once that lane's copies have landed.
            const uint64_t pol_p = a.stream_p ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_last();
            const int kblocks = a.K / 32;
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int i = 0; i < nkt; ++i) {
                const bool ok =
                    mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_limit, &g_device_status);
                if (!__all_sync(0xffffffffu, ok))
                    break;
                uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                const int kt = kt0 + i;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[stage], Cf::P_BYTES + a.q_box_rows * 128);
                    tma_load_2d(st, &tmP, &full[stage], kt * 128, p0, pol_p);
                    tma_load_2d(st + Cf::P_BYTES, &tmQ, &full[stage], kt * 128, q0, pol_q);
                }
                uint8_t *sf_s = st + Cf::P_BYTES + Cf::Q_BYTES;
                copy_sf_rows_async<G>(sf_s, a.sfP, a.ldsP, a.rowsP, kblocks, p0, kt, lane);
#pragma unroll
                for (int r = 0; r < Cf::NQ; ++r)
                    copy_sf_rows_async<G>(sf_s + Cf::SFP_BYTES + r * G * kSfAtomBytes, a.sfQ, a.ldsQ,
                                          a.rowsQ, kblocks, q0 + r * kSfRowBlock, kt, lane);
                cp_async_mbar_arrive(&full[stage]);
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (lane == 0 && *abort_flag) {
                for (int i = max(0, issued - STAGES); i < issued; ++i)
                    mbar_wait_drain(&full[i % STAGES], (i / STAGES) & 1u, a.wait_limit);
            }
        } else if (a.sf_rowmajor && nkt > 0 && warp == 4) {
            // Whole warp: lane 0 issues the operand TMAs; every lane builds its
            // lines of the stage's scale atoms from row-major scales it loaded
            // one stage ahead (so the global loads overlap the ring wait).
            const uint64_t pol_p = a.stream_p ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_last();
            const int kblocks = a.K / 32;
            uint32_t wp[4][G];
            uint32_t wq[Cf::NQ][4][G];
            auto load_sf = [&](int kt) {
                load_sf_rows(a.sfP, a.ldsP, a.rowsP, kblocks, p0, kt, a.sf_vec8, lane, wp);
#pragma unroll
                for (int r = 0; r < Cf::NQ; ++r)
                    load_sf_rows(a.sfQ, a.ldsQ, a.rowsQ, kblocks, q0 + r * kSfRowBlock, kt,
                                 a.sf_vec8, lane, wq[r]);
            };
            load_sf(kt0);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int i = 0; i < nkt; ++i) {
                const bool ok =
                    mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_limit, &g_device_status);
                if (!__all_sync(0xffffffffu, ok))
                    break;
                uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                const int kt = kt0 + i;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[stage], Cf::P_BYTES + a.q_box_rows * 128);
                    tma_load_2d(st, &tmP, &full[stage], kt * 128, p0, pol_p);
                    tma_load_2d(st + Cf::P_BYTES, &tmQ, &full[stage], kt * 128, q0, pol_q);
                }
                uint8_t *sf_s = st + Cf::P_BYTES + Cf::Q_BYTES;
                store_sf_lines(sf_s, wp, lane);
#pragma unroll
                for (int r = 0; r < Cf::NQ; ++r)
                    store_sf_lines(sf_s + Cf::SFP_BYTES + r * G * kSfAtomBytes, wq[r], lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&full[stage]);
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (i + 1 < nkt)
                    load_sf(kt + 1);
            }
            if (lane == 0 && *abort_flag) {
                for (int i = max(0, issued - STAGES); i < issued; ++i)
                    mbar_wait_drain(&full[i % STAGES], (i / STAGES) & 1u, a.wait_limit);
            }
        } else if (!a.sf_rowmajor && lane == 0 && nkt > 0) {
            // Prepacked scales: three threads (warps 4, 6, 7) issue the P tile,
            // the Q tile and the 1-D bulk copies of the stage's relaid scale
            // atoms; each arrives on the stage's full barrier with its bytes.
            const int role = warp == 4 ? 0 : warp - 5;
            const uint64_t pol_p = a.stream_p ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_last();
            const uint8_t *sfp = a.sfP + static_cast<int64_t>(p0 / kSfRowBlock) * a.sf_rb_stride;
            const uint8_t *sfq = a.sfQ + static_cast<int64_t>(q0 / kSfRowBlock) * a.sf_rb_stride;
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int i = 0; i < nkt; ++i) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_limit,
                               &g_device_status))
                    break;
                uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                const int kt = kt0 + i;
                if (role == 0) {
                    mbar_arrive_expect_tx(&full[stage], Cf::P_BYTES);
                    tma_load_2d(st, &tmP, &full[stage], kt * 128, p0, pol_p);
                } else if (role == 1) {
                    mbar_arrive_expect_tx(&full[stage], a.q_box_rows * 128);
                    tma_load_2d(st + Cf::P_BYTES, &tmQ, &full[stage], kt * 128, q0, pol_q);
                } else {
                    mbar_arrive_expect_tx(&full[stage], Cf::SFP_BYTES + Cf::SFQ_BYTES);
                    // Stage kt's G k-groups: atoms G kt .. G kt + G - 1 of each block.
                    const int64_t sf_off = static_cast<int64_t>(kt) * G * kSfAtomBytes;
                    bulk_load(st + Cf::P_BYTES + Cf::Q_BYTES, sfp + sf_off, Cf::SFP_BYTES,
                              &full[stage], pol_p);
#pragma unroll
                    for (int r = 0; r < Cf::NQ; ++r)
                        bulk_load(st + Cf::P_BYTES + Cf::Q_BYTES + Cf::SFP_BYTES +
                                      r * G * kSfAtomBytes,
                                  sfq + r * a.sf_rb_stride + sf_off, G * kSfAtomBytes,
                                  &full[stage], pol_q);
                }
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (*abort_flag) {
                // Let the copies already issued land before the CTA exits.
                for (int i = max(0, issued - STAGES); i < issued; ++i)
                    mbar_wait_drain(&full[i % STAGES], (i / STAGES) & 1u, a.wait_limit);
            }
        }
        }
    } else if (warp == 5) {
        // ---------------------------------------------------- MMA issuer --
        if (lane == 0 && nkt > 0) {
            const uint32_t idesc = FMT == 0   ? idesc_mxf4(kTileM, BN)
                                   : FMT == 2 ? idesc_nvf4(kTileM, BN)
                                              : a.idesc8;
            const uint32_t t_sf = tmem + BN;
            // A 64-row Q tile uses the upper or lower half of its 128-row atom.
            // (Row-major scales are built relative to q0, so no offset there.)
            const uint32_t q_off = (BN < 128 && !a.sf_rowmajor)
                                       ? static_cast<uint32_t>((q0 % kSfRowBlock) / 32)
                                       : 0u;
            int stage = 0;
            uint32_t phase = 0;
            for (int i = 0; i < nkt; ++i) {
                // The scale writers arrive on sf_full only after they saw the
                // stage's full barrier, so it stands for both: one poll per
                // stage (each poll delays this thread's next MMA issue).
                if (!mbar_wait(&sf_full[stage], phase, abort_flag, a.wait_limit, &g_device_status))
                    break;
                tc_fence_after();
                uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                const uint32_t sfp_t = t_sf + stage * Cf::SF_COLS;
                const uint32_t sfq_t = sfp_t + Cf::SF_COLS_P;
                const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(st));
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_addr(st + Cf::P_BYTES));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if constexpr (FMT == 2) {
                        // K=64: the four 16-K scale bytes of word j.
                        mma_nvf4(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfp_t + j * 4,
                                 sfq_t + j * 4 * Cf::NQ + q_off, (i > 0 || j > 0) ? 1u : 0u);
                    } else if constexpr (FMT == 0) {
                        // K=64: bytes 0-1 / 2-3 of k-group j / 2.
                        const uint32_t sf_id = (j & 1) * 2;
                        mma_mxf4(tmem, adesc + 2 * j, bdesc + 2 * j, idesc_sf_ids(idesc, sf_id, sf_id),
                                 sfp_t + (j >> 1) * 4, sfq_t + (j >> 1) * 4 * Cf::NQ + q_off,
                                 (i > 0 || j > 0) ? 1u : 0u);
                    } else {
                        // K=32: byte j of the stage's single k-group.
                        mma_mxf8(tmem, adesc + 2 * j, bdesc + 2 * j, idesc_sf_ids(idesc, j, j), sfp_t,
                                 sfq_t + q_off, (i > 0 || j > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            mma_commit(acc_full);
            if (*abort_flag)
                mbar_wait_drain(acc_full, 0, a.wait_limit);   // MMAs in flight land first
        }
    } else {
        // ------------------------------------------------- scale writers --
        if (nkt > 0)
            write_stage_scales<Cf>(smem, full, sf_full, tmem + (static_cast<uint32_t>(warp * 32) << 16),
                                   nkt, kt0, a.sf_rowmajor && a.sf_tma, lane, abort_flag,
                                   a.wait_limit);
        // ------------------------------------------------------ epilogue --
        bool ok = nkt > 0 && mbar_wait(acc_full, 0, abort_flag, a.wait_limit, &g_device_status);
        ok = __all_sync(0xffffffffu, ok);
        // C, D and the workspace may belong to the preceding work.
        pdl_wait_prerequisites();
        if (ok) {
            tc_fence_after();
            const int row = warp * 32 + lane;
            const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
            if (a.split_k > 1 && a.cluster_reduce) {
                // Park this split's partial in this CTA's shared memory (the
                // ring: every MMA has read its last stage).
                float *part = reinterpret_cast<float *>(smem);
                const int stride = cluster_part_stride(a.part_cols);
                const int cols = min(a.part_cols, (SWAP ? a.M : a.N) - q0);
                const int nch = (cols + 3) / 4;
#pragma unroll 1
                for (int c0 = 0; c0 < cols; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c0, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (c0 / 4 + i < nch)
                            *reinterpret_cast<float4 *>(part + row * stride + c0 + 4 * i) =
                                make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                }
            } else if (a.split_k > 1) {
                // Park this split's partial (its valid columns) in the tile's slot.
                float *slot = partial_slot(a, tile, z);
                const int cols = min(a.part_cols, (SWAP ? a.M : a.N) - q0);
#pragma unroll 1
                for (int c0 = 0; c0 < cols; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c0, r);
                    tmem_ld_wait(r);
                    park_partial_chunk(a, slot, row, c0, r);
                }
                __threadfence();
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    if (SWAP && q0 + c0 >= a.M)
                        break;                                   // padding columns of D^T
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c0, r);
                    tmem_ld_wait(r);
                    if (!SWAP) {
                        const int m = p0 + row;
                        if (m < a.M && q0 + c0 < a.N)
                            store_row_chunk(a, m, q0 + c0, r);
                    } else {
                        store_col_chunk(a, q0 + c0, p0 + row, r);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (a.split_k > 1 && a.cluster_reduce) {
        // Every partial of the tile is in its CTA's shared memory once the
        // cluster barrier completes; the second barrier keeps this CTA's
        // partial alive until its peers have read it.
        pdl_wait_prerequisites();
        if (a.beta != 0.0f)
            prefetch_c_share<SWAP>(a, p0, q0, threadIdx.x);
        cluster_sync();
        reduce_tile_cluster<SWAP>(a, smem_addr(smem), cluster_part_stride(a.part_cols), p0, q0,
                                  threadIdx.x);
        cluster_sync();
    } else if (a.split_k > 1 && nkt > 0) {
        // Count this CTA into its tile (its partial rows are written and
        // fenced); the CTA that completes the count reduces the tile.
        if (threadIdx.x == 0 && !*abort_flag) {
            const bool last = tile_count_done(a.tile_count + tile, a.epoch, a.split_k);
            // The tile is complete: clear its counter for the next use of the
            // workspace (a CUDA-graph replay repeats this call's tag).
            if (last)
                atomicExch(a.tile_count + tile, 0ull);
            *last_flag = last ? 1 : 0;
        }
        __syncthreads();
        if (*last_flag) {
            __threadfence();
            pdl_wait_prerequisites();
            reduce_tile<SWAP>(a, tile, p0, q0, threadIdx.x);
        }
    }
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, Cf::TMEM_COLS);
    }
}

}  // namespace mxfp4

#include "gemm_pair.cuh"

namespace mxfp4 {

// ----------------------------------------------------------- host side --

template <int BN, int STAGES, bool SWAP, int FMT, int MINB>
static cudaError_t launch_cfg(const GemmArgs &a, const CUtensorMap &tmP, const CUtensorMap &tmQ,
                              const CUtensorMap &tmSP, const CUtensorMap &tmSQ, dim3 grid,
                              cudaStream_t stream)
{
    using Cf = CfgFor<BN, STAGES, FMT>;
    auto kern = gemm_mxf4_kernel<BN, STAGES, SWAP, FMT, MINB>;
    // Opt in to the large dynamic shared memory once per device.
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !configured[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        configured[dev].store(1, std::memory_order_relaxed);
    }
    // Programmatic dependent launch: the grid may start while the preceding
    // work on the stream drains; the kernel waits for it (griddepcontrol.wait)
    // before the accesses that depend on it.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.cluster_reduce) {
        // The split_k CTAs of a tile (grid z) form one cluster.
        if (static_cast<int>(grid.z) != a.split_k || a.split_k > 8 ||
            kTileM * cluster_part_stride(a.part_cols) * 4 > STAGES * Cf::STAGE_BYTES)
            return cudaErrorInvalidConfiguration;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = static_cast<unsigned>(a.split_k);
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, a, tmP, tmQ, tmSP, tmSQ);
}

size_t gemm_smem_bytes(const GemmShape &s)
{
    switch (s.tile_n) {
    case 256: return s.stages == 4 ? Cfg<256, 4>::SMEM_BYTES : 0;
    case 128: return s.stages == 6 ? Cfg<128, 6>::SMEM_BYTES : 0;
    case 64:
        return s.stages == 4 ? Cfg<64, 4>::SMEM_BYTES : s.stages == 8 ? Cfg<64, 8>::SMEM_BYTES : 0;
    default: return 0;
    }
}

bool gemm_config_exists(const GemmShape &s)
{
    if (!s.swap)
        return (s.tile_n == 256 && s.stages == 4) || (s.tile_n == 128 && s.stages == 6) ||
               (s.tile_n == 64 && s.stages == 8);
    return s.tile_n == 64 && s.stages == 4;
}

template <int FMT>
static cudaError_t launch_gemm_fmt(const GemmArgs &a, const CUtensorMap &tmP, const CUtensorMap &tmQ,
                                   const CUtensorMap &tmSP, const CUtensorMap &tmSQ,
                                   const GemmShape &s, dim3 grid, cudaStream_t stream)
{
    if (!s.swap) {
        if (s.tile_n == 256 && s.stages == 4)
            return launch_cfg<256, 4, false, FMT, 1>(a, tmP, tmQ, tmSP, tmSQ, grid, stream);
        if (s.tile_n == 128 && s.stages == 6)
            return launch_cfg<128, 6, false, FMT, 1>(a, tmP, tmQ, tmSP, tmSQ, grid, stream);
        if (s.tile_n == 64 && s.stages == 8)
            return launch_cfg<64, 8, false, FMT, 1>(a, tmP, tmQ, tmSP, tmSQ, grid, stream);
    } else {
        // Two CTAs per SM (the plan's slots for skinny shapes).
        if (s.tile_n == 64 && s.stages == 4)
            return launch_cfg<64, 4, true, FMT, 2>(a, tmP, tmQ, tmSP, tmSQ, grid, stream);
    }
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemm(const GemmArgs &a, const CUtensorMap &tmP, const CUtensorMap &tmQ,
                        const CUtensorMap &tmSP, const CUtensorMap &tmSQ, const GemmShape &s,
                        dim3 grid, cudaStream_t stream)
{
    if (s.nv) {
        // NVFP4 one-tile form: skinny shapes (swap-AB) with row-major scales
        // by TMA; everything else runs the CTA-pair kernel.
        if (!s.swap || s.tile_n != 64 || s.stages != 4 || !a.sf_rowmajor || !a.sf_tma)
            return cudaErrorInvalidConfiguration;
        return launch_cfg<64, 4, true, 2, 2>(a, tmP, tmQ, tmSP, tmSQ, grid, stream);
    }
    if (!s.fp8)
        return launch_gemm_fmt<0>(a, tmP, tmQ, tmSP, tmSQ, s, grid, stream);
    // kind::mxf8f6f4 element codes: E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5.
    auto known = [](int f) { return f == 0 || f == 1 || (f >= 3 && f <= 5); };
    if (!known(a.fmt_p) || !known(a.fmt_q))
        return cudaErrorInvalidValue;
    GemmArgs b = a;
    b.idesc8 = idesc_mxf8(kTileM, s.tile_n, static_cast<uint32_t>(a.fmt_p),
                          static_cast<uint32_t>(a.fmt_q));
    return launch_gemm_fmt<1>(b, tmP, tmQ, tmSP, tmSQ, s, grid, stream);
}

// The compiled pair configurations: MXFP4 with 6 stages of 256 K, NVFP4 with
// 5 (its larger scale slots leave room in tensor memory for five).
constexpr int kPairStages = 6;
constexpr int kPairStagesNv = 5;

size_t gemm_pair_smem_bytes() { return PairCfg<kPairStages, false>::SMEM_BYTES; }

template <int STAGES, bool NV>
static cudaError_t launch_pair_kernel(const GemmArgs &a, int tiles_p, int tiles_q, int ctas,
                                      const CUtensorMap &tmA, const CUtensorMap &tmB,
                                      const CUtensorMap &tmSA, const CUtensorMap &tmSB,
                                      cudaStream_t stream)
{
    using PC = PairCfg<STAGES, NV>;
    auto kern = gemm_mxf4_pair<STAGES, NV>;
    static std::atomic<int> max_clusters[64];   // per device; 0 = not yet queried
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(PC::THREADS);
    cfg.dynamicSmemBytes = PC::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int limit = dev < 64 ? max_clusters[dev].load() : 0;
    if (limit == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PC::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        // The kernel is persistent: every cluster must be resident at once.
        cfg.gridDim = dim3(2);
        e = cudaOccupancyMaxActiveClusters(&limit, kern, &cfg);
        if (e != cudaSuccess)
            return e;
        if (limit <= 0)
            return cudaErrorInvalidConfiguration;
        if (dev < 64)
            max_clusters[dev] = limit;
    }
    int clusters = ctas / 2;
    clusters = clusters < limit ? clusters : limit;
    if (clusters <= 0)
        return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * 2));
    // A programmatic dependent of the preceding work: the prologue overlaps
    // it, and every role waits for it (griddepcontrol.wait) before touching
    // memory it may write.  Right after this library's scale relayout
    // (a.ab_early) only the scale loads and the epilogue wait: the relayout
    // itself waited for the work before it.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    PairSched ps;
    ps.tiles_p = tiles_p;
    ps.tiles_q = tiles_q;
    ps.kt = a.kt_total;
    ps.group = tiles_p < 8 ? tiles_p : 8;
    return cudaLaunchKernelEx(&cfg, kern, a, ps, tmA, tmB, tmSA, tmSB);
}

cudaError_t launch_gemm_pair(const GemmArgs &a, int tiles_p, int tiles_q, int ctas,
                             const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const CUtensorMap &tmSA, const CUtensorMap &tmSB, bool nv,
                             cudaStream_t stream)
{
    if (nv)
        return launch_pair_kernel<kPairStagesNv, true>(a, tiles_p, tiles_q, ctas, tmA, tmB, tmSA,
                                                       tmSB, stream);
    return launch_pair_kernel<kPairStages, false>(a, tiles_p, tiles_q, ctas, tmA, tmB, tmSA, tmSB,
                                                  stream);
}

// Test hook: one wait on an mbarrier nobody arrives at.
__global__ void wait_probe_kernel(long long limit)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait(&bar, 0, &abort_flag, limit, &g_device_status);
}

cudaError_t launch_wait_probe(long long limit, cudaStream_t stream)
{
    wait_probe_kernel<<<1, 32, 0, stream>>>(limit);
    return cudaGetLastError();
}

cudaError_t read_device_status(int *status, int reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(status, g_device_status, sizeof(int));
    if (e != cudaSuccess || !reset)
        return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
}

}  // namespace mxfp4
