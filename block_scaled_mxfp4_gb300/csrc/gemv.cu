// Block-scaled MXFP4 GEMV for M <= 2 rows of A (decode-style shapes).
//
//   D[m, n] = alpha * sum_k A[m, k] B[n, k] + beta * C[m, n]
//
// with A and B E2M1 codes, each 1x32 K block scaled by its E8M0 exponent
// (page "asm_f4gemm -- driving aiter's gfx950 MXFP4 GEMM code objects",
// formula and section "Data layouts"; the scale multiplies its block's
// products before they are accumulated, page "CDNA4 dense MFMA builtins",
// section "Mixed-precision with scaling").
//
// At M <= 2 the product is a matrix-vector product bound by the HBM stream
// of B (N*K/2 bytes, ~1 FLOP per byte), so it runs on the CUDA cores instead
// of padding M up to a tensor-core tile: every warp streams kGemvRows rows of
// B with 16-byte coalesced loads (lane l of a warp load takes K block 32c + l
// of chunk c), two or three chunks in flight per warp, one launch, no
// workspace.  Per 16 loaded bytes (one 32-element K block of one row):
//   - cvt.rn.f16x2.e2m1x2 turns each byte (two codes) into two exact halves;
//   - packed f16 multiply-adds form the block's 32 code products in four
//     chains of four per half (products of E2M1 values have <= 4 significant
//     bits; a chain stays <= 4*36 in steps of 1/4, exact in f16), pairs of
//     chains are added in f16 (still exact) and the halves summed in fp32:
//     the block sum is exact (|sum| <= 32*36);
//   - the block sum is scaled by 2^(ea-127) * 2^(eb-127) (exact in range) and
//     added to the row's fp32 accumulator (the one rounding per block, as in
//     the tensor-core MMA).
// The lanes' accumulators are combined by a fixed xor-shuffle tree, so the
// result is the same on every run; alpha, beta*C and the one bf16 rounding
// follow.  A and B use the same code-to-half conversion, so the products pair
// the codes of equal k whichever half each nibble lands in.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace mxfp4 {

namespace {

constexpr int kGemvRows = 4;    // B rows per warp
// 1024-element K chunks in flight per warp (fewer for M = 2: registers).
template <int M>
__host__ __device__ constexpr int gemv_depth() { return M == 1 ? 3 : 2; }
constexpr int kGemvMaxWarps = 16;

// Eight E2M1 codes (4 bytes) -> four f16x2 holding the exact values.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t *h)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

__device__ __forceinline__ __half2 as_h2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }

// Exact sum of the 32 code products of one K block (16 f16x2 of each side):
// four f16x2 chains of four products (each half <= 4 * 36 in steps of 1/4,
// exact in f16), pairs of chains added in f16 (<= 8 products, still exact),
// then the four halves summed in fp32 (exact).
__device__ __forceinline__ float block_dot(const uint32_t *a, const uint32_t *b)
{
    __half2 p0 = __hmul2(as_h2(a[0]), as_h2(b[0]));
    __half2 p1 = __hmul2(as_h2(a[1]), as_h2(b[1]));
    __half2 p2 = __hmul2(as_h2(a[2]), as_h2(b[2]));
    __half2 p3 = __hmul2(as_h2(a[3]), as_h2(b[3]));
#pragma unroll
    for (int i = 4; i < 16; i += 4) {
        p0 = __hfma2(as_h2(a[i]), as_h2(b[i]), p0);
        p1 = __hfma2(as_h2(a[i + 1]), as_h2(b[i + 1]), p1);
        p2 = __hfma2(as_h2(a[i + 2]), as_h2(b[i + 2]), p2);
        p3 = __hfma2(as_h2(a[i + 3]), as_h2(b[i + 3]), p3);
    }
    const float2 f0 = __half22float2(__hadd2(p0, p1));
    const float2 f1 = __half22float2(__hadd2(p2, p3));
    return (f0.x + f0.y) + (f1.x + f1.y);
}

// 2^(e - 127) for an E8M0 byte; 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_float(uint32_t e)
{
    const uint32_t bits = e == 0 ? 0x00400000u : e == 255 ? 0x7FC00000u : e << 23;
    return __uint_as_float(bits);
}

__device__ __forceinline__ uint4 ld_stream_v4(const uint8_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Byte offset of scale (row, K block) in a relaid scale buffer (see
// mxfp4_scale_relayout): atom (row / 128, blk / 4), line row % 32, word
// (row % 128) / 32, byte blk % 4.
__device__ __forceinline__ int64_t relaid_sf_offset(int row, int blk, int64_t groups)
{
    const int64_t atom = static_cast<int64_t>(row / kSfRowBlock) * groups + blk / 4;
    const int r = row % kSfRowBlock;
    return atom * kSfAtomBytes + 16 * (r % 32) + 4 * (r / 32) + (blk % 4);
}

template <int M>
__global__ void __launch_bounds__(kGemvMaxWarps * 32)
    gemv_mxf4_kernel(const GemvArgs g)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int kblocks = g.K / 32;
    const int nchunks = (kblocks + 31) / 32;
    const int groups_n = (g.N + kGemvRows - 1) / kGemvRows;
    const int64_t sf_groups_k = sf_groups(g.K);
    constexpr int kGemvDepth = gemv_depth<M>();

    for (int grp = blockIdx.x * (blockDim.x >> 5) + warp; grp < groups_n;
         grp += gridDim.x * (blockDim.x >> 5)) {
        const int n0 = grp * kGemvRows;
        float acc[M][kGemvRows];
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r)
                acc[m][r] = 0.0f;

        uint4 bq[kGemvDepth][kGemvRows];
        uint32_t sbq[kGemvDepth][kGemvRows];
        uint4 aq[kGemvDepth][M];
        uint32_t saq[kGemvDepth][M];
        auto load = [&](int d, int c) {
            const int blk = c * 32 + lane;
            const bool ok = blk < kblocks;
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r) {
                const int n = n0 + r;
                if (ok && n < g.N) {
                    bq[d][r] = ld_stream_v4(g.B + static_cast<int64_t>(n) * g.ldb_bytes + blk * 16);
                    sbq[d][r] = g.sf_relaid ? g.SB[relaid_sf_offset(n, blk, sf_groups_k)]
                                            : g.SB[static_cast<int64_t>(n) * g.ld_sb + blk];
                } else {
                    bq[d][r] = make_uint4(0u, 0u, 0u, 0u);
                    sbq[d][r] = 127u;
                }
            }
#pragma unroll
            for (int m = 0; m < M; ++m) {
                if (ok) {
                    aq[d][m] = __ldg(reinterpret_cast<const uint4 *>(
                        g.A + static_cast<int64_t>(m) * g.lda_bytes + blk * 16));
                    saq[d][m] = g.sf_relaid ? g.SA[relaid_sf_offset(m, blk, sf_groups_k)]
                                            : g.SA[static_cast<int64_t>(m) * g.ld_sa + blk];
                } else {
                    aq[d][m] = make_uint4(0u, 0u, 0u, 0u);
                    saq[d][m] = 127u;
                }
            }
        };
        auto compute = [&](int d) {
            uint32_t ah[M][16];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                e2m1x8_to_f16x2(aq[d][m].x, &ah[m][0]);
                e2m1x8_to_f16x2(aq[d][m].y, &ah[m][4]);
                e2m1x8_to_f16x2(aq[d][m].z, &ah[m][8]);
                e2m1x8_to_f16x2(aq[d][m].w, &ah[m][12]);
            }
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r) {
                uint32_t bh[16];
                e2m1x8_to_f16x2(bq[d][r].x, &bh[0]);
                e2m1x8_to_f16x2(bq[d][r].y, &bh[4]);
                e2m1x8_to_f16x2(bq[d][r].z, &bh[8]);
                e2m1x8_to_f16x2(bq[d][r].w, &bh[12]);
                const float sb = e8m0_to_float(sbq[d][r]);
#pragma unroll
                for (int m = 0; m < M; ++m)
                    acc[m][r] = fmaf(block_dot(ah[m], bh) * e8m0_to_float(saq[d][m]), sb,
                                     acc[m][r]);
            }
        };

#pragma unroll
        for (int d = 0; d < kGemvDepth; ++d)
            if (d < nchunks)
                load(d, d);
        for (int c = 0; c < nchunks; c += kGemvDepth) {
#pragma unroll
            for (int d = 0; d < kGemvDepth; ++d) {
                if (c + d < nchunks) {
                    compute(d);
                    if (c + d + kGemvDepth < nchunks)
                        load(d, c + d + kGemvDepth);
                }
            }
        }

        // Fixed-order tree over the lanes; every lane ends with the totals.
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    acc[m][r] += __shfl_xor_sync(0xffffffffu, acc[m][r], off);

#pragma unroll
        for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r) {
                const int n = n0 + r;
                if (lane == m * kGemvRows + r && m < g.M && n < g.N) {
                    float v = g.alpha * acc[m][r];
                    if (g.beta != 0.0f)
                        v = fmaf(g.beta,
                                 __uint_as_float(static_cast<uint32_t>(
                                                     g.C[static_cast<int64_t>(m) * g.ldc + n])
                                                 << 16),
                                 v);
                    __nv_bfloat16 b = __float2bfloat16_rn(v);
                    g.D[static_cast<int64_t>(m) * g.ldd + n] = *reinterpret_cast<uint16_t *>(&b);
                }
            }
        }
    }
}

}  // namespace

void gemv_launch_shape(int N, int sms, int *ctas, int *threads)
{
    const int groups_n = (N + kGemvRows - 1) / kGemvRows;
    const int s = sms > 0 ? sms : 152;
    int w = (groups_n + s - 1) / s;
    if (w < 1)
        w = 1;
    if (w > kGemvMaxWarps)
        w = kGemvMaxWarps;
    int c = (groups_n + w - 1) / w;
    if (c > 65535)
        c = 65535;
    *ctas = c;
    *threads = w * 32;
}

cudaError_t launch_gemv(const GemvArgs &g, int sms, cudaStream_t stream)
{
    int ctas = 0, threads = 0;
    gemv_launch_shape(g.N, sms, &ctas, &threads);
    if (g.M == 1)
        gemv_mxf4_kernel<1><<<ctas, threads, 0, stream>>>(g);
    else if (g.M == 2)
        gemv_mxf4_kernel<2><<<ctas, threads, 0, stream>>>(g);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace mxfp4
