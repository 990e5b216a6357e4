// MXFP4 quantiser: bf16 rows [rows, K] -> packed E2M1 codes [rows, K/2] and
// E8M0 scale codes [rows, K/32] -- the operands mxfp4_gemm takes.
//
// Per 1x32 block (the workloads' operand rule; E2M1 values and nibble order
// from page "asm_f4gemm -- driving aiter's gfx950 MXFP4 GEMM code objects",
// section "Data layouts"):
//   s = floor(log2(amax / 6)), the largest integer with 6 * 2^s <= amax
//       (s = 0 for an all-zero block), clamped to [-127, 127]; scale = s + 127;
//   code_i = x_i / 2^s rounded to the nearest E2M1 value, ties to even,
//       saturating at +-6, sign copied from x_i; element 2i in the low nibble.
//
// One thread per block: it loads the block's 64 bytes (four 16-byte loads;
// a warp covers 2 KB of a row contiguously), takes amax with packed bf16
// max, derives s from amax's exponent and leading significand bits (6 * 2^s
// <= 1.m * 2^E  <=>  s <= E + 2 - [1.m < 1.5] ... see below), scales by the
// exact power of two 2^-s, and converts pairs with cvt.rn.satfinite.e2m1x2
// (round to nearest even, saturating at the largest finite value 6).  The
// 16 bytes of codes go out in one store (coalesced across the warp), the
// scale byte beside them.  Bandwidth-bound: 2 bytes in, 17/32 bytes out per
// element.
#include <cuda_bf16.h>

#include "internal.h"

namespace mxfp4 {

namespace {

constexpr int kQuantThreads = 256;

// Largest s with 6 * 2^s <= a for a finite a > 0 (float bits): a = f * 2^e
// with f in [1, 2) (or a subnormal), and 6 * 2^s = 1.5 * 2^(s + 2), so
// s = e - 2 when f >= 1.5, else e - 3.
__device__ __forceinline__ int block_exponent(float amax)
{
    if (amax == 0.0f)
        return 0;
    const uint32_t bits = __float_as_uint(amax);
    const int biased = static_cast<int>((bits >> 23) & 0xFFu);
    int s;
    if (biased == 0) {
        s = -127;                                   // below 2^-126: clamps
    } else {
        const int e = biased - 127;
        s = (bits & 0x400000u) ? e - 2 : e - 3;     // f >= 1.5 iff the top significand bit is set
    }
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// Two floats -> one byte of two E2M1 codes: `lo` in bits 0-3, `hi` in 4-7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kQuantThreads)
    quantize_kernel(uint8_t *__restrict__ Q, int64_t ldq_bytes, uint8_t *__restrict__ S,
                    int64_t lds, const uint16_t *__restrict__ X, int64_t ldx, int rows, int kblocks)
{
    const int64_t total = static_cast<int64_t>(rows) * kblocks;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = g / kblocks;
        const int b = static_cast<int>(g - r * kblocks);
        const uint4 *src = reinterpret_cast<const uint4 *>(X + r * ldx + b * 32);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = __ldcs(src + i);
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        // amax over the 32 magnitudes (sign bits cleared, compared as floats)
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
        const int s = block_exponent(amax);
        // 2^-s as a float (s in [-127, 127]: 2^127 is normal, 2^-127 subnormal)
        const float inv = s == 127 ? __uint_as_float(0x00400000u)
                                   : __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
        uint32_t out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t x2 = w[4 * q + j];            // elements 2i (low), 2i+1 (high)
                word |= e2m1x2(bf16_lo(x2) * inv, bf16_hi(x2) * inv) << (8 * j);
            }
            out[q] = word;
        }
        *reinterpret_cast<uint4 *>(Q + r * ldq_bytes + b * 16) = make_uint4(out[0], out[1], out[2], out[3]);
        S[r * lds + b] = static_cast<uint8_t>(s + 127);
    }
}

// ---------------------------------------------------------------- MXFP8 --
// bf16 rows -> one E4M3 / E5M2 code per element [rows, K] (or E2M3 / E3M2 /
// E2M1 codes in the padded forms the GEMM reads) + E8M0 scales.
// Per 1x32 block: s = floor(log2 amax) - emax (emax 8 for E4M3, 15 for
// E5M2, 2 for E2M3 and E2M1, 4 for E3M2: the exponent of the format's
// largest binade, the OCP MX rule;
// s = 0 for an all-zero block; clamped to [-127, 127]); codes = x / 2^s
// converted with cvt.rn.satfinite (nearest, ties to even, saturating at the
// largest finite value).  One thread per block; its 32 codes leave in two
// 16-byte stores.

// floor(log2 amax) - emax from amax's float exponent (a subnormal amax is
// below 2^-126 and clamps).
__device__ __forceinline__ int block_exponent8(float amax, int emax)
{
    if (amax == 0.0f)
        return 0;
    const int biased = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
    const int s = biased == 0 ? -127 : biased - 127 - emax;
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// Two floats -> two 8-bit codes: `lo` in bits 0-7, `hi` in bits 8-15.
template <int FMT>
__device__ __forceinline__ uint32_t f8x2(float lo, float hi)
{
    uint32_t r;
    if constexpr (FMT == 0)
        asm("{\n\t.reg .b16 t;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
            "cvt.u32.u16 %0, t;\n\t}"
            : "=r"(r)
            : "f"(hi), "f"(lo));
    else
        asm("{\n\t.reg .b16 t;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 t, %1, %2;\n\t"
            "cvt.u32.u16 %0, t;\n\t}"
            : "=r"(r)
            : "f"(hi), "f"(lo));
    return r;
}

// Two floats -> two 6-bit codes: `lo` in bits 0-5, `hi` in bits 8-13
// (FMT 3: E2M3, 4: E3M2).
template <int FMT>
__device__ __forceinline__ uint32_t f6x2(float lo, float hi)
{
    uint32_t r;
    if constexpr (FMT == 3)
        asm("{\n\t.reg .b16 t;\n\t"
            "cvt.rn.satfinite.e2m3x2.f32 t, %1, %2;\n\t"
            "cvt.u32.u16 %0, t;\n\t}"
            : "=r"(r)
            : "f"(hi), "f"(lo));
    else
        asm("{\n\t.reg .b16 t;\n\t"
            "cvt.rn.satfinite.e3m2x2.f32 t, %1, %2;\n\t"
            "cvt.u32.u16 %0, t;\n\t}"
            : "=r"(r)
            : "f"(hi), "f"(lo));
    return r;
}

// 16 six-bit codes (c[i] < 64) -> the padded 16-byte group the GEMM reads:
// code i in bits 6i .. 6i+5 of the first 12 bytes (little-endian), then 4
// zero bytes.
__device__ __forceinline__ uint4 pack_fp6_group(const uint32_t *c)
{
    uint4 g;
    g.x = c[0] | (c[1] << 6) | (c[2] << 12) | (c[3] << 18) | (c[4] << 24) | (c[5] << 30);
    g.y = (c[5] >> 2) | (c[6] << 4) | (c[7] << 10) | (c[8] << 16) | (c[9] << 22) | (c[10] << 28);
    g.z = (c[10] >> 4) | (c[11] << 2) | (c[12] << 8) | (c[13] << 14) | (c[14] << 20) |
          (c[15] << 26);
    g.w = 0u;
    return g;
}

// FMT: the ABI's format codes -- 0: E4M3, 1: E5M2 (one code per byte);
// 3: E2M3, 4: E3M2, 5: E2M1 (the padded 16-elements-per-16-bytes forms).
template <int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quantize8_kernel(uint8_t *__restrict__ Q, int64_t ldq, uint8_t *__restrict__ S, int64_t lds,
                     const uint16_t *__restrict__ X, int64_t ldx, int rows, int kblocks)
{
    constexpr int kEmax = FMT == 0 ? 8 : FMT == 1 ? 15 : FMT == 4 ? 4 : 2;
    const int64_t total = static_cast<int64_t>(rows) * kblocks;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = g / kblocks;
        const int b = static_cast<int>(g - r * kblocks);
        const uint4 *src = reinterpret_cast<const uint4 *>(X + r * ldx + b * 32);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = __ldcs(src + i);
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
        const int s = block_exponent8(amax, kEmax);
        const float inv = s == 127 ? __uint_as_float(0x00400000u)
                                   : __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
        uint4 *dst = reinterpret_cast<uint4 *>(Q + r * ldq + b * 32);
        if constexpr (FMT <= 1) {
            uint32_t out[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                // elements 4q .. 4q+3 (two bf16 pairs) -> one 32-bit word of codes
                const uint32_t lo = f8x2<FMT>(bf16_lo(w[2 * q]) * inv, bf16_hi(w[2 * q]) * inv);
                const uint32_t hi =
                    f8x2<FMT>(bf16_lo(w[2 * q + 1]) * inv, bf16_hi(w[2 * q + 1]) * inv);
                out[q] = lo | (hi << 16);
            }
            dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
            dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
        } else if constexpr (FMT == 5) {
            // Each 16 elements: 8 bytes of nibble pairs, then 8 zero bytes.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t word[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t v = 0u;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t p = w[8 * h + 4 * q + j];
                        v |= e2m1x2(bf16_lo(p) * inv, bf16_hi(p) * inv) << (8 * j);
                    }
                    word[q] = v;
                }
                dst[h] = make_uint4(word[0], word[1], 0u, 0u);
            }
        } else {
            uint32_t c[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t v = f6x2<FMT>(bf16_lo(w[i]) * inv, bf16_hi(w[i]) * inv);
                c[2 * i] = v & 0x3Fu;
                c[2 * i + 1] = (v >> 8) & 0x3Fu;
            }
            dst[0] = pack_fp6_group(c);
            dst[1] = pack_fp6_group(c + 16);
        }
        S[r * lds + b] = static_cast<uint8_t>(s + 127);
    }
}

}  // namespace

cudaError_t launch_quantize8(uint8_t *Q, int64_t ldq, uint8_t *S, int64_t lds, const uint16_t *X,
                             int64_t ldx, int rows, int K, int fmt, int sms, cudaStream_t stream)
{
    const int kblocks = K / 32;
    const int64_t total = static_cast<int64_t>(rows) * kblocks;
    int64_t blocks = (total + kQuantThreads - 1) / kQuantThreads;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 16;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    const unsigned g = static_cast<unsigned>(blocks);
    switch (fmt) {
    case 0: quantize8_kernel<0><<<g, kQuantThreads, 0, stream>>>(Q, ldq, S, lds, X, ldx, rows, kblocks); break;
    case 1: quantize8_kernel<1><<<g, kQuantThreads, 0, stream>>>(Q, ldq, S, lds, X, ldx, rows, kblocks); break;
    case 3: quantize8_kernel<3><<<g, kQuantThreads, 0, stream>>>(Q, ldq, S, lds, X, ldx, rows, kblocks); break;
    case 4: quantize8_kernel<4><<<g, kQuantThreads, 0, stream>>>(Q, ldq, S, lds, X, ldx, rows, kblocks); break;
    case 5: quantize8_kernel<5><<<g, kQuantThreads, 0, stream>>>(Q, ldq, S, lds, X, ldx, rows, kblocks); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize(uint8_t *Q, int64_t ldq_bytes, uint8_t *S, int64_t lds,
                            const uint16_t *X, int64_t ldx, int rows, int K, int sms,
                            cudaStream_t stream)
{
    const int kblocks = K / 32;
    const int64_t total = static_cast<int64_t>(rows) * kblocks;
    int64_t blocks = (total + kQuantThreads - 1) / kQuantThreads;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 16;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    quantize_kernel<<<static_cast<unsigned>(blocks), kQuantThreads, 0, stream>>>(
        Q, ldq_bytes, S, lds, X, ldx, rows, kblocks);
    return cudaGetLastError();
}

}  // namespace mxfp4
