"""Seeded synthetic inputs for the block-scaled MXFP4 GEMM.

This module only *produces bytes*: packed fp4x2 E2M1 operands, row-major E8M0
scales and bf16 C.  It holds none of the GEMM's arithmetic, so both the CUDA
path and the CPU oracle can consume what it makes without sharing code.

Formats (page "asm_f4gemm -- driving aiter's gfx950 MXFP4 GEMM code objects",
section "Data layouts"):
  * A [M, K/2] and B [N, K/2] bytes, row-major; byte i of a row holds element
    2i in the low nibble and element 2i+1 in the high nibble.
  * E2M1 codes: bit 3 is the sign, bits 2..0 index the magnitudes
    {0, .5, 1, 1.5, 2, 3, 4, 6}.
  * One E8M0 scale byte per 32 consecutive K elements, row-major [rows, K/32].

Workloads are the five shapes of the GB300 target list (tiny, decode, mid,
large, skinny-M wide-K), plus an identity case.  Values follow each recipe:
  * tiny:   codes uniform over all 16, scale exponent uniform in {-4..4}.
  * others: x ~ N(0,1) (skinny: U[-1,1]); per 1x32 block the scale exponent is
    s = floor(log2(max|x| / 6)) (s = 0 for an all-zero block, clamped to
    [-127, 127]); the element code is x / 2^s rounded to nearest E2M1 with
    ties to the even mantissa and saturation at +-6; the sign bit copies
    sign(x).
Draw order within a workload: A, then B, then C, each drawn row-chunk by
row-chunk in C order from one numpy PCG64 generator seeded per workload.

MXFP8 problems (page "CDNA4 dense MFMA builtins": FP8 = E4M3, BF8 = E5M2,
scaled per block like FP4) hold one 8-bit code per element, A [M, K] and
B [N, K], with the same E8M0 scales [rows, K/32].  Their values are
x ~ N(0,1) (or U[-1,1]) with the OCP MX scale rule per 1x32 block,
s = floor(log2(max|x|)) - emax (emax 8 for E4M3, 15 for E5M2; s = 0 for an
all-zero block), and x / 2^s cast to the format by torch's float8 conversion
(nearest, ties to even) after clamping to the largest finite value.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

_ROW_CHUNK = 1024


@dataclasses.dataclass
class Problem:
    """One GEMM instance: D = alpha * A . B^T + beta * C (all host numpy)."""

    name: str
    M: int
    N: int
    K: int
    A: np.ndarray            # uint8 [M, K/2] packed E2M1
    B: np.ndarray            # uint8 [N, K/2] packed E2M1
    SA: np.ndarray           # uint8 [M, K/32] E8M0
    SB: np.ndarray           # uint8 [N, K/32] E8M0
    C: Optional[np.ndarray]  # uint16 [M, N] bf16 bits, or None
    alpha: float
    beta: float
    seed: int


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes [rows, K] into bytes [rows, K/2]: even k -> low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.ndim == 2 and codes.shape[1] % 2 == 0
    lo = codes[:, 0::2] & 0xF
    hi = codes[:, 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack_fp4: bytes [rows, K/2] -> codes [rows, K]."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the bits.

    Used only to turn the N(0, sigma) draws for C into bf16 input bytes.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = r.astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def _block_scale_exponents(x: np.ndarray) -> np.ndarray:
    """s = floor(log2(blockmax / 6)) per 1x32 block, 0 for all-zero blocks."""
    rows, K = x.shape
    amax = np.abs(x).reshape(rows, K // 32, 32).max(axis=2)
    _, e = np.frexp(amax / 6.0)           # amax/6 = f * 2^e, f in [0.5, 1)
    s = (e - 1).astype(np.int64)          # exact floor(log2(.)) for > 0
    s[amax == 0] = 0
    return np.clip(s, -127, 127)


def _e2m1_codes_rne_sat(y: np.ndarray) -> np.ndarray:
    """Nearest-even E2M1 magnitude code of |y| with saturation at 6.

    Decision points are the midpoints of {0,.5,1,1.5,2,3,4,6}; a tie goes to
    the neighbour whose mantissa bit is 0 (codes 0,2,4,6).
    """
    a = np.abs(y)
    code = ((a > 0.25).astype(np.uint8) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
            + (a > 2.5) + (a >= 3.5) + (a > 5.0))
    return code.astype(np.uint8)


def quantize_rows(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantise float64 rows [rows, K] (K % 32 == 0) to (packed codes, E8M0)."""
    rows, K = x.shape
    assert K % 32 == 0
    s = _block_scale_exponents(x)
    y = np.ldexp(x.reshape(rows, K // 32, 32), -s[:, :, None]).reshape(rows, K)
    mag = _e2m1_codes_rne_sat(y)
    sign = np.signbit(x).astype(np.uint8) << 3
    codes = mag | sign
    return pack_fp4(codes), (s + 127).astype(np.uint8)


def _quantized_operand(rng: np.random.Generator, rows: int, K: int, dist: str):
    packed = np.empty((rows, K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    for r0 in range(0, rows, _ROW_CHUNK):
        r1 = min(rows, r0 + _ROW_CHUNK)
        if dist == "normal":
            x = rng.standard_normal((r1 - r0, K))
        elif dist == "uniform":
            x = rng.uniform(-1.0, 1.0, size=(r1 - r0, K))
        else:
            raise ValueError(dist)
        packed[r0:r1], scales[r0:r1] = quantize_rows(x)
    return packed, scales


def _uniform_code_operand(rng: np.random.Generator, rows: int, K: int):
    codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    scales = (rng.integers(-4, 5, size=(rows, K // 32)) + 127).astype(np.uint8)
    return pack_fp4(codes), scales


def _bf16_normal(rng: np.random.Generator, rows: int, cols: int, sigma: float):
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, _ROW_CHUNK):
        r1 = min(rows, r0 + _ROW_CHUNK)
        x = sigma * rng.standard_normal((r1 - r0, cols))
        out[r0:r1] = f32_to_bf16_bits(x.astype(np.float32))
    return out


# name -> (M, N, K, seed, value recipe, alpha, beta, C sigma or None)
WORKLOADS = {
    "tiny":   (128, 256, 512, 0, "codes", 1.0, 0.0, None),
    "decode": (1, 8192, 8192, 1, "normal", 1.0, 0.0, None),
    "mid":    (512, 1024, 2048, 2, "normal", 0.5, 0.5, 1.0),
    "large":  (8192, 8192, 8192, 3, "normal", 1.0, 0.0, None),
    "skinny": (64, 7168, 16384, 4, "uniform", 1.0, 1.0, 0.1),
}


def make_problem(name: str, M: int, N: int, K: int, seed: int, values: str,
                 alpha: float, beta: float, c_sigma: Optional[float]) -> Problem:
    """Draw one problem of any shape with one of the workload value recipes."""
    if K % 32 != 0:
        raise ValueError("K must be a multiple of 32 (one E8M0 scale per 32)")
    rng = np.random.default_rng(seed)
    if values == "codes":
        A, SA = _uniform_code_operand(rng, M, K)
        B, SB = _uniform_code_operand(rng, N, K)
    else:
        A, SA = _quantized_operand(rng, M, K, values)
        B, SB = _quantized_operand(rng, N, K, values)
    C = _bf16_normal(rng, M, N, c_sigma) if c_sigma is not None else None
    return Problem(name, M, N, K, A, B, SA, SB, C, float(alpha), float(beta), seed)


def workload(name: str) -> Problem:
    M, N, K, seed, values, alpha, beta, c_sigma = WORKLOADS[name]
    return make_problem(name, M, N, K, seed, values, alpha, beta, c_sigma)


def make_problem_nv(name: str, M: int, N: int, K: int, seed: int, alpha: float, beta: float,
                    c_sigma: Optional[float], scale_lo: int = 0x28,
                    scale_hi: int = 0x48) -> Problem:
    """An NVFP4 problem: packed E2M1 codes drawn uniformly from all 16, and
    one UE4M3 scale byte per 16 K drawn uniformly from [scale_lo, scale_hi]
    (the default 0x28..0x48 spans 0.25 .. 4); SA and SB are [rows, K/16]."""
    if K % 32 != 0:
        raise ValueError("K must be a multiple of 32")
    rng = np.random.default_rng(seed)
    A = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    SA = rng.integers(scale_lo, scale_hi + 1, size=(M, K // 16)).astype(np.uint8)
    SB = rng.integers(scale_lo, scale_hi + 1, size=(N, K // 16)).astype(np.uint8)
    C = _bf16_normal(rng, M, N, c_sigma) if c_sigma is not None else None
    return Problem(name, M, N, K, A, B, SA, SB, C, float(alpha), float(beta), seed)


def identity_problem(M: int = 128, N: int = 256, K: int = 512, seed: int = 0) -> Problem:
    """B[n, k] = 1 iff n == k (code 2, scale code 127); A as in 'tiny'.

    With all scales 127 the product is D[m, n] = A[m, n] for n < min(N, K).
    """
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(M, K), dtype=np.uint8)
    A = pack_fp4(codes)
    SA = np.full((M, K // 32), 127, dtype=np.uint8)
    bcodes = np.zeros((N, K), dtype=np.uint8)
    idx = np.arange(min(N, K))
    bcodes[idx, idx] = 2
    B = pack_fp4(bcodes)
    SB = np.full((N, K // 32), 127, dtype=np.uint8)
    return Problem("identity", M, N, K, A, B, SA, SB, None, 1.0, 0.0, seed)


# ---------------------------------------------------------------- MXFP8 --

# format name -> (oracle format code, largest element exponent, largest finite)
FP8_FORMATS = {"e4m3": (1, 8, 448.0), "e5m2": (2, 15, 57344.0)}
# 6-bit formats: (oracle format code, largest element exponent, largest
# finite, exponent bits, mantissa bits, bias).  Stored 16 codes per 16 bytes.
FP6_FORMATS = {"e2m3": (3, 2, 7.5, 2, 3, 1), "e3m2": (4, 4, 28.0, 3, 2, 3)}
# E2M1 in the same padded form (16 codes in the first 8 of every 16 bytes),
# the form in which it mixes with the 8- and 6-bit formats.
FP4P_FORMATS = {"e2m1": (5, 2, 6.0, 2, 1, 1)}
SUBBYTE_FORMATS = {**FP6_FORMATS, **FP4P_FORMATS}
BYTE_FORMATS = {**{k: v[0] for k, v in FP8_FORMATS.items()},
                **{k: v[0] for k, v in SUBBYTE_FORMATS.items()}}


@dataclasses.dataclass
class Problem8:
    """One MXFP8 / MXFP6 GEMM instance: A [M, K] and B [N, K] bytes."""

    name: str
    M: int
    N: int
    K: int
    fmt_a: str               # "e4m3", "e5m2" (one code per byte), "e2m3", "e3m2" (16
    fmt_b: str               # codes in 12 of every 16 bytes) or "e2m1" (16 in 8 of 16)
    A: np.ndarray            # uint8 [M, K]
    B: np.ndarray            # uint8 [N, K]
    SA: np.ndarray           # uint8 [M, K/32] E8M0
    SB: np.ndarray           # uint8 [N, K/32] E8M0
    C: Optional[np.ndarray]  # uint16 [M, N] bf16 bits, or None
    alpha: float
    beta: float
    seed: int


def quantize_rows_fp8(x: np.ndarray, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """Quantise float64 rows [rows, K] (K % 32 == 0) to (8-bit codes, E8M0)."""
    import torch
    rows, K = x.shape
    assert K % 32 == 0
    _, emax, top = FP8_FORMATS[fmt]
    amax = np.abs(x).reshape(rows, K // 32, 32).max(axis=2)
    _, e = np.frexp(amax)                 # amax = f * 2^e, f in [0.5, 1)
    s = (e - 1 - emax).astype(np.int64)   # floor(log2(amax)) - emax
    s[amax == 0] = 0
    s = np.clip(s, -127, 127)
    y = np.ldexp(x.reshape(rows, K // 32, 32), -s[:, :, None]).reshape(rows, K)
    y = np.clip(y, -top, top)
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    codes = torch.from_numpy(np.ascontiguousarray(y)).to(dt).view(torch.uint8).numpy()
    return codes.astype(np.uint8), (s + 127).astype(np.uint8)


def pack_fp6(codes: np.ndarray) -> np.ndarray:
    """[rows, K] 6-bit codes (K % 16 == 0) -> [rows, K] bytes: every 16 codes
    packed little-endian (code i in bits 6i..6i+5) into 12 bytes, then 4
    zero bytes -- the FP6 operand layout of the GEMM."""
    rows, K = codes.shape
    bits = ((codes.astype(np.int64)[..., None] >> np.arange(6)) & 1).astype(np.uint8)
    body = np.packbits(bits.reshape(rows, K // 16, 96), axis=2, bitorder="little")
    out = np.zeros((rows, K // 16, 16), dtype=np.uint8)
    out[:, :, :12] = body
    return out.reshape(rows, K)


def pack_fp4_padded(codes: np.ndarray) -> np.ndarray:
    """[rows, K] 4-bit codes (K % 16 == 0) -> [rows, K] bytes: every 16 codes
    two per byte (element 2i in the low nibble of byte i) in 8 bytes, then 8
    zero bytes."""
    rows, K = codes.shape
    c = codes.astype(np.uint8).reshape(rows, K // 16, 8, 2)
    out = np.zeros((rows, K // 16, 16), dtype=np.uint8)
    out[:, :, :8] = c[..., 0] | (c[..., 1] << 4)
    return out.reshape(rows, K)


def quantize_rows_fp6(x: np.ndarray, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """Quantise float64 rows [rows, K] (K % 32 == 0) to (padded FP6 or E2M1
    bytes, E8M0): scale 2^(floor(log2 amax) - emax) per 32 (the OCP MX rule),
    then each element to the nearest value of the format, ties to the even
    code, saturating at the largest."""
    rows, K = x.shape
    assert K % 32 == 0
    _, emax, top, ebits, mbits, bias = SUBBYTE_FORMATS[fmt]
    amax = np.abs(x).reshape(rows, K // 32, 32).max(axis=2)
    _, e = np.frexp(amax)
    s = (e - 1 - emax).astype(np.int64)
    s[amax == 0] = 0
    s = np.clip(s, -127, 127)
    y = np.ldexp(x.reshape(rows, K // 32, 32), -s[:, :, None]).reshape(rows, K)
    a = np.minimum(np.abs(y), top)
    _, ea = np.frexp(a)
    binade = np.maximum(ea - 1, 1 - bias)               # exponent of a's binade
    sig = np.rint(np.ldexp(a, mbits - binade)).astype(np.int64)   # ties to even
    carry = sig >= (2 << mbits)                         # rounded up into the next binade
    binade = np.where(carry, binade + 1, binade)
    sig = np.where(carry, sig >> 1, sig)
    normal = sig >= (1 << mbits)
    efield = np.where(normal, binade + bias, 0)
    mfield = np.where(normal, sig - (1 << mbits), sig)
    width = 1 + ebits + mbits
    codes = (np.signbit(y).astype(np.int64) << (width - 1)) | (efield << mbits) | mfield
    packed = pack_fp6(codes) if width == 6 else pack_fp4_padded(codes)
    return packed, (s + 127).astype(np.uint8)


def _quantized_operand8(rng: np.random.Generator, rows: int, K: int, dist: str, fmt: str):
    codes = np.empty((rows, K), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    for r0 in range(0, rows, _ROW_CHUNK):
        r1 = min(rows, r0 + _ROW_CHUNK)
        if dist == "normal":
            x = rng.standard_normal((r1 - r0, K))
        elif dist == "uniform":
            x = rng.uniform(-1.0, 1.0, size=(r1 - r0, K))
        else:
            raise ValueError(dist)
        quant = quantize_rows_fp6 if fmt in SUBBYTE_FORMATS else quantize_rows_fp8
        codes[r0:r1], scales[r0:r1] = quant(x, fmt)
    return codes, scales


def make_problem8(name: str, M: int, N: int, K: int, seed: int, fmt_a: str, fmt_b: str,
                  values: str, alpha: float, beta: float, c_sigma: Optional[float]) -> Problem8:
    """Draw one MXFP8 / MXFP6 problem (A in fmt_a, B in fmt_b)."""
    if K % 32 != 0:
        raise ValueError("K must be a multiple of 32 (one E8M0 scale per 32)")
    if fmt_a not in BYTE_FORMATS or fmt_b not in BYTE_FORMATS:
        raise ValueError("formats are 'e4m3', 'e5m2', 'e2m3', 'e3m2' or 'e2m1'")
    rng = np.random.default_rng(seed)
    A, SA = _quantized_operand8(rng, M, K, values, fmt_a)
    B, SB = _quantized_operand8(rng, N, K, values, fmt_b)
    C = _bf16_normal(rng, M, N, c_sigma) if c_sigma is not None else None
    return Problem8(name, M, N, K, fmt_a, fmt_b, A, B, SA, SB, C, float(alpha), float(beta), seed)


# name -> (M, N, K, seed, fmt A, fmt B, value recipe, alpha, beta, C sigma or None)
WORKLOADS8 = {
    "large8":  (8192, 8192, 8192, 5, "e4m3", "e4m3", "normal", 1.0, 0.0, None),
    "decode8": (1, 8192, 8192, 6, "e4m3", "e4m3", "normal", 1.0, 0.0, None),
    "mixed8":  (512, 1024, 2048, 7, "e4m3", "e5m2", "normal", 0.5, 0.5, 1.0),
    "large6":  (8192, 8192, 8192, 8, "e2m3", "e2m3", "normal", 1.0, 0.0, None),
    "mixed6":  (512, 1024, 2048, 9, "e3m2", "e4m3", "normal", 0.5, 0.5, 1.0),
}


def workload8(name: str) -> Problem8:
    M, N, K, seed, fa, fb, values, alpha, beta, c_sigma = WORKLOADS8[name]
    return make_problem8(name, M, N, K, seed, fa, fb, values, alpha, beta, c_sigma)
