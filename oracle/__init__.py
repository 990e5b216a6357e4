"""CPU oracle for the block-scaled MXFP4 GEMM (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package; the product path never does.

Two independent exact evaluations of

    D[M,N] (bf16) = alpha * A[M,K] (mxfp4) * B[N,K]^T (mxfp4) + beta * C[M,N]

are offered (page "asm_f4gemm -- driving aiter's gfx950 MXFP4 GEMM code
objects", sections "Data layouts" and "Verification"):

* ``gemm`` / ``gemm_sampled``: the plain C oracle in ``oracle.c`` (decode each
  element, accumulate in double in k order, round once to bf16).
* ``dequant`` + ``acc_numpy``: dequantise with numpy from the page's value
  list and ``np.ldexp``, then one float64 matrix product (a library routine
  used as one step).  Both are exact at the test sizes, so their double sums
  agree bit for bit.

``gemm8`` / ``gemm8_sampled`` take 8-bit (E4M3, E5M2) or 6-bit (E2M3, E3M2)
elements with the same scales.

``gemm_nv`` / ``gemm_nv_sampled`` take the same packed E2M1 operands with
one unsigned-E4M3 (UE4M3) scale per 16 K elements (NVFP4), and
``dequant_nv`` + ``acc_numpy_nv`` are its numpy counterpart.

``quantize`` is the oracle of the MXFP4 quantiser (bf16 rows -> packed E2M1
codes + E8M0 scales) that produces the GEMM's operands.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def bind(path: str) -> ctypes.CDLL:
    """Load a compiled copy of oracle.c and declare its signatures."""
    L = ctypes.CDLL(path)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    L.oracle_e2m1_value.restype = ctypes.c_double
    L.oracle_e2m1_value.argtypes = [ctypes.c_uint]
    L.oracle_e8m0_value.restype = ctypes.c_double
    L.oracle_e8m0_value.argtypes = [ctypes.c_uint]
    L.oracle_bf16_rne.restype = ctypes.c_uint16
    L.oracle_bf16_rne.argtypes = [ctypes.c_double]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_fp4_code.restype = ctypes.c_uint
    L.oracle_fp4_code.argtypes = [u8p, ctypes.c_int64]
    L.oracle_host_cores.restype = ctypes.c_int
    L.oracle_host_cores.argtypes = []
    L.oracle_gemm.restype = i64
    L.oracle_gemm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              u8p, i64, u8p, i64, u8p, i64, u8p, i64,
                              ctypes.c_double, ctypes.c_double, u16p, i64,
                              u16p, i64, dp, dp, ctypes.c_int]
    L.oracle_gemm_sampled.restype = i64
    L.oracle_gemm_sampled.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      u8p, i64, u8p, i64, u8p, i64, u8p, i64,
                                      ctypes.c_double, ctypes.c_double, u16p, i64,
                                      ctypes.POINTER(ctypes.c_int64), i64,
                                      u16p, dp, dp, ctypes.c_int]
    L.oracle_fp8_value.restype = ctypes.c_double
    L.oracle_fp8_value.argtypes = [ctypes.c_uint, ctypes.c_int]
    L.oracle_fp6_value.restype = ctypes.c_double
    L.oracle_fp6_value.argtypes = [ctypes.c_uint, ctypes.c_int]
    L.oracle_fp6_code.restype = ctypes.c_uint
    L.oracle_fp6_code.argtypes = [u8p, ctypes.c_int64]
    L.oracle_fp4_padded_code.restype = ctypes.c_uint
    L.oracle_fp4_padded_code.argtypes = [u8p, ctypes.c_int64]
    L.oracle_gemm8.restype = i64
    L.oracle_gemm8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               u8p, i64, u8p, i64, u8p, i64, u8p, i64,
                               ctypes.c_double, ctypes.c_double, u16p, i64,
                               u16p, i64, dp, dp, ctypes.c_int]
    L.oracle_gemm8_sampled.restype = i64
    L.oracle_gemm8_sampled.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, u8p, i64, u8p, i64, u8p, i64, u8p, i64,
                                       ctypes.c_double, ctypes.c_double, u16p, i64,
                                       ctypes.POINTER(ctypes.c_int64), i64,
                                       u16p, dp, dp, ctypes.c_int]
    L.oracle_quantize8.restype = ctypes.c_int
    L.oracle_quantize8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, u16p, i64, u8p, i64,
                                   u8p, i64]
    L.oracle_quantize.restype = ctypes.c_int
    L.oracle_quantize.argtypes = [ctypes.c_int, ctypes.c_int, u16p, i64, u8p, i64, u8p, i64]
    L.oracle_ue4m3_value.restype = ctypes.c_double
    L.oracle_ue4m3_value.argtypes = [ctypes.c_uint]
    L.oracle_gemm_nv.restype = i64
    L.oracle_gemm_nv.argtypes = L.oracle_gemm.argtypes
    L.oracle_gemm_nv_sampled.restype = i64
    L.oracle_gemm_nv_sampled.argtypes = L.oracle_gemm_sampled.argtypes
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def _ptr(a: Optional[np.ndarray], ctype):
    if a is None:
        return ctypes.POINTER(ctype)()
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def e8m0_value(code: int) -> float:
    return lib().oracle_e8m0_value(code)


# MXFP8 / MXFP6 element formats, and E2M1 in the padded form (the codes the
# oracle's fmt arguments take).
E4M3, E5M2, E2M3, E3M2, E2M1P = 1, 2, 3, 4, 5


def fp8_value(code: int, fmt: int) -> float:
    """Value of an 8-bit E4M3 (fmt 1) or E5M2 (fmt 2) element code."""
    return lib().oracle_fp8_value(int(code), int(fmt))


def ue4m3_value(code: int) -> float:
    """Value of an NVFP4 block-scale byte (unsigned E4M3; NaN for 0x7F and
    for bytes with bit 7 set, which are not UE4M3 codes)."""
    return lib().oracle_ue4m3_value(int(code))


def fp6_value(code: int, fmt: int) -> float:
    """Value of a 6-bit E2M3 (fmt 3) or E3M2 (fmt 4) element code."""
    return lib().oracle_fp6_value(int(code), int(fmt))


def fp4_padded_code(row: np.ndarray, k: int) -> int:
    """Code of element k of an E2M1 row in the padded form (16 codes, two per
    byte, in the first 8 of every 16 bytes), as the oracle reads it."""
    r = np.ascontiguousarray(row, dtype=np.uint8)
    return int(lib().oracle_fp4_padded_code(_ptr(r, ctypes.c_uint8), int(k)))


def fp6_code(row: np.ndarray, k: int) -> int:
    """Code of element k of an FP6 row in the padded form (16 codes packed
    little-endian into the first 12 of every 16 bytes), as the oracle reads it."""
    r = np.ascontiguousarray(row, dtype=np.uint8)
    return int(lib().oracle_fp6_code(_ptr(r, ctypes.c_uint8), int(k)))


def fp4_code(packed_row: np.ndarray, k: int) -> int:
    """Code of element k of a packed row, as the oracle unpacks it."""
    row = np.ascontiguousarray(packed_row, dtype=np.uint8)
    return int(lib().oracle_fp4_code(_ptr(row, ctypes.c_uint8), int(k)))


def bf16_rne(x: float) -> int:
    return int(lib().oracle_bf16_rne(float(x)))


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def host_cores() -> int:
    return lib().oracle_host_cores()


def _check_operands(A, B, SA, SB, M, N, K):
    for name, arr, rows, cols in (("A", A, M, K // 2), ("B", B, N, K // 2),
                                  ("SA", SA, M, K // 32), ("SB", SB, N, K // 32)):
        if arr.dtype != np.uint8 or arr.ndim != 2 or arr.shape[0] < rows or arr.shape[1] < cols:
            raise ValueError(f"{name}: bad shape {arr.shape} / dtype {arr.dtype}")


def gemm(A, B, SA, SB, M, N, K, alpha=1.0, beta=0.0, C=None, want_acc=False,
         nthreads=0):
    """Full oracle GEMM. Returns (D bf16 bits [M,N], acc or None, sum|ab| [M,N], inexact)."""
    A, B, SA, SB = (np.ascontiguousarray(x) for x in (A, B, SA, SB))
    _check_operands(A, B, SA, SB, M, N, K)
    Cc = None if beta == 0.0 or C is None else np.ascontiguousarray(C, dtype=np.uint16)
    D = np.zeros((M, N), dtype=np.uint16)
    acc = np.zeros((M, N), dtype=np.float64) if want_acc else None
    sabs = np.zeros((M, N), dtype=np.float64)
    r = lib().oracle_gemm(M, N, K, _ptr(A, ctypes.c_uint8), A.shape[1] * 2,
                          _ptr(B, ctypes.c_uint8), B.shape[1] * 2,
                          _ptr(SA, ctypes.c_uint8), SA.shape[1],
                          _ptr(SB, ctypes.c_uint8), SB.shape[1],
                          float(alpha), float(beta), _ptr(Cc, ctypes.c_uint16),
                          0 if Cc is None else Cc.shape[1],
                          _ptr(D, ctypes.c_uint16), N, _ptr(acc, ctypes.c_double),
                          _ptr(sabs, ctypes.c_double), int(nthreads))
    if r < 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return D, acc, sabs, int(r)


def gemm_sampled(A, B, SA, SB, M, N, K, pairs, alpha=1.0, beta=0.0, C=None,
                 nthreads=0):
    """Oracle at (m, n) pairs [P, 2]. Returns (D bits [P], acc [P], sum|ab| [P], inexact)."""
    A, B, SA, SB = (np.ascontiguousarray(x) for x in (A, B, SA, SB))
    _check_operands(A, B, SA, SB, M, N, K)
    pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    Cc = None if beta == 0.0 or C is None else np.ascontiguousarray(C, dtype=np.uint16)
    P = pairs.shape[0]
    D = np.zeros(P, dtype=np.uint16)
    acc = np.zeros(P, dtype=np.float64)
    sabs = np.zeros(P, dtype=np.float64)
    r = lib().oracle_gemm_sampled(M, N, K, _ptr(A, ctypes.c_uint8), A.shape[1] * 2,
                                  _ptr(B, ctypes.c_uint8), B.shape[1] * 2,
                                  _ptr(SA, ctypes.c_uint8), SA.shape[1],
                                  _ptr(SB, ctypes.c_uint8), SB.shape[1],
                                  float(alpha), float(beta), _ptr(Cc, ctypes.c_uint16),
                                  0 if Cc is None else Cc.shape[1],
                                  pairs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), P,
                                  _ptr(D, ctypes.c_uint16), _ptr(acc, ctypes.c_double),
                                  _ptr(sabs, ctypes.c_double), int(nthreads))
    if r < 0:
        raise ValueError("oracle_gemm_sampled rejected its arguments")
    return D, acc, sabs, int(r)


def _check_operands_nv(A, B, SA, SB, M, N, K):
    for name, arr, rows, cols in (("A", A, M, K // 2), ("B", B, N, K // 2),
                                  ("SA", SA, M, K // 16), ("SB", SB, N, K // 16)):
        if arr.dtype != np.uint8 or arr.ndim != 2 or arr.shape[0] < rows or arr.shape[1] < cols:
            raise ValueError(f"{name}: bad shape {arr.shape} / dtype {arr.dtype}")


def gemm_nv(A, B, SA, SB, M, N, K, alpha=1.0, beta=0.0, C=None, want_acc=False, nthreads=0):
    """Full NVFP4 oracle GEMM (packed E2M1 A, B; UE4M3 scales [rows, K/16]).
    Returns (D bf16 bits [M,N], acc or None, sum|ab| [M,N], inexact)."""
    A, B, SA, SB = (np.ascontiguousarray(x) for x in (A, B, SA, SB))
    _check_operands_nv(A, B, SA, SB, M, N, K)
    Cc = None if beta == 0.0 or C is None else np.ascontiguousarray(C, dtype=np.uint16)
    D = np.zeros((M, N), dtype=np.uint16)
    acc = np.zeros((M, N), dtype=np.float64) if want_acc else None
    sabs = np.zeros((M, N), dtype=np.float64)
    r = lib().oracle_gemm_nv(M, N, K, _ptr(A, ctypes.c_uint8), A.shape[1] * 2,
                             _ptr(B, ctypes.c_uint8), B.shape[1] * 2,
                             _ptr(SA, ctypes.c_uint8), SA.shape[1],
                             _ptr(SB, ctypes.c_uint8), SB.shape[1],
                             float(alpha), float(beta), _ptr(Cc, ctypes.c_uint16),
                             0 if Cc is None else Cc.shape[1],
                             _ptr(D, ctypes.c_uint16), N, _ptr(acc, ctypes.c_double),
                             _ptr(sabs, ctypes.c_double), int(nthreads))
    if r < 0:
        raise ValueError("oracle_gemm_nv rejected its arguments")
    return D, acc, sabs, int(r)


def gemm_nv_sampled(A, B, SA, SB, M, N, K, pairs, alpha=1.0, beta=0.0, C=None, nthreads=0):
    """NVFP4 oracle at (m, n) pairs [P, 2]. Returns (D bits [P], acc [P], sum|ab| [P], inexact)."""
    A, B, SA, SB = (np.ascontiguousarray(x) for x in (A, B, SA, SB))
    _check_operands_nv(A, B, SA, SB, M, N, K)
    pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    Cc = None if beta == 0.0 or C is None else np.ascontiguousarray(C, dtype=np.uint16)
    P = pairs.shape[0]
    D = np.zeros(P, dtype=np.uint16)
    acc = np.zeros(P, dtype=np.float64)
    sabs = np.zeros(P, dtype=np.float64)
    r = lib().oracle_gemm_nv_sampled(M, N, K, _ptr(A, ctypes.c_uint8), A.shape[1] * 2,
                                     _ptr(B, ctypes.c_uint8), B.shape[1] * 2,
                                     _ptr(SA, ctypes.c_uint8), SA.shape[1],
                                     _ptr(SB, ctypes.c_uint8), SB.shape[1],
                                     float(alpha), float(beta), _ptr(Cc, ctypes.c_uint16),
                                     0 if Cc is None else Cc.shape[1],
                                     pairs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), P,
                                     _ptr(D, ctypes.c_uint16), _ptr(acc, ctypes.c_double),
                                     _ptr(sabs, ctypes.c_double), int(nthreads))
    if r < 0:
        raise ValueError("oracle_gemm_nv_sampled rejected its arguments")
    return D, acc, sabs, int(r)


def _check_operands8(A, B, SA, SB, M, N, K, fmt_a, fmt_b):
    fmts = (E4M3, E5M2, E2M3, E3M2, E2M1P)
    if fmt_a not in fmts or fmt_b not in fmts:
        raise ValueError("fmt_a / fmt_b must be E4M3 (1), E5M2 (2), E2M3 (3), E3M2 (4) "
                         "or E2M1P (5)")
    for name, arr, rows, cols in (("A", A, M, K), ("B", B, N, K),
                                  ("SA", SA, M, K // 32), ("SB", SB, N, K // 32)):
        if arr.dtype != np.uint8 or arr.ndim != 2 or arr.shape[0] < rows or arr.shape[1] < cols:
            raise ValueError(f"{name}: bad shape {arr.shape} / dtype {arr.dtype}")


def gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha=1.0, beta=0.0, C=None, want_acc=False,
          nthreads=0):
    """Full MXFP8 / MXFP6 oracle GEMM (A [M, K], B [N, K]: one byte per element;
    FP6 rows in the padded 16-codes-per-16-bytes form).
    Returns (D bf16 bits [M,N], acc or None, sum|ab| [M,N], inexact)."""
    A, B, SA, SB = (np.ascontiguousarray(x) for x in (A, B, SA, SB))
    _check_operands8(A, B, SA, SB, M, N, K, fmt_a, fmt_b)
    Cc = None if beta == 0.0 or C is None else np.ascontiguousarray(C, dtype=np.uint16)
    D = np.zeros((M, N), dtype=np.uint16)
    acc = np.zeros((M, N), dtype=np.float64) if want_acc else None
    sabs = np.zeros((M, N), dtype=np.float64)
    r = lib().oracle_gemm8(M, N, K, int(fmt_a), int(fmt_b), _ptr(A, ctypes.c_uint8), A.shape[1],
                           _ptr(B, ctypes.c_uint8), B.shape[1],
                           _ptr(SA, ctypes.c_uint8), SA.shape[1],
                           _ptr(SB, ctypes.c_uint8), SB.shape[1],
                           float(alpha), float(beta), _ptr(Cc, ctypes.c_uint16),
                           0 if Cc is None else Cc.shape[1],
                           _ptr(D, ctypes.c_uint16), N, _ptr(acc, ctypes.c_double),
                           _ptr(sabs, ctypes.c_double), int(nthreads))
    if r < 0:
        raise ValueError("oracle_gemm8 rejected its arguments")
    return D, acc, sabs, int(r)


def gemm8_sampled(A, B, SA, SB, M, N, K, fmt_a, fmt_b, pairs, alpha=1.0, beta=0.0, C=None,
                  nthreads=0):
    """MXFP8 oracle at (m, n) pairs [P, 2]. Returns (D bits [P], acc [P], sum|ab| [P], inexact)."""
    A, B, SA, SB = (np.ascontiguousarray(x) for x in (A, B, SA, SB))
    _check_operands8(A, B, SA, SB, M, N, K, fmt_a, fmt_b)
    pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    Cc = None if beta == 0.0 or C is None else np.ascontiguousarray(C, dtype=np.uint16)
    P = pairs.shape[0]
    D = np.zeros(P, dtype=np.uint16)
    acc = np.zeros(P, dtype=np.float64)
    sabs = np.zeros(P, dtype=np.float64)
    r = lib().oracle_gemm8_sampled(M, N, K, int(fmt_a), int(fmt_b), _ptr(A, ctypes.c_uint8),
                                   A.shape[1], _ptr(B, ctypes.c_uint8), B.shape[1],
                                   _ptr(SA, ctypes.c_uint8), SA.shape[1],
                                   _ptr(SB, ctypes.c_uint8), SB.shape[1],
                                   float(alpha), float(beta), _ptr(Cc, ctypes.c_uint16),
                                   0 if Cc is None else Cc.shape[1],
                                   pairs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), P,
                                   _ptr(D, ctypes.c_uint16), _ptr(acc, ctypes.c_double),
                                   _ptr(sabs, ctypes.c_double), int(nthreads))
    if r < 0:
        raise ValueError("oracle_gemm8_sampled rejected its arguments")
    return D, acc, sabs, int(r)


# --- second exact evaluation: numpy dequantisation + one float64 product ----

_E2M1_LIST = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def dequant(packed: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    """float64 [rows, K] values: page value list x 2^(e-127) per 1x32 block."""
    packed = np.asarray(packed, dtype=np.uint8)[:, : K // 2]
    codes = np.empty((packed.shape[0], K), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    mag = _E2M1_LIST[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    e = np.asarray(scales, dtype=np.int64)[:, : K // 32]
    sc = np.where(e == 255, np.nan, np.ldexp(1.0, (e - 127).astype(np.int32)))
    return val * np.repeat(sc, 32, axis=1)


def acc_numpy(A, B, SA, SB, K) -> np.ndarray:
    """sum_k a(m,k) b(n,k) as one float64 matmul of the dequantised operands."""
    return dequant(A, SA, K) @ dequant(B, SB, K).T


def ue4m3_table() -> np.ndarray:
    """float64 [256]: UE4M3 byte -> value from its bit fields (exponent bits
    6..3, bias 7, mantissa bits 2..0; exponent 0 subnormal); 0x7F and every
    byte with bit 7 set -> NaN."""
    c = np.arange(256)
    e = (c >> 3) & 15
    m = c & 7
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    return np.where((c >= 0x7F), np.nan, v)


def dequant_nv(packed: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    """float64 [rows, K] values: E2M1 value list x the UE4M3 scale of each 1x16 block."""
    packed = np.asarray(packed, dtype=np.uint8)[:, : K // 2]
    codes = np.empty((packed.shape[0], K), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    mag = _E2M1_LIST[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    sc = ue4m3_table()[np.asarray(scales, dtype=np.uint8)[:, : K // 16]]
    return val * np.repeat(sc, 16, axis=1)


def acc_numpy_nv(A, B, SA, SB, K) -> np.ndarray:
    """NVFP4 sum_k a(m,k) b(n,k) as one float64 matmul of the dequantised operands."""
    return dequant_nv(A, SA, K) @ dequant_nv(B, SB, K).T


def quantize(X_bits, rows, K):
    """MXFP4 quantisation of bf16 rows (see oracle.c): returns (packed codes
    uint8 [rows, K/2], scale codes uint8 [rows, K/32])."""
    X = np.ascontiguousarray(X_bits, dtype=np.uint16)
    if X.ndim != 2 or X.shape[0] < rows or X.shape[1] < K:
        raise ValueError(f"X: bad shape {X.shape}")
    Q = np.zeros((rows, K // 2), dtype=np.uint8)
    S = np.zeros((rows, K // 32), dtype=np.uint8)
    r = lib().oracle_quantize(rows, K, _ptr(X, ctypes.c_uint16), X.shape[1],
                              _ptr(Q, ctypes.c_uint8), K // 2, _ptr(S, ctypes.c_uint8), K // 32)
    if r != 0:
        raise ValueError("oracle_quantize rejected the sizes")
    return Q, S


def quantize8(X_bits, rows, K, fmt, fill=0):
    """MXFP8 quantiser (fmt E4M3 / E5M2, or E2M3 / E3M2 / E2M1P into the
    padded 16-per-16-bytes forms): bf16 bits [rows, K] -> (bytes uint8
    [rows, K], E8M0 scales uint8 [rows, K/32])."""
    X = np.ascontiguousarray(X_bits, dtype=np.uint16)
    Q = np.full((rows, K), fill, dtype=np.uint8)       # fill: what the output held before
    S = np.zeros((rows, K // 32), dtype=np.uint8)
    r = lib().oracle_quantize8(rows, K, int(fmt), _ptr(X, ctypes.c_uint16), X.shape[1],
                               _ptr(Q, ctypes.c_uint8), K, _ptr(S, ctypes.c_uint8), K // 32)
    if r != 0:
        raise ValueError("oracle_quantize8 rejected its arguments")
    return Q, S
