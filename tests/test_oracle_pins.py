"""Pins for the CPU oracle: things the pages and the mathematics fix.

Every check here compares the oracle with something other than itself:
golden values the page prints, closed forms, a brute force in exact rational
arithmetic with its own decode and its own rounding search, and a library
float64 matrix product.  ``test_oracle_mutants`` then plants plausible
mistakes in copies of oracle.c and shows that each one fails a check.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --- exact references written from the format definitions -----------------

def page_e2m1_values():
    """E2M1 code -> Fraction, from the page's value list (golden fixture)."""
    return {int(c): Fraction(v) if v not in ("-0.0",) else Fraction(0)
            for c, v in read_golden("e2m1_values.txt")}


def bf16_bits_to_fraction(bits):
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    v = Fraction(f, 2 ** 133) if e == 0 else Fraction(128 + f) * Fraction(2) ** (e - 134)
    return -v if bits & 0x8000 else v


_BF16_POS = None


def bf16_positive_table():
    """Every non-negative finite bf16 value in increasing order, with its bits."""
    global _BF16_POS
    if _BF16_POS is None:
        _BF16_POS = [(bf16_bits_to_fraction(b), b) for b in range(0x7F80)]
    return _BF16_POS


def bf16_rne_by_search(y: Fraction) -> int:
    """Nearest bf16 to an exact rational by searching the value set; ties to
    the neighbour with an even bit pattern; beyond the largest finite value
    by half a spacing -> infinity."""
    table = bf16_positive_table()
    a = abs(y)
    sign = 0x8000 if y < 0 else 0
    top = table[-1][0]
    half_gap = (top - table[-2][0]) / 2
    if a >= top + half_gap:
        return sign | 0x7F80
    lo, hi = 0, len(table) - 1
    while lo < hi:                      # first entry >= a
        mid = (lo + hi) // 2
        if table[mid][0] < a:
            lo = mid + 1
        else:
            hi = mid
    v_hi, b_hi = table[lo]
    if v_hi == a or lo == 0:
        return sign | b_hi
    v_lo, b_lo = table[lo - 1]
    d_lo, d_hi = a - v_lo, v_hi - a
    if d_lo < d_hi:
        return sign | b_lo
    if d_hi < d_lo:
        return sign | b_hi
    return sign | (b_lo if b_lo % 2 == 0 else b_hi)


def page_decode_row(packed_row, K):
    """Codes of a packed row per the page: element 2i low nibble, 2i+1 high."""
    codes = []
    for i in range(K // 2):
        byte = int(packed_row[i])
        codes.append(byte & 0xF)
        codes.append(byte >> 4)
    return codes


def brute_force_gemm(A, B, SA, SB, M, N, K, alpha, beta, C):
    """Exact rational D (as bf16 bits) from the definition, pure Python."""
    vals = page_e2m1_values()
    two = Fraction(2)
    ra = [page_decode_row(A[m], K) for m in range(M)]
    rb = [page_decode_row(B[n], K) for n in range(N)]
    D = np.zeros((M, N), dtype=np.uint16)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = vals[ra[m][k]] * two ** (int(SA[m, k // 32]) - 127)
                b = vals[rb[n][k]] * two ** (int(SB[n, k // 32]) - 127)
                acc += a * b
            y = Fraction(alpha) * acc
            if beta != 0.0:
                y += Fraction(beta) * bf16_bits_to_fraction(int(C[m, n]))
            D[m, n] = bf16_rne_by_search(y)
    return D


def same_value(d1, d2):
    """bf16 bit arrays equal by value (+0 == -0)."""
    d1 = np.asarray(d1, dtype=np.uint16)
    d2 = np.asarray(d2, dtype=np.uint16)
    z1 = (d1 & 0x7FFF) == 0
    z2 = (d2 & 0x7FFF) == 0
    return bool(np.all((d1 == d2) | (z1 & z2)))


def bf16_to_f64(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def random_case(rng, M, N, K, scale_lo=120, scale_hi=134):
    A = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    SA = rng.integers(scale_lo, scale_hi + 1, size=(M, K // 32)).astype(np.uint8)
    SB = rng.integers(scale_lo, scale_hi + 1, size=(N, K // 32)).astype(np.uint8)
    # C: bf16 with exponents 2^-8 .. 2^8 (fields 119..135), either sign, so
    # that alpha * acc + beta * C stays exact in double at these sizes.
    e = rng.integers(119, 136, size=(M, N)).astype(np.uint16)
    f = rng.integers(0, 128, size=(M, N)).astype(np.uint16)
    sgn = rng.integers(0, 2, size=(M, N)).astype(np.uint16)
    C = (sgn << 15) | (e << 7) | f
    return A, B, SA, SB, C


# --- check functions (shared with the mutant test) -------------------------

def check_e2m1_golden(o):
    for code, v in read_golden("e2m1_values.txt"):
        got = o.e2m1_value(int(code))
        assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v)), code


def check_e2m1_bitfields(o):
    # OCP E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0;
    # exponent 0 is subnormal: m * 0.5.
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        v = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert o.e2m1_value(code) == (-v if s else v)


def check_e8m0(o):
    for code, v in read_golden("e8m0_values.txt"):
        got = o.e8m0_value(int(code, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v), code
    for e in range(1, 255):
        assert o.e8m0_value(e) == math.ldexp(1.0, e - 127)


def check_nibble_order(o):
    for byte, even, odd in read_golden("nibble_order.txt"):
        row = np.array([0x00, int(byte, 16), 0x00], dtype=np.uint8)
        assert o.fp4_code(row, 2) == int(even)
        assert o.fp4_code(row, 3) == int(odd)


def check_bf16_golden(o):
    for hx, bits, *_ in read_golden("bf16_rounding.txt"):
        assert o.bf16_rne(float.fromhex(hx)) == int(bits, 16), hx


def check_bf16_roundtrip(o):
    for b in range(0, 0x10000, 7):
        if (b & 0x7F80) == 0x7F80 and (b & 0x7F):
            continue                                 # NaN patterns
        assert o.bf16_rne(o.bf16_to_double(b)) == b, hex(b)


def check_bf16_midpoints(o, n=3000):
    rng = np.random.default_rng(11)
    for b in rng.integers(1, 0x7F7F, size=n):
        b = int(b)
        lo, hi = bf16_bits_to_fraction(b), bf16_bits_to_fraction(b + 1)
        mid = (lo + hi) / 2
        want = b if b % 2 == 0 else b + 1
        assert o.bf16_rne(float(mid)) == want
        eps = (hi - lo) / 1024
        assert o.bf16_rne(float(mid - eps)) == b
        assert o.bf16_rne(float(mid + eps)) == b + 1


def check_identity(o):
    from block_scaled_mxfp4_gb300 import inputs
    p = inputs.identity_problem()
    D, _, _, inexact = o.gemm(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K)
    assert inexact == 0
    vals = page_e2m1_values()
    for m in range(p.M):
        codes = page_decode_row(p.A[m], p.K)
        want = np.array([float(vals[codes[n]]) for n in range(p.N)])
        assert np.array_equal(bf16_to_f64(D[m]), want), m


def check_identity_scaled(o):
    # B = I with unit scales, A with random scales: D[m,n] = a(m, n) exactly.
    from block_scaled_mxfp4_gb300 import inputs
    rng = np.random.default_rng(5)
    p = inputs.identity_problem(M=8, N=64, K=64, seed=5)
    SA = rng.integers(120, 135, size=(8, 2)).astype(np.uint8)
    D, _, _, _ = o.gemm(p.A, p.B, SA, p.SB, 8, 64, 64)
    vals = page_e2m1_values()
    for m in range(8):
        codes = page_decode_row(p.A[m], 64)
        want = [float(vals[codes[n]] * Fraction(2) ** (int(SA[m, n // 32]) - 127))
                for n in range(64)]
        assert np.array_equal(bf16_to_f64(D[m]), np.array(want))


def check_alpha_beta(o):
    rng = np.random.default_rng(3)
    M, N, K = 6, 10, 64
    A, B, SA, SB, C = random_case(rng, M, N, K)
    zeroA = np.zeros_like(A)
    # A = 0: D = round(beta * C); beta = 2^-1 keeps it exact.
    D, _, _, _ = o.gemm(zeroA, B, SA, SB, M, N, K, alpha=1.0, beta=0.5, C=C)
    want = np.array([[o.bf16_rne(0.5 * o.bf16_to_double(int(c))) for c in row] for row in C])
    assert same_value(D, want)
    # alpha = 0, beta = 1: D = C.
    D, _, _, _ = o.gemm(A, B, SA, SB, M, N, K, alpha=0.0, beta=1.0, C=C)
    assert same_value(D, C)
    # D(alpha = 2^j) = 2^j * D(alpha = 1) away from overflow / subnormals.
    D1, acc, _, _ = o.gemm(A, B, SA, SB, M, N, K, alpha=1.0, want_acc=True)
    D8, _, _, _ = o.gemm(A, B, SA, SB, M, N, K, alpha=8.0)
    assert np.array_equal(bf16_to_f64(D8), 8.0 * bf16_to_f64(D1))
    # beta = 0 never reads C, even if it holds NaN.
    Cnan = np.full((M, N), 0x7FC0, dtype=np.uint16)
    D0, _, _, _ = o.gemm(A, B, SA, SB, M, N, K, alpha=1.0, beta=0.0, C=Cnan)
    assert same_value(D0, D1)
    # beta = 1, alpha = 1 adds C (exact here): D = round(acc + C).
    D2, _, _, inexact = o.gemm(A, B, SA, SB, M, N, K, alpha=1.0, beta=1.0, C=C)
    want = np.array([[o.bf16_rne(acc[m, n] + o.bf16_to_double(int(C[m, n])))
                      for n in range(N)] for m in range(M)])
    assert same_value(D2, want)


def check_brute_force(o, cases=24):
    rng = np.random.default_rng(2024)
    shapes = [(1, 1, 32), (2, 3, 64), (3, 2, 96), (4, 4, 32), (1, 4, 128), (4, 1, 64)]
    for i in range(cases):
        M, N, K = shapes[i % len(shapes)]
        A, B, SA, SB, C = random_case(rng, M, N, K)
        alpha = [1.0, 0.5, -2.0, 0.75][i % 4]
        beta = [0.0, 1.0, 0.5, -0.25][(i // 4) % 4]
        D, _, _, inexact = o.gemm(A, B, SA, SB, M, N, K, alpha=alpha, beta=beta, C=C)
        assert inexact == 0, (i, M, N, K)
        want = brute_force_gemm(A, B, SA, SB, M, N, K, alpha, beta, C)
        assert same_value(D, want), (i, M, N, K)


def check_all_code_pairs(o):
    # K = 32: A row m holds code ca at k = 0, B row n holds code cb at k = 0;
    # every (ca, cb) pair and several scale pairs; D = round(va*vb*2^(ea+eb-254)).
    vals = page_e2m1_values()
    M = N = 16
    K = 32
    A = np.zeros((M, K // 2), dtype=np.uint8)
    B = np.zeros((N, K // 2), dtype=np.uint8)
    A[:, 0] = np.arange(16, dtype=np.uint8)          # element 0 = code m
    B[:, 0] = np.arange(16, dtype=np.uint8)
    for ea, eb in ((127, 127), (125, 131), (140, 100), (1, 254), (60, 60)):
        SA = np.full((M, 1), ea, dtype=np.uint8)
        SB = np.full((N, 1), eb, dtype=np.uint8)
        D, _, _, _ = o.gemm(A, B, SA, SB, M, N, K)
        for ca in range(16):
            for cb in range(16):
                y = vals[ca] * vals[cb] * Fraction(2) ** (ea + eb - 254)
                assert same_value([D[ca, cb]], [bf16_rne_by_search(y)]), (ca, cb, ea, eb)


def check_numpy_crosscheck(o):
    from block_scaled_mxfp4_gb300 import inputs
    for name in ("tiny",):
        p = inputs.workload(name)
        _, acc, _, inexact = o.gemm(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K, want_acc=True)
        assert inexact == 0
        assert np.array_equal(acc, o.acc_numpy(p.A, p.B, p.SA, p.SB, p.K))
    rng = np.random.default_rng(9)
    A, B, SA, SB, _ = random_case(rng, 37, 29, 320)
    _, acc, _, inexact = o.gemm(A, B, SA, SB, 37, 29, 320, want_acc=True)
    assert inexact == 0
    assert np.array_equal(acc, o.acc_numpy(A, B, SA, SB, 320))


def check_rounding_is_only_error(o):
    # The page reports max_rel_err 0.003891 without split-K: one bf16
    # rounding of the exact result, whose worst case is 1/257.
    (_, page_val), = read_golden("verification_error.txt")
    worst = Fraction(1, 257)
    assert round(float(worst), 6) == float(page_val)
    x = 1.0 + 2.0 ** -8
    assert abs(o.bf16_to_double(o.bf16_rne(x)) - x) / x == float(worst)
    rng = np.random.default_rng(21)
    A, B, SA, SB, _ = random_case(rng, 24, 40, 256)
    D, acc, _, _ = o.gemm(A, B, SA, SB, 24, 40, 256, want_acc=True)
    nz = acc != 0
    rel = np.abs(bf16_to_f64(D)[nz] - acc[nz]) / np.abs(acc[nz])
    assert rel.max() <= float(worst)


def check_sampled_matches_full(o):
    rng = np.random.default_rng(4)
    M, N, K = 9, 13, 96
    A, B, SA, SB, C = random_case(rng, M, N, K)
    D, acc, sabs, _ = o.gemm(A, B, SA, SB, M, N, K, alpha=0.5, beta=1.0, C=C, want_acc=True)
    pairs = np.array([(m, n) for m in range(M) for n in range(N)])[::3]
    Ds, accs, sabss, _ = o.gemm_sampled(A, B, SA, SB, M, N, K, pairs, alpha=0.5, beta=1.0, C=C)
    assert np.array_equal(Ds, D[pairs[:, 0], pairs[:, 1]])
    assert np.array_equal(accs, acc[pairs[:, 0], pairs[:, 1]])
    assert np.array_equal(sabss, sabs[pairs[:, 0], pairs[:, 1]])


def check_gemm_single_rounding(o):
    # Three 32-blocks whose products sum to 1 + 2^-8 + 2^-26: just above the
    # bf16 tie between 1 and 1 + 2^-7, so one rounding gives 1 + 2^-7, while
    # a float intermediate would land on the tie and give 1.0.
    K = 96
    A = np.zeros((1, K // 2), dtype=np.uint8)
    B = np.zeros((1, K // 2), dtype=np.uint8)
    for blk in range(3):
        A[0, blk * 16] = 0x02                 # element 32*blk = 1.0
        B[0, blk * 16] = 0x02
    SA = np.array([[127, 119, 114]], dtype=np.uint8)
    SB = np.array([[127, 127, 114]], dtype=np.uint8)
    D, acc, _, inexact = o.gemm(A, B, SA, SB, 1, 1, K, want_acc=True)
    exact = Fraction(1) + Fraction(1, 2 ** 8) + Fraction(1, 2 ** 26)
    assert inexact == 0 and acc[0, 0] == float(exact)
    assert int(D[0, 0]) == bf16_rne_by_search(exact) == 0x3F81


# ------------------------------------------------------------- quantiser --

def _bf16_bits(values):
    from block_scaled_mxfp4_gb300 import inputs
    return inputs.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


def check_quant_golden(o):
    rows = read_golden("quantize_rounding.txt")
    for x, code in rows:
        blk = np.zeros((1, 32), dtype=np.float32)
        blk[0, 0] = 6.0                      # block max 6 -> scale exponent 0
        blk[0, 1] = float(x)
        Q, S = o.quantize(_bf16_bits(blk), 1, 32)
        assert S[0, 0] == 127, (x, S[0, 0])
        got = int(Q[0, 0] >> 4)              # element 1: high nibble of byte 0
        assert got == int(code), (x, got, code)


def check_quant_scale_rule(o):
    # 6 * 2^s <= amax < 6 * 2^(s+1) for every block (s = code - 127), s = 0
    # for an all-zero block, and the clamp at +-127.
    rng = np.random.default_rng(7)
    rows, K = 24, 256
    x = rng.standard_normal((rows, K)) * np.ldexp(1.0, rng.integers(-60, 60, size=(rows, 1)))
    x[3, 32:64] = 0.0
    x[5, :32] = np.ldexp(1.0, -133)          # tiny: clamps to s = -127
    x[6, :32] = 5.9375                       # bf16-exact, just below 6
    x[7, :32] = 6.0
    x[8, :32] = -12.0
    bits = _bf16_bits(x)
    Q, S = o.quantize(bits, rows, K)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for r in range(rows):
        for b in range(K // 32):
            amax = float(np.max(np.abs(xv[r, 32 * b:32 * b + 32])))
            s = int(S[r, b]) - 127
            if amax == 0.0:
                assert s == 0
            elif s == -127:
                assert amax < 6.0 * 2.0 ** -126
            else:
                assert 6.0 * 2.0 ** s <= amax < 6.0 * 2.0 ** (s + 1), (r, b, amax, s)
    assert S[6, 0] == 126 and S[7, 0] == 127 and S[8, 0] == 128


def check_quant_nearest_brute_force(o):
    # Every element's code is the nearest of the 16 E2M1 values to x / 2^s
    # (exact rational distances), ties to the even code, saturating at 6,
    # with the sign of x.
    from fractions import Fraction
    rng = np.random.default_rng(8)
    rows, K = 6, 128
    x = rng.standard_normal((rows, K)) * 3.0
    x[0, :8] = [0.25, -0.25, 2.5, -3.5, 5.0, 0.75, -0.0, 0.0]
    bits = _bf16_bits(x)
    Q, S = o.quantize(bits, rows, K)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mags = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    for r in range(rows):
        for k in range(K):
            s = int(S[r, k // 32]) - 127
            y = abs(Fraction(xv[r, k])) / Fraction(2) ** s
            if y >= 6:
                want = 7
            else:
                d = [abs(y - m) for m in mags]
                best = min(d)
                cands = [c for c in range(8) if d[c] == best]
                want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
            if np.signbit(xv[r, k]):
                want |= 8
            byte = int(Q[r, k // 2])
            got = (byte >> 4) if k % 2 else (byte & 0xF)
            assert got == want, (r, k, xv[r, k], s, got, want)


def check_quant_matches_generator(o):
    # The package's input generator implements the same rule independently
    # (numpy); on bf16-representable data both give the same bytes.
    from block_scaled_mxfp4_gb300 import inputs
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((40, 512)) * np.ldexp(1.0, rng.integers(-8, 8, size=(40, 1))))
    bits = _bf16_bits(x)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Qg, Sg = inputs.quantize_rows(xv)
    Qo, So = o.quantize(bits, 40, 512)
    assert np.array_equal(So, Sg)
    assert np.array_equal(Qo, Qg)


# --- MXFP8 (E4M3 / E5M2 elements, E8M0 per 32) -----------------------------

def fp8_fraction(code, fmt):
    """Exact value of an 8-bit code from the format's field widths (test-side
    decoder): E4M3 = 1/4/3 bits, bias 7; E5M2 = 1/5/2 bits, bias 15.  Returns
    None for the NaN / infinity codes."""
    mbits, ebits, bias = (3, 4, 7) if fmt == 1 else (2, 5, 15)
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if fmt == 1 and e == 15 and m == 7:
        return None
    if fmt == 2 and e == 31:
        return None
    if e == 0:
        v = Fraction(m, 2 ** mbits) * Fraction(2) ** (1 - bias)
    else:
        v = (1 + Fraction(m, 2 ** mbits)) * Fraction(2) ** (e - bias)
    return -v if code & 0x80 else v


def fp8_torch_decode(codes, fmt):
    import torch
    dt = torch.float8_e4m3fn if fmt == 1 else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(dt).double().numpy()


def random_case8(rng, M, N, K, fmt_a, fmt_b, scale_lo=124, scale_hi=130):
    """Random codes of each format with magnitudes in [2^-4, 2^5) (plus
    zeros and, for E4M3, subnormals), scales near 1, C with exponents
    2^-8 .. 2^8: exact in double at these sizes.  (Codes spanning a whole
    format would not be: E5M2 alone spans 2^-16 .. 2^15.8.)"""
    def finite_codes(fmt, shape):
        mbits, bias = (3, 7) if fmt == 1 else (2, 15)
        e = rng.integers(bias - 4, bias + 5, size=shape)
        m = rng.integers(0, 1 << mbits, size=shape)
        c = (e << mbits) | m
        kind = rng.random(shape)
        c = np.where(kind < 0.08, 0, c)
        if fmt == 1:
            c = np.where((kind >= 0.08) & (kind < 0.14), m, c)      # subnormals
        c = c | (rng.integers(0, 2, size=shape) << 7)
        return c.astype(np.uint8)
    A = finite_codes(fmt_a, (M, K))
    B = finite_codes(fmt_b, (N, K))
    SA = rng.integers(scale_lo, scale_hi + 1, size=(M, K // 32)).astype(np.uint8)
    SB = rng.integers(scale_lo, scale_hi + 1, size=(N, K // 32)).astype(np.uint8)
    e = rng.integers(119, 136, size=(M, N)).astype(np.uint16)
    f = rng.integers(0, 128, size=(M, N)).astype(np.uint16)
    sgn = rng.integers(0, 2, size=(M, N)).astype(np.uint16)
    C = (sgn << 15) | (e << 7) | f
    return A, B, SA, SB, C


def check_fp8_golden(o):
    for fmt, code, v in read_golden("fp8_values.txt"):
        got = o.fp8_value(int(code, 16), int(fmt))
        if v == "nan":
            assert got != got, (fmt, code)
        elif v in ("inf", "-inf"):
            assert got == float(v), (fmt, code, got)
        else:
            assert got == float(v) and math.copysign(1.0, got) == math.copysign(1.0, float(v)), \
                (fmt, code, got, v)


def check_fp8_all_codes(o):
    """Every code of both formats: the oracle's decode equals the test-side
    field decoder and torch's float8 decoding (NaN and infinity included)."""
    codes = np.arange(256, dtype=np.uint8)
    for fmt in (1, 2):
        ref = fp8_torch_decode(codes.reshape(1, -1), fmt)[0]
        for c in range(256):
            got = o.fp8_value(c, fmt)
            want = fp8_fraction(c, fmt)
            if want is None:
                assert (got != got and ref[c] != ref[c]) or (math.isinf(got) and got == ref[c]), (fmt, c)
            else:
                assert math.isfinite(got) and Fraction(got) == want and got == ref[c], \
                    (fmt, c, got, want, ref[c])


def brute_force_gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha, beta, C):
    two = Fraction(2)
    D = np.zeros((M, N), dtype=np.uint16)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = fp8_fraction(int(A[m, k]), fmt_a) * two ** (int(SA[m, k // 32]) - 127)
                b = fp8_fraction(int(B[n, k]), fmt_b) * two ** (int(SB[n, k // 32]) - 127)
                acc += a * b
            y = Fraction(alpha) * acc
            if beta != 0.0:
                y += Fraction(beta) * bf16_bits_to_fraction(int(C[m, n]))
            D[m, n] = bf16_rne_by_search(y)
    return D


def check_fp8_brute_force(o, cases=8):
    rng = np.random.default_rng(81)
    for i in range(cases):
        fmt_a, fmt_b = [(1, 1), (1, 2), (2, 1), (2, 2)][i % 4]
        M, N, K = 3, 4, 64
        A, B, SA, SB, C = random_case8(rng, M, N, K, fmt_a, fmt_b)
        alpha, beta = [(1.0, 0.0), (0.5, 0.25), (-2.0, 1.0), (0.75, -0.5)][i % 4]
        D, _, _, inexact = o.gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha=alpha, beta=beta, C=C)
        assert inexact == 0
        want = brute_force_gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha, beta, C)
        assert same_value(D, want), (i, D, want)


def check_fp8_torch_crosscheck(o):
    """The exact double sum equals one float64 matmul of torch-decoded,
    scaled operands (exact at these sizes)."""
    rng = np.random.default_rng(82)
    for fmt_a, fmt_b in ((1, 1), (2, 1)):
        M, N, K = 24, 40, 256
        A, B, SA, SB, _ = random_case8(rng, M, N, K, fmt_a, fmt_b)
        _, acc, _, inexact = o.gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, want_acc=True)
        assert inexact == 0
        sa = np.repeat(np.ldexp(1.0, SA.astype(np.int64) - 127), 32, axis=1)
        sb = np.repeat(np.ldexp(1.0, SB.astype(np.int64) - 127), 32, axis=1)
        ref = (fp8_torch_decode(A, fmt_a) * sa) @ (fp8_torch_decode(B, fmt_b) * sb).T
        assert np.array_equal(acc, ref)


def check_fp8_identity(o):
    """B = I (E4M3 1.0 = 0x38, all scales 1): D is A's values, which bf16
    holds exactly (3 mantissa bits), scaled by A's block scale."""
    rng = np.random.default_rng(83)
    M, N, K = 16, 64, 96
    A, _, SA, _, _ = random_case8(rng, M, N, K, 1, 1, 125, 129)
    B = np.zeros((N, K), dtype=np.uint8)
    idx = np.arange(min(N, K))
    B[idx, idx] = 0x38
    SB = np.full((N, K // 32), 127, dtype=np.uint8)
    D, _, _, inexact = o.gemm8(A, B, SA, SB, M, N, K, 1, 1)
    assert inexact == 0
    vals = fp8_torch_decode(A[:, :N], 1) * np.ldexp(1.0, SA[:, np.arange(N) // 32].astype(np.int64) - 127)
    want = (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert same_value(D, want)


def check_fp8_sampled_matches_full(o):
    rng = np.random.default_rng(84)
    M, N, K = 20, 30, 128
    A, B, SA, SB, C = random_case8(rng, M, N, K, 2, 1)
    D, _, _, _ = o.gemm8(A, B, SA, SB, M, N, K, 2, 1, alpha=0.5, beta=1.0, C=C)
    pairs = np.stack([rng.integers(0, M, 50), rng.integers(0, N, 50)], axis=1)
    Ds, _, _, _ = o.gemm8_sampled(A, B, SA, SB, M, N, K, 2, 1, pairs, alpha=0.5, beta=1.0, C=C)
    assert np.array_equal(Ds, D[pairs[:, 0], pairs[:, 1]])


def check_fp8_exactness_flag(o):
    """E5M2 products from 57344^2 (~2^31.6) down to (2^-16)^2 = 2^-32 in one
    sum: sum|ab| / granule exceeds 2^52, which the oracle must report; a row
    of moderate values must not be flagged."""
    K = 64
    A = np.zeros((2, K), dtype=np.uint8)
    B = np.zeros((1, K), dtype=np.uint8)
    A[0, 0], A[0, 1] = 0x7B, 0x01          # 57344 and 2^-16
    B[0, 0], B[0, 1] = 0x7B, 0x01
    A[1, :4] = 0x3C                        # 1.0
    B[0, 2:6] = 0x3D                       # 1.25
    S = np.full((2, K // 32), 127, dtype=np.uint8)
    _, _, _, inexact = o.gemm8(A, B, S, S[:1], 2, 1, K, 2, 2)
    assert inexact == 1, inexact


def check_quant8_golden(o):
    for fmt, bmax, x, code in read_golden("quantize8_rounding.txt"):
        blk = np.zeros((1, 32), dtype=np.float64)
        blk[0, 0] = float(bmax)
        blk[0, 1] = float(x)
        Q, S = o.quantize8(_bf16_bits(blk), 1, 32, int(fmt))
        assert S[0, 0] == 127, (fmt, x, S[0, 0])
        assert int(Q[0, 1]) == int(code, 16), (fmt, x, hex(Q[0, 1]), code)


def check_quant8_scale_rule(o):
    # 2^(s + emax) <= amax < 2^(s + emax + 1), s = 0 for an all-zero block,
    # and the clamps at -127 / 127.
    rng = np.random.default_rng(17)
    rows, K = 20, 256
    x = rng.standard_normal((rows, K)) * np.ldexp(1.0, rng.integers(-70, 70, size=(rows, 1)))
    x[3, 32:64] = 0.0
    x[5, :32] = np.ldexp(1.0, -133)
    x[6, :32] = 255.0                        # bf16-exact, just below 256: s = -1 for E4M3
    bits = _bf16_bits(x)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for fmt, emax in ((1, 8), (2, 15)):
        Q, S = o.quantize8(bits, rows, K, fmt)
        for r in range(rows):
            for b in range(K // 32):
                amax = float(np.max(np.abs(xv[r, 32 * b:32 * b + 32])))
                s = int(S[r, b]) - 127
                if amax == 0.0:
                    assert s == 0
                elif s == -127:
                    assert amax < 2.0 ** (-126 + emax)
                else:
                    assert 2.0 ** (s + emax) <= amax < 2.0 ** (s + emax + 1), (fmt, r, b, amax, s)


def check_quant8_nearest_brute_force(o):
    # Every code is the nearest finite value of the format to |x| / 2^s
    # (exact rational distances over all codes), ties to the even code,
    # saturating at the largest finite value, with the sign of x.
    rng = np.random.default_rng(18)
    rows, K = 4, 96
    x = rng.standard_normal((rows, K)) * 5.0
    x[0, :6] = [0.0, -0.0, 1.0625, -3.0, 1e-3, 250.0]
    bits = _bf16_bits(x)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for fmt in (1, 2):
        top = 0x7E if fmt == 1 else 0x7B
        vals = [fp8_fraction(c, fmt) for c in range(top + 1)]
        Q, S = o.quantize8(bits, rows, K, fmt)
        for r in range(rows):
            for k in range(K):
                s = int(S[r, k // 32]) - 127
                y = abs(Fraction(xv[r, k])) / Fraction(2) ** s
                if y >= vals[top]:
                    want = top
                else:
                    d = [abs(y - v) for v in vals]
                    best = min(d)
                    cands = [c for c in range(top + 1) if d[c] == best]
                    want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
                if np.signbit(xv[r, k]):
                    want |= 0x80
                assert int(Q[r, k]) == want, (fmt, r, k, xv[r, k], s, hex(Q[r, k]), hex(want))


def check_quant8_matches_generator(o):
    # The input generator's MXFP8 rule (numpy scale + torch's float8 cast,
    # an independent implementation) gives the same bytes on bf16 data.
    from block_scaled_mxfp4_gb300 import inputs
    rng = np.random.default_rng(19)
    x = rng.standard_normal((16, 512)) * np.ldexp(1.0, rng.integers(-8, 8, size=(16, 1)))
    bits = _bf16_bits(x)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for name, fmt in (("e4m3", 1), ("e5m2", 2)):
        Qg, Sg = inputs.quantize_rows_fp8(xv, name)
        Qo, So = o.quantize8(bits, 16, 512, fmt)
        assert np.array_equal(So, Sg)
        assert np.array_equal(Qo, Qg)


# --- MXFP6 (E2M3 / E3M2 elements, 16 codes per 16 bytes, E8M0 per 32) -----

def fp6_fraction(code, fmt):
    """Exact value of a 6-bit code from the format's field widths (test-side
    decoder): E2M3 = 1/2/3 bits, bias 1; E3M2 = 1/3/2 bits, bias 3."""
    ebits, mbits, bias = (2, 3, 1) if fmt == 3 else (3, 2, 3)
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if e == 0:
        v = Fraction(m, 2 ** mbits) * Fraction(2) ** (1 - bias)
    else:
        v = (1 + Fraction(m, 2 ** mbits)) * Fraction(2) ** (e - bias)
    return -v if code & 0x20 else v


def pack_fp6(codes, pad=None):
    """Test-side packer: [rows, K] 6-bit codes -> [rows, K] bytes, each 16
    codes little-endian in 12 bytes followed by 4 padding bytes (`pad`
    [rows, K/16, 4] or zeros)."""
    rows, K = codes.shape
    bits = ((np.asarray(codes, dtype=np.int64)[..., None] >> np.arange(6)) & 1).astype(np.uint8)
    body = np.packbits(bits.reshape(rows, K // 16, 96), axis=2, bitorder="little")
    out = np.zeros((rows, K // 16, 16), dtype=np.uint8)
    out[:, :, :12] = body
    if pad is not None:
        out[:, :, 12:] = pad
    return out.reshape(rows, K)


def unpack_fp6(rows_bytes):
    """Test-side unpacker (np.unpackbits), the inverse of pack_fp6."""
    rows, K = rows_bytes.shape
    bits = np.unpackbits(rows_bytes.reshape(rows, K // 16, 16)[:, :, :12], axis=2,
                         bitorder="little")
    return (bits.reshape(rows, K // 16, 16, 6).astype(np.int64) << np.arange(6)).sum(axis=3) \
        .reshape(rows, K)


def random_case6(rng, M, N, K, fmt_a, fmt_b, scale_lo=122, scale_hi=132):
    """Codes uniform over all 64 values of each FP6 format (an FP8 operand,
    fmt 1 or 2, takes random_case8's codes) with random padding bytes,
    scales near 1 and C with exponents 2^-8 .. 2^8."""
    A8, B8, SA, SB, C = random_case8(rng, M, N, K, 1 if fmt_a >= 3 else fmt_a,
                                     1 if fmt_b >= 3 else fmt_b, scale_lo, scale_hi)
    def operand(fmt, rows, fp8):
        if fmt < 3:
            return fp8, None
        codes = rng.integers(0, 64, size=(rows, K))
        pad = rng.integers(0, 256, size=(rows, K // 16, 4)).astype(np.uint8)
        return pack_fp6(codes, pad), codes
    A, ca = operand(fmt_a, M, A8)
    B, cb = operand(fmt_b, N, B8)
    return A, B, SA, SB, C, ca, cb


def element_fraction(row_bytes, codes, k, fmt):
    if fmt >= 3:
        return fp6_fraction(int(codes[k]), fmt)
    return fp8_fraction(int(row_bytes[k]), fmt)


def check_fp6_golden(o):
    for fmt, code, v in read_golden("fp6_values.txt"):
        got = o.fp6_value(int(code, 2), int(fmt))
        assert got == float(v) and math.copysign(1.0, got) == math.copysign(1.0, float(v)), \
            (fmt, code, got, v)


def check_fp6_all_codes(o):
    """Every code of both formats: the oracle's decode equals the test-side
    field decoder; codes 0..31 increase strictly, bit 5 negates; the largest
    values are 7.5 and 28; and every value is exactly representable in the
    8-bit format with the same mantissa width and a wider exponent range
    (E2M3 in E4M3, E3M2 in E5M2, by torch's float8 types)."""
    import torch
    for fmt, top, dt in ((3, 7.5, torch.float8_e4m3fn), (4, 28.0, torch.float8_e5m2)):
        vals = [o.fp6_value(c, fmt) for c in range(64)]
        for c in range(64):
            assert Fraction(vals[c]) == fp6_fraction(c, fmt), (fmt, c, vals[c])
            assert vals[c ^ 0x20] == -vals[c] and math.copysign(1, vals[c ^ 0x20]) != \
                math.copysign(1, vals[c]), (fmt, c)
        assert all(vals[c] < vals[c + 1] for c in range(31)), fmt
        assert vals[31] == top and vals[63] == -top
        t = torch.tensor(vals, dtype=torch.float64)
        assert torch.equal(t.to(dt).double(), t), fmt


def check_fp6_layout(o):
    """The oracle reads element k of a padded FP6 row where an independent
    unpacker does, ignores the padding bytes, and a lone code at any
    position reads back only there."""
    rng = np.random.default_rng(91)
    codes = rng.integers(0, 64, size=(3, 96))
    pad = rng.integers(0, 256, size=(3, 6, 4)).astype(np.uint8)
    rows = pack_fp6(codes, pad)
    assert np.array_equal(unpack_fp6(rows), codes)
    for r in range(3):
        assert [o.fp6_code(rows[r], k) for k in range(96)] == codes[r].tolist()
    for k in range(32):
        one = np.zeros((1, 32), dtype=np.int64)
        one[0, k] = 0b101101
        row = pack_fp6(one)[0]
        assert [o.fp6_code(row, i) for i in range(32)] == one[0].tolist(), k


def brute_force_gemm6(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha, beta, C, ca, cb):
    two = Fraction(2)
    D = np.zeros((M, N), dtype=np.uint16)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = element_fraction(A[m], None if ca is None else ca[m], k, fmt_a)
                b = element_fraction(B[n], None if cb is None else cb[n], k, fmt_b)
                acc += a * two ** (int(SA[m, k // 32]) - 127) * b * two ** (int(SB[n, k // 32]) - 127)
            y = Fraction(alpha) * acc
            if beta != 0.0:
                y += Fraction(beta) * bf16_bits_to_fraction(int(C[m, n]))
            D[m, n] = bf16_rne_by_search(y)
    return D


def check_fp6_brute_force(o, cases=8):
    rng = np.random.default_rng(92)
    for i in range(cases):
        fmt_a, fmt_b = [(3, 3), (4, 4), (3, 4), (1, 3), (4, 2), (3, 1), (4, 3), (2, 4)][i % 8]
        M, N, K = 3, 4, 64
        A, B, SA, SB, C, ca, cb = random_case6(rng, M, N, K, fmt_a, fmt_b)
        alpha, beta = [(1.0, 0.0), (0.5, 0.25), (-2.0, 1.0), (0.75, -0.5)][i % 4]
        D, _, _, inexact = o.gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha=alpha, beta=beta, C=C)
        assert inexact == 0
        want = brute_force_gemm6(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha, beta, C, ca, cb)
        assert same_value(D, want), (i, fmt_a, fmt_b, D, want)


def check_fp6_numpy_crosscheck(o):
    """The exact double sum equals one float64 matmul of operands decoded by
    the test-side unpacker and field decoder (exact at these sizes)."""
    rng = np.random.default_rng(93)
    for fmt_a, fmt_b in ((3, 4), (4, 3)):
        M, N, K = 24, 40, 256
        A, B, SA, SB, _, ca, cb = random_case6(rng, M, N, K, fmt_a, fmt_b)
        _, acc, _, inexact = o.gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, want_acc=True)
        assert inexact == 0
        table = {f: np.array([float(fp6_fraction(c, f)) for c in range(64)]) for f in (3, 4)}
        sa = np.repeat(np.ldexp(1.0, SA.astype(np.int64) - 127), 32, axis=1)
        sb = np.repeat(np.ldexp(1.0, SB.astype(np.int64) - 127), 32, axis=1)
        ref = (table[fmt_a][unpack_fp6(A)] * sa) @ (table[fmt_b][unpack_fp6(B)] * sb).T
        assert np.array_equal(acc, ref)


# --- E2M1 in the padded form (16 codes per 16 bytes), mixed with FP8 / FP6 ---

def pack_fp4_padded(codes, pad=None):
    """Test-side packer: [rows, K] 4-bit codes -> [rows, K] bytes, each 16
    codes two per byte (even element in the low nibble) in 8 bytes followed
    by 8 padding bytes (`pad` [rows, K/16, 8] or zeros)."""
    rows, K = codes.shape
    c = np.asarray(codes, dtype=np.uint8).reshape(rows, K // 16, 8, 2)
    out = np.zeros((rows, K // 16, 16), dtype=np.uint8)
    out[:, :, :8] = c[..., 0] | (c[..., 1] << 4)
    if pad is not None:
        out[:, :, 8:] = pad
    return out.reshape(rows, K)


def random_case4p(rng, M, N, K, fmt_a, fmt_b):
    """Padded E2M1 operands (fmt 5; random codes and padding) with the other
    side from random_case6; returns the codes of padded operands too."""
    A, B, SA, SB, C, ca, cb = random_case6(rng, M, N, K, 1 if fmt_a == 5 else fmt_a,
                                           1 if fmt_b == 5 else fmt_b)
    def operand(fmt, rows, X, codes):
        if fmt != 5:
            return X, codes
        c = rng.integers(0, 16, size=(rows, K))
        return pack_fp4_padded(c, rng.integers(0, 256, size=(rows, K // 16, 8))), c
    A, ca = operand(fmt_a, M, A, ca)
    B, cb = operand(fmt_b, N, B, cb)
    return A, B, SA, SB, C, ca, cb


def check_fp4_padded_layout(o):
    """The oracle reads element k of a padded E2M1 row where the packer put
    it, ignores the padding bytes, and a lone code reads back only there."""
    rng = np.random.default_rng(95)
    codes = rng.integers(0, 16, size=(3, 64))
    rows = pack_fp4_padded(codes, rng.integers(0, 256, size=(3, 4, 8)))
    for r in range(3):
        assert [o.fp4_padded_code(rows[r], k) for k in range(64)] == codes[r].tolist()
    for k in range(32):
        one = np.zeros((1, 32), dtype=np.int64)
        one[0, k] = 0b1011
        row = pack_fp4_padded(one)[0]
        assert [o.fp4_padded_code(row, i) for i in range(32)] == one[0].tolist(), k


def check_fp4_padded_equals_packed(o):
    """E2M1 x E2M1 through the padded form equals the MXFP4 oracle on the
    same codes in packed rows: D and the exact sum, bit for bit."""
    rng = np.random.default_rng(96)
    M, N, K = 12, 20, 128
    ca = rng.integers(0, 16, size=(M, K))
    cb = rng.integers(0, 16, size=(N, K))
    _, _, SA, SB, C = random_case(rng, M, N, K)
    packed = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    D1, acc1, _, i1 = o.gemm(packed(ca), packed(cb), SA, SB, M, N, K, alpha=0.5, beta=1.0, C=C,
                             want_acc=True)
    D2, acc2, _, i2 = o.gemm8(pack_fp4_padded(ca), pack_fp4_padded(cb), SA, SB, M, N, K, 5, 5,
                              alpha=0.5, beta=1.0, C=C, want_acc=True)
    assert i1 == 0 and i2 == 0
    assert np.array_equal(D1, D2) and np.array_equal(acc1, acc2)


def check_fp4_padded_brute_force(o, cases=6):
    """Padded E2M1 mixed with FP8 and FP6 on either side: exact rational
    brute force with the page's E2M1 values."""
    rng = np.random.default_rng(97)
    e2m1 = page_e2m1_values()
    two = Fraction(2)
    for i in range(cases):
        fmt_a, fmt_b = [(5, 1), (3, 5), (5, 4), (2, 5), (5, 5), (5, 3)][i % 6]
        M, N, K = 3, 4, 64
        A, B, SA, SB, C, ca, cb = random_case4p(rng, M, N, K, fmt_a, fmt_b)
        D, _, _, inexact = o.gemm8(A, B, SA, SB, M, N, K, fmt_a, fmt_b, alpha=0.75, beta=-0.5,
                                   C=C)
        assert inexact == 0
        def val(X, codes, r, k, fmt):
            if fmt == 5:
                return e2m1[int(codes[r, k])]
            return element_fraction(X[r], None if codes is None else codes[r], k, fmt)
        want = np.zeros((M, N), dtype=np.uint16)
        for m in range(M):
            for n in range(N):
                acc = sum(val(A, ca, m, k, fmt_a) * two ** (int(SA[m, k // 32]) - 127) *
                          val(B, cb, n, k, fmt_b) * two ** (int(SB[n, k // 32]) - 127)
                          for k in range(K))
                y = Fraction(0.75) * acc + Fraction(-0.5) * bf16_bits_to_fraction(int(C[m, n]))
                want[m, n] = bf16_rne_by_search(y)
        assert same_value(D, want), (i, fmt_a, fmt_b, D, want)


def check_fp4_padded_exactness_flag(o):
    """E2M1 0.5 x E5M2 2^-16 (granule 2^-17) in one sum with 6 x 57344 x 2^17
    (~2^35.4): sum|ab| / granule ~ 2^52.4, which the oracle must report; a
    granule taken two binades too coarse would miss it."""
    K = 64
    ca = np.zeros((1, K), dtype=np.int64)
    ca[0, 0], ca[0, 32] = 1, 7                      # 0.5 and 6
    A = pack_fp4_padded(ca)
    B = np.zeros((1, K), dtype=np.uint8)
    B[0, 0], B[0, 32] = 0x01, 0x7B                  # 2^-16 and 57344
    SA = np.full((1, 2), 127, dtype=np.uint8)
    SB = np.array([[127, 144]], dtype=np.uint8)     # second block x 2^17
    _, _, _, inexact = o.gemm8(A, B, SA, SB, 1, 1, K, 5, 2)
    assert inexact == 1, inexact
    SB[0, 1] = 140                                  # ~2^48.4 granules: exact
    _, _, _, inexact = o.gemm8(A, B, SA, SB, 1, 1, K, 5, 2)
    assert inexact == 0, inexact


def _sub_codes(Q, fmt):
    """Test-side unpacking of a quantiser's padded output into codes."""
    if fmt == 5:
        rows, K = Q.shape
        g = Q.reshape(rows, K // 16, 16)[:, :, :8].astype(np.int64)
        return np.stack([g & 15, g >> 4], axis=3).reshape(rows, K)
    return unpack_fp6(Q)


def check_quant_sub_nearest_and_scale(o):
    """FP6 and padded E2M1 quantisation: the scale satisfies 2^(s + emax) <=
    amax < 2^(s + emax + 1) (emax 2, 4, 2); every code is the nearest value
    of the format to |x| / 2^s, ties to the even code, saturating, with the
    sign of x; the padding bytes are written as zeros."""
    rng = np.random.default_rng(24)
    rows, K = 4, 96
    x = rng.standard_normal((rows, K)) * 5.0
    x[0, :7] = [0.0, -0.0, 1.0625, -3.0, 1e-3, 250.0, -1e-30]
    bits = _bf16_bits(x)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    e2m1 = page_e2m1_values()
    for fmt, emax, sign in ((3, 2, 0x20), (4, 4, 0x20), (5, 2, 0x8)):
        top = 7 if fmt == 5 else 31
        vals = [e2m1[c] if fmt == 5 else fp6_fraction(c, fmt) for c in range(top + 1)]
        Q, S = o.quantize8(bits, rows, K, fmt, fill=0xA5)
        pad = Q.reshape(rows, K // 16, 16)[:, :, (8 if fmt == 5 else 12):]
        assert not pad.any(), fmt
        codes = _sub_codes(Q, fmt)
        for r in range(rows):
            for b in range(K // 32):
                s = int(S[r, b]) - 127
                amax = max(abs(Fraction(v)) for v in xv[r, 32 * b:32 * b + 32])
                if amax:
                    assert Fraction(2) ** (s + emax) <= amax < Fraction(2) ** (s + emax + 1)
            for k in range(K):
                s = int(S[r, k // 32]) - 127
                y = abs(Fraction(xv[r, k])) / Fraction(2) ** s
                if y >= vals[top]:
                    want = top
                else:
                    d = [abs(y - v) for v in vals]
                    cands = [c for c in range(top + 1) if d[c] == min(d)]
                    want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
                if np.signbit(xv[r, k]):
                    want |= sign
                assert int(codes[r, k]) == want, (fmt, r, k, xv[r, k], s, codes[r, k], want)


def check_quant_sub_matches_generator(o):
    """The input generator's sub-byte rule (numpy: scale, round half to even
    on the significand, field assembly, packing) gives the same bytes."""
    from block_scaled_mxfp4_gb300 import inputs
    rng = np.random.default_rng(25)
    x = rng.standard_normal((16, 512)) * np.ldexp(1.0, rng.integers(-8, 8, size=(16, 1)))
    bits = _bf16_bits(x)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for name, fmt in (("e2m3", 3), ("e3m2", 4), ("e2m1", 5)):
        Qg, Sg = inputs.quantize_rows_fp6(xv, name)
        Qo, So = o.quantize8(bits, 16, 512, fmt)
        assert np.array_equal(So, Sg), name
        assert np.array_equal(Qo, Qg), name


# --- NVFP4: packed E2M1 with one unsigned-E4M3 scale per 16 K -----------

def ue4m3_fraction(code):
    """Exact value of a UE4M3 scale byte from its fields (test side): the
    E4M3 field decoder above with the sign bit 0.  None for 0x7F (NaN) and
    for bytes with bit 7 set (not UE4M3 codes)."""
    if code & 0x80:
        return None
    return fp8_fraction(code, 1)


def random_case_nv(rng, M, N, K):
    """All 16 E2M1 codes; scales from 2^-3 to 2^3 with some zeros and
    subnormals (codes 0x01-0x07); C with exponents 2^-8 .. 2^8."""
    A = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)

    def scales(rows):
        c = rng.integers(0x20, 0x51, size=(rows, K // 16))
        kind = rng.random((rows, K // 16))
        c = np.where(kind < 0.05, 0, c)
        c = np.where((kind >= 0.05) & (kind < 0.12), rng.integers(1, 8, size=c.shape), c)
        return c.astype(np.uint8)
    e = rng.integers(119, 136, size=(M, N)).astype(np.uint16)
    f = rng.integers(0, 128, size=(M, N)).astype(np.uint16)
    sgn = rng.integers(0, 2, size=(M, N)).astype(np.uint16)
    C = (sgn << 15) | (e << 7) | f
    return A, B, scales(M), scales(N), C


def brute_force_gemm_nv(A, B, SA, SB, M, N, K, alpha, beta, C):
    vals = page_e2m1_values()
    ra = [page_decode_row(A[m], K) for m in range(M)]
    rb = [page_decode_row(B[n], K) for n in range(N)]
    D = np.zeros((M, N), dtype=np.uint16)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = vals[ra[m][k]] * ue4m3_fraction(int(SA[m, k // 16]))
                b = vals[rb[n][k]] * ue4m3_fraction(int(SB[n, k // 16]))
                acc += a * b
            y = Fraction(alpha) * acc
            if beta != 0.0:
                y += Fraction(beta) * bf16_bits_to_fraction(int(C[m, n]))
            D[m, n] = bf16_rne_by_search(y)
    return D


def check_ue4m3_values(o):
    """Every byte: the oracle's UE4M3 decode equals the E4M3 golden values
    (positive codes), the test-side field decoder and the numpy table; 0x7F
    and bytes with bit 7 set are NaN."""
    golden = {int(code, 16): v for fmt, code, v in read_golden("fp8_values.txt") if int(fmt) == 1}
    table = o.ue4m3_table()
    for c in range(256):
        got = o.ue4m3_value(c)
        want = ue4m3_fraction(c)
        if want is None:
            assert got != got and table[c] != table[c], c
        else:
            assert math.isfinite(got) and Fraction(got) == want and table[c] == got, (c, got, want)
            if c in golden:
                assert golden[c] != "nan" and got == float(golden[c]), (c, got, golden[c])


def check_nv_block_16(o):
    """Closed forms with all elements 1.0: each 16-element block contributes
    16 * sa_b * sb_b, so scales 1, 2, 4, 8 on A's four blocks give 240, and
    1, 1/2, 1/4, 1/8 on B's give 30."""
    K = 64
    ones = np.full((1, K // 2), 0x22, dtype=np.uint8)          # code 2 = 1.0
    unit = np.full((1, K // 16), 0x38, dtype=np.uint8)         # UE4M3 1.0
    up = np.array([[0x38, 0x40, 0x48, 0x50]], dtype=np.uint8)  # 1, 2, 4, 8
    down = np.array([[0x38, 0x30, 0x28, 0x20]], dtype=np.uint8)
    D, acc, _, inexact = o.gemm_nv(ones, ones, up, unit, 1, 1, K, want_acc=True)
    assert inexact == 0 and acc[0, 0] == 240.0 and bf16_to_f64(D)[0, 0] == 240.0
    D, acc, _, _ = o.gemm_nv(ones, ones, unit, down, 1, 1, K, want_acc=True)
    assert acc[0, 0] == 30.0 and bf16_to_f64(D)[0, 0] == 30.0


def check_nv_brute_force(o, cases=6):
    rng = np.random.default_rng(91)
    for i in range(cases):
        M, N, K = 3, 4, 64
        A, B, SA, SB, C = random_case_nv(rng, M, N, K)
        alpha, beta = [(1.0, 0.0), (0.5, 0.25), (-2.0, 1.0)][i % 3]
        D, _, _, inexact = o.gemm_nv(A, B, SA, SB, M, N, K, alpha=alpha, beta=beta, C=C)
        assert inexact == 0
        want = brute_force_gemm_nv(A, B, SA, SB, M, N, K, alpha, beta, C)
        assert same_value(D, want), (i, D, want)


def check_nv_numpy_crosscheck(o):
    """The exact double sum equals one float64 matmul of the numpy-dequantised
    operands, and the sampled form equals the full one."""
    rng = np.random.default_rng(92)
    M, N, K = 24, 40, 256
    A, B, SA, SB, C = random_case_nv(rng, M, N, K)
    D, acc, _, inexact = o.gemm_nv(A, B, SA, SB, M, N, K, alpha=0.5, beta=0.75, C=C, want_acc=True)
    assert inexact == 0
    assert np.array_equal(acc, o.acc_numpy_nv(A, B, SA, SB, K))
    pairs = np.array([(0, 0), (23, 39), (5, 17), (11, 2)])
    Ds, accs, _, _ = o.gemm_nv_sampled(A, B, SA, SB, M, N, K, pairs, alpha=0.5, beta=0.75, C=C)
    assert np.array_equal(Ds, D[pairs[:, 0], pairs[:, 1]])
    assert np.array_equal(accs, acc[pairs[:, 0], pairs[:, 1]])


def check_nv_exactness_flag(o):
    """One block with both scales at the smallest subnormal 2^-9 next to 1008
    products of (6 * 448)^2: sum|ab| spans more than 2^52 granules of the
    tiny block's products (2^-20), which the oracle must report -- the
    scales' ulp exponents enter the granule.  With that block at 448 too
    the sum is exact."""
    K = 1024
    A = np.full((1, K // 2), 0x77, dtype=np.uint8)             # 6.0
    A[0, :8] = 0x11                                            # block 0: 0.5
    B = np.full((1, K // 2), 0x77, dtype=np.uint8)
    SA = np.full((1, K // 16), 0x7E, dtype=np.uint8)           # 448
    SB = np.full((1, K // 16), 0x7E, dtype=np.uint8)
    SA[0, 0] = SB[0, 0] = 0x01                                 # 2^-9
    _, _, _, inexact = o.gemm_nv(A, B, SA, SB, 1, 1, K)
    assert inexact == 1
    SA[0, 0] = SB[0, 0] = 0x7E
    _, _, _, inexact = o.gemm_nv(A, B, SA, SB, 1, 1, K)
    assert inexact == 0


def check_nv_rejects_non_ue4m3(o):
    A = np.zeros((2, 16), dtype=np.uint8)
    S = np.full((2, 2), 0x38, dtype=np.uint8)
    o.gemm_nv(A, A, S, S, 2, 2, 32)
    bad = S.copy()
    bad[1, 1] = 0xB8                                           # sign bit set
    for args in ((bad, S), (S, bad)):
        try:
            o.gemm_nv(A, A, args[0], args[1], 2, 2, 32)
        except ValueError:
            continue
        raise AssertionError("a scale byte with bit 7 set was accepted")


ALL_CHECKS = [check_gemm_single_rounding, check_e2m1_golden, check_e2m1_bitfields, check_e8m0,
              check_nibble_order,
              check_bf16_golden, check_bf16_roundtrip, check_bf16_midpoints,
              check_identity, check_identity_scaled, check_alpha_beta,
              check_brute_force, check_all_code_pairs, check_numpy_crosscheck,
              check_rounding_is_only_error, check_sampled_matches_full,
              check_quant_golden, check_quant_scale_rule, check_quant_nearest_brute_force,
              check_quant_matches_generator,
              check_fp8_golden, check_fp8_all_codes, check_fp8_brute_force,
              check_fp8_torch_crosscheck, check_fp8_identity, check_fp8_sampled_matches_full,
              check_fp8_exactness_flag, check_quant8_golden, check_quant8_scale_rule,
              check_quant8_nearest_brute_force, check_quant8_matches_generator,
              check_fp6_golden, check_fp6_all_codes, check_fp6_layout, check_fp6_brute_force,
              check_fp6_numpy_crosscheck, check_fp4_padded_layout, check_fp4_padded_equals_packed,
              check_fp4_padded_brute_force, check_fp4_padded_exactness_flag,
              check_quant_sub_nearest_and_scale, check_quant_sub_matches_generator,
              check_ue4m3_values, check_nv_block_16, check_nv_brute_force,
              check_nv_numpy_crosscheck, check_nv_exactness_flag, check_nv_rejects_non_ue4m3]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod)


def test_exactness_violation_is_reported(oracle_mod):
    # Scales 2^-126 and 2^127 in one row make sum|ab| / granule exceed 2^52:
    # the double sum may round, and the oracle must say so.
    K = 64
    A = np.full((1, K // 2), 0x77, dtype=np.uint8)       # all 6.0
    B = np.full((1, K // 2), 0x11, dtype=np.uint8)       # all 0.5
    SA = np.array([[1, 254]], dtype=np.uint8)
    SB = np.array([[127, 127]], dtype=np.uint8)
    _, _, _, inexact = oracle_mod.gemm(A, B, SA, SB, 1, 1, K)
    assert inexact == 1
    # A non-dyadic alpha makes alpha * acc round in double: reported too.
    SA2 = np.array([[127, 127]], dtype=np.uint8)
    _, _, _, inexact = oracle_mod.gemm(A, B, SA2, SB, 1, 1, K, alpha=0.1)
    assert inexact == 1
    _, _, _, inexact = oracle_mod.gemm(A, B, SA2, SB, 1, 1, K, alpha=0.5)
    assert inexact == 0


def test_inexact_outputs_are_flagged_and_within_one_ulp(oracle_mod):
    # beta * C many binades below alpha * acc: y = p1 + p2 rounds in double,
    # the oracle must flag it, and it is still within 1 bf16 ulp of exact.
    rng = np.random.default_rng(77)
    M, N, K = 4, 4, 32
    A, B, SA, SB, _ = random_case(rng, M, N, K)
    C = np.full((M, N), 0x0301, dtype=np.uint16)         # ~2^-120
    D, _, _, inexact = oracle_mod.gemm(A, B, SA, SB, M, N, K, alpha=0.75, beta=-0.25, C=C)
    assert inexact > 0
    want = brute_force_gemm(A, B, SA, SB, M, N, K, 0.75, -0.25, C)
    assert np.all(np.abs(D.astype(np.int64) - want.astype(np.int64)) <= 1)


def test_rejects_bad_arguments(oracle_mod):
    A = np.zeros((2, 16), dtype=np.uint8)
    S = np.full((2, 1), 127, dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle_mod.gemm(A, A, S, S, 2, 2, 33)                 # K % 32 != 0
    with pytest.raises(ValueError):
        oracle_mod.gemm_sampled(A, A, S, S, 2, 2, 32, [(2, 0)])  # m out of range


def test_workload_generator_rules():
    """The generator follows the stated recipe (scale rule, saturation, RNE)."""
    from block_scaled_mxfp4_gb300 import inputs
    vals = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    # Ties go to the even mantissa, large values saturate.
    y = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, 0.2, 0.3])
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, 0.0, 0.5]
    got = [vals[c] for c in inputs._e2m1_codes_rne_sat(y)]
    assert got == want
    # Scale exponent floor(log2(amax/6)); the block max saturates to 6.
    x = np.zeros((1, 32))
    x[0, 3] = -13.0                      # 13/6 in [2, 4): s = 1, 13/2 = 6.5 -> 6
    x[0, 4] = 1.0                        # 1/2 = 0.5 -> code 1
    packed, sc = inputs.quantize_rows(x)
    assert sc[0, 0] == 128
    codes = inputs.unpack_fp4(packed)[0]
    assert codes[3] == 8 | 7 and codes[4] == 1 and codes[0] == 0
    # Same seed -> same bytes.
    p1, p2 = inputs.workload("tiny"), inputs.workload("tiny")
    assert np.array_equal(p1.A, p2.A) and np.array_equal(p1.SB, p2.SB)
    assert p1.SA.min() >= 123 and p1.SA.max() <= 131
