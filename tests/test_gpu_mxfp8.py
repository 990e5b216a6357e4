"""MXFP8 / MXFP6 GEMM (E4M3 / E5M2 / E2M3 / E3M2 elements, one E8M0 scale per
32) on the GPU through the C ABI, element by element against the oracle.

Bound, as for MXFP4: |D_gpu - D_ref| <= ulp_bf16(D_ref) + 2^-20 * sum|a_k b_k|.
"""
import numpy as np
import pytest

import block_scaled_mxfp4_gb300 as mx
from block_scaled_mxfp4_gb300 import inputs
from parity_util import assert_within_bound, bf16_bits_to_f64, d_to_bits, sample_pairs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ABI_FMT = {"e4m3": mx.MXFP8_E4M3, "e5m2": mx.MXFP8_E5M2, "e2m3": mx.MXFP6_E2M3,
           "e3m2": mx.MXFP6_E3M2, "e2m1": mx.MXFP4_E2M1_PADDED}
ORACLE_FMT = inputs.BYTE_FORMATS


@pytest.fixture(scope="session", autouse=True)
def _built():
    from block_scaled_mxfp4_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class Dev8:
    """A problem's operands on the GPU."""

    def __init__(self, p):
        self.p = p
        d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
        self.A, self.B, self.SA, self.SB = d(p.A), d(p.B), d(p.SA), d(p.SB)
        self.C = None
        if p.C is not None:
            self.C = d(np.ascontiguousarray(p.C).view(np.int16)).view(torch.bfloat16)


def run8(dev, split_k=0):
    p = dev.p
    D = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_bytes = mx.mxfp8_gemm_workspace_size(p.M, p.N, p.K, split_k)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    C = dev.C if p.beta != 0.0 else None
    mx.mxfp8_gemm(D, D.stride(0), C, 0 if C is None else C.stride(0), dev.A, dev.A.stride(0),
                  dev.B, dev.B.stride(0), dev.SA, dev.SA.stride(0), dev.SB, dev.SB.stride(0),
                  ABI_FMT[p.fmt_a], ABI_FMT[p.fmt_b], float(p.alpha), float(p.beta),
                  p.M, p.N, p.K, split_k, ws if ws_bytes else None, ws_bytes)
    torch.cuda.synchronize()
    return d_to_bits(D)


def oracle_full(oracle_mod, p):
    D, _, sabs, inexact = oracle_mod.gemm8(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K,
                                           ORACLE_FMT[p.fmt_a], ORACLE_FMT[p.fmt_b],
                                           alpha=p.alpha, beta=p.beta, C=p.C)
    assert inexact == 0
    return D, sabs


# (M, N, K, fmt A, fmt B, alpha, beta, C sigma): one-tile configurations
# 128x256, 128x128 and 128x64 tiles, swap-AB for M <= 64, K with a half-full
# last stage (K % 128 != 0), ragged M and N, mixed formats, alpha / beta with C,
# and a grid of more tiles than SMs (scales relaid in a separate pass).
CASES = [
    (128, 256, 512, "e4m3", "e4m3", 1.0, 0.0, None),
    (300, 520, 1024, "e4m3", "e5m2", 0.5, 1.0, 1.0),
    (1000, 700, 288, "e5m2", "e4m3", 1.0, 0.0, None),
    (257, 300, 160, "e5m2", "e5m2", 2.0, 0.0, None),
    (1, 4096, 2048, "e4m3", "e4m3", 1.0, 0.0, None),
    (2, 1000, 1024, "e4m3", "e5m2", 1.0, 0.5, 0.1),
    (33, 100, 384, "e4m3", "e4m3", 1.0, 0.0, None),
    (64, 2048, 4096, "e5m2", "e4m3", 1.0, 1.0, 0.1),
    (2000, 2600, 256, "e4m3", "e4m3", 1.0, 0.0, None),
]


@pytest.mark.parametrize("M,N,K,fa,fb,alpha,beta,cs", CASES,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}-{c[3]}x{c[4]}" for c in CASES])
def test_mxfp8_parity(oracle_mod, M, N, K, fa, fb, alpha, beta, cs):
    p = inputs.make_problem8("p8", M, N, K, M + N + K, fa, fb, "normal", alpha, beta, cs)
    Dref, sabs = oracle_full(oracle_mod, p)
    assert_within_bound(run8(Dev8(p)), Dref, sabs, p.alpha, f"mxfp8 {M}x{N}x{K} {fa}x{fb}")


# FP6 (16 codes packed in 12 of every 16 bytes): both formats, mixed with
# each other and with FP8, on the same kernel paths as CASES.
CASES6 = [
    (128, 256, 512, "e2m3", "e2m3", 1.0, 0.0, None),
    (300, 520, 1024, "e3m2", "e4m3", 0.5, 1.0, 1.0),
    (1000, 700, 288, "e2m3", "e3m2", 1.0, 0.0, None),
    (1, 4096, 2048, "e2m3", "e2m3", 1.0, 0.0, None),
    (33, 100, 384, "e5m2", "e2m3", 1.0, 0.0, None),
    (64, 2048, 4096, "e3m2", "e3m2", 1.0, 1.0, 0.1),
    (2000, 2600, 256, "e2m3", "e4m3", 1.0, 0.0, None),
]


@pytest.mark.parametrize("M,N,K,fa,fb,alpha,beta,cs", CASES6,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}-{c[3]}x{c[4]}" for c in CASES6])
def test_mxfp6_parity(oracle_mod, M, N, K, fa, fb, alpha, beta, cs):
    p = inputs.make_problem8("p6", M, N, K, M + N + K + 6, fa, fb, "normal", alpha, beta, cs)
    Dref, sabs = oracle_full(oracle_mod, p)
    assert_within_bound(run8(Dev8(p)), Dref, sabs, p.alpha, f"mxfp6 {M}x{N}x{K} {fa}x{fb}")


def test_mxfp6_padding_bytes_are_not_read():
    """Random bytes in the 4 padding bytes of every 16: D is unchanged."""
    p = inputs.make_problem8("pad6", 256, 384, 512, 17, "e2m3", "e3m2", "normal", 1.0, 0.0, None)
    want = run8(Dev8(p))
    rng = np.random.default_rng(17)
    for X in (p.A, p.B):
        v = X.reshape(X.shape[0], -1, 16)
        v[:, :, 12:] = rng.integers(0, 256, size=v[:, :, 12:].shape, dtype=np.uint8)
    assert np.array_equal(run8(Dev8(p)), want)


# E2M1 in the padded form (16 codes in 8 of every 16 bytes), mixed with the
# 8- and 6-bit formats on either side.
CASES4P = [
    (128, 256, 512, "e2m1", "e4m3", 1.0, 0.0, None),
    (300, 520, 1024, "e5m2", "e2m1", 0.5, 1.0, 1.0),
    (1, 4096, 2048, "e2m1", "e2m3", 1.0, 0.0, None),
    (64, 2048, 4096, "e3m2", "e2m1", 1.0, 1.0, 0.1),
    (1000, 700, 288, "e2m1", "e2m1", 1.0, 0.0, None),
]


@pytest.mark.parametrize("M,N,K,fa,fb,alpha,beta,cs", CASES4P,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}-{c[3]}x{c[4]}" for c in CASES4P])
def test_padded_e2m1_mixed_parity(oracle_mod, M, N, K, fa, fb, alpha, beta, cs):
    p = inputs.make_problem8("p4p", M, N, K, M + N + K + 4, fa, fb, "normal", alpha, beta, cs)
    Dref, sabs = oracle_full(oracle_mod, p)
    assert_within_bound(run8(Dev8(p)), Dref, sabs, p.alpha, f"padded e2m1 {M}x{N}x{K} {fa}x{fb}")


def test_padded_e2m1_padding_bytes_are_not_read():
    p = inputs.make_problem8("pad4", 256, 384, 512, 19, "e2m1", "e4m3", "normal", 1.0, 0.0, None)
    want = run8(Dev8(p))
    v = p.A.reshape(p.A.shape[0], -1, 16)
    v[:, :, 8:] = np.random.default_rng(19).integers(0, 256, size=v[:, :, 8:].shape,
                                                     dtype=np.uint8)
    assert np.array_equal(run8(Dev8(p)), want)


def test_mxfp6_large_sampled(oracle_mod):
    """The 8192^3 E2M3 workload, as the benchmark runs it, on sampled outputs."""
    p = inputs.workload8("large6")
    pairs = sample_pairs(p.M, p.N, 3000, 10)
    Dr, _, sabs, inexact = oracle_mod.gemm8_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K,
                                                    ORACLE_FMT[p.fmt_a], ORACLE_FMT[p.fmt_b],
                                                    pairs, alpha=p.alpha, beta=p.beta, C=p.C)
    assert inexact == 0
    D = run8(Dev8(p))
    assert_within_bound(D[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, "large6")


@pytest.mark.parametrize("split", [1, 2, 4, 8])
def test_mxfp8_split_k(oracle_mod, split):
    p = inputs.make_problem8("p8s", 48, 1536, 4096, 11, "e4m3", "e4m3", "normal", 1.0, 0.5, 1.0)
    Dref, sabs = oracle_full(oracle_mod, p)
    assert_within_bound(run8(Dev8(p), split_k=split), Dref, sabs, p.alpha, f"mxfp8 split {split}")


def test_mxfp8_plan_uses_one_tile_kernel():
    for M, N, K in [(8192, 8192, 8192), (1, 8192, 8192), (512, 1024, 2048)]:
        p = mx.mxfp8_plan_gemm(M, N, K, 0, 0)
        assert p.pair == 0 and p.tile_k == 128


@pytest.mark.parametrize("name", ["decode8", "mixed8", "mixed6"])
def test_mxfp8_workloads_full(oracle_mod, name):
    p = inputs.workload8(name)
    Dref, sabs = oracle_full(oracle_mod, p)
    assert_within_bound(run8(Dev8(p)), Dref, sabs, p.alpha, name)


def test_mxfp8_large_sampled(oracle_mod):
    """The 8192^3 E4M3 workload, as the benchmark runs it, on sampled outputs."""
    p = inputs.workload8("large8")
    pairs = sample_pairs(p.M, p.N, 3000, 9)
    Dr, _, sabs, inexact = oracle_mod.gemm8_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K,
                                                    ORACLE_FMT[p.fmt_a], ORACLE_FMT[p.fmt_b],
                                                    pairs, alpha=p.alpha, beta=p.beta, C=p.C)
    assert inexact == 0
    D = run8(Dev8(p))
    assert_within_bound(D[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, "large8")
    assert not np.isnan(bf16_bits_to_f64(D)).any()


def test_mxfp8_nan_scale_propagates(oracle_mod):
    """Scale code 0xFF (NaN) in one block of A row 3: that row is NaN, others not."""
    p = inputs.make_problem8("nan8", 128, 256, 256, 5, "e4m3", "e4m3", "normal", 1.0, 0.0, None)
    p.SA[3, 2] = 0xFF
    D = bf16_bits_to_f64(run8(Dev8(p)))
    assert np.isnan(D[3]).all()
    assert not np.isnan(np.delete(D, 3, axis=0)).any()


@pytest.mark.parametrize("fa,fb", [("e4m3", "e5m2"), ("e2m3", "e2m1")])
@pytest.mark.parametrize("M,N,K,split", [(300, 520, 1024, 0), (1, 4096, 2048, 0), (2000, 2600, 256, 0),
                                         (48, 1536, 4096, 4)])
def test_mxfp8_prepacked_matches(M, N, K, split, fa, fb):
    """Scales relaid once with mxfp4_scale_relayout (K in elements):
    mxfp8_gemm_prepacked equals mxfp8_gemm bit for bit, for 8-bit operands
    and for the padded 6- and 4-bit forms."""
    p = inputs.make_problem8("pp8", M, N, K, 3, fa, fb, "normal", 1.0, 0.5, 1.0)
    dev = Dev8(p)
    ref = run8(dev, split_k=split)
    sfa = torch.empty(mx.mxfp4_scale_relayout_size(M, K), dtype=torch.uint8, device="cuda")
    sfb = torch.empty(mx.mxfp4_scale_relayout_size(N, K), dtype=torch.uint8, device="cuda")
    mx.mxfp4_scale_relayout(sfa, dev.SA, M, K, K // 32)
    mx.mxfp4_scale_relayout(sfb, dev.SB, N, K, K // 32)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = mx.mxfp8_gemm_prepacked_workspace_size(M, N, K, split)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    mx.mxfp8_gemm_prepacked(D, N, dev.C, N, dev.A, K, dev.B, K, sfa, sfb, ABI_FMT[p.fmt_a],
                            ABI_FMT[p.fmt_b], p.alpha, p.beta, M, N, K, split, ws if wsb else None,
                            wsb)
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D), ref)


# ------------------------------------------------------------ quantiser --

def _special_rows(K):
    """Rows that exercise the quantiser's edges: an all-zero block, signed
    zeros, ties at both formats' block maxima, saturation, bf16 extremes and
    subnormal-range blocks."""
    rows = np.zeros((8, K))
    rows[1, ::2] = -0.0
    rows[1, 1::4] = 1.0
    rows[2, :32] = 256.0
    rows[2, 1:8] = [1.0625, 1.1875, 460.0, 480.0, 0.0029296875, 0.0009765625, -1.5]
    rows[3, :32] = 32768.0
    rows[3, 1:8] = [1.125, 1.375, 61440.0, 57344.0, 2.288818359375e-05, 7.62939453125e-06, -1.25]
    rows[4, :] = 3.3895313892515355e38          # bf16 max
    rows[4, 1::3] = -1e38
    rows[5, :] = np.ldexp(1.0, -133)             # bf16 subnormal: the scale clamps at -127
    rows[6, :] = np.ldexp(1.0, -126) * 3.0
    rows[7, :] = 511.0                           # just below 512: E4M3 saturates at 448
    return rows


def _bf16(x):
    return inputs.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _run_q8(bits, fmt, ldq_pad=0, ldx_pad=0, lds_pad=0):
    rows, K = bits.shape
    Xh = np.zeros((rows, K + ldx_pad), dtype=np.uint16)
    Xh[:, :K] = bits
    X = torch.from_numpy(Xh.view(np.int16)).cuda()
    Q = torch.full((rows, K + ldq_pad), 0xAB, dtype=torch.uint8, device="cuda")
    S = torch.full((rows, K // 32 + lds_pad), 0xCD, dtype=torch.uint8, device="cuda")
    mx.mxfp8_quantize(Q, Q.stride(0), S, S.stride(0), X, X.stride(0), rows, K, ABI_FMT[fmt])
    torch.cuda.synchronize()
    return Q.cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m3", "e3m2", "e2m1"])
def test_mxfp8_quantize_bit_exact(oracle_mod, fmt):
    rng = np.random.default_rng(31 + list(ABI_FMT).index(fmt))
    K = 1024
    x = rng.standard_normal((120, K)) * np.ldexp(1.0, rng.integers(-40, 40, size=(120, 1)))
    bits = _bf16(np.concatenate([x, _special_rows(K)]))
    Q, S = _run_q8(bits, fmt)
    Qr, Sr = oracle_mod.quantize8(bits, bits.shape[0], K, ORACLE_FMT[fmt])
    assert np.array_equal(S, Sr)
    bad = np.argwhere(Q != Qr)
    assert bad.size == 0, [(tuple(i), hex(Q[tuple(i)]), hex(Qr[tuple(i)])) for i in bad[:8]]


def test_mxfp8_quantize_strided(oracle_mod):
    rng = np.random.default_rng(33)
    K = 512
    bits = _bf16(rng.standard_normal((40, K)) * 7.0)
    Q, S = _run_q8(bits, "e5m2", ldq_pad=48, ldx_pad=64, lds_pad=5)
    Qr, Sr = oracle_mod.quantize8(bits, 40, K, 2)
    assert np.array_equal(Q[:, :K], Qr) and np.array_equal(S[:, :K // 32], Sr)
    assert (Q[:, K:] == 0xAB).all() and (S[:, K // 32:] == 0xCD).all()   # padding untouched


def test_mxfp8_quantize_then_gemm(oracle_mod):
    """Activations quantised on the GPU (E4M3) times E5M2 weights: the GEMM
    on the GPU's codes matches the oracle GEMM on the oracle's codes."""
    rng = np.random.default_rng(34)
    M, N, K = 200, 384, 1024
    xa = _bf16(rng.standard_normal((M, K)))
    QA, SA = _run_q8(xa, "e4m3")
    QAr, SAr = oracle_mod.quantize8(xa, M, K, 1)
    assert np.array_equal(QA, QAr) and np.array_equal(SA, SAr)
    w = inputs.make_problem8("qw", N, 32, K, 35, "e5m2", "e5m2", "normal", 1.0, 0.0, None)
    p = inputs.Problem8("q8gemm", M, N, K, "e4m3", "e5m2", QA, w.A, SA, w.SA, None, 1.0, 0.0, 0)
    Dref, sabs = oracle_full(oracle_mod, p)
    assert_within_bound(run8(Dev8(p)), Dref, sabs, 1.0, "quantise -> mxfp8 gemm")


@pytest.mark.parametrize("fa,fb", [("e2m3", "e3m2"), ("e2m1", "e2m3")])
def test_subbyte_quantize_strided_then_gemm(oracle_mod, fa, fb):
    """Both operands quantised on the GPU into padded forms, with row strides
    and a pre-filled output: bit-exact codes (padding written as zeros, the
    bytes past K untouched), then the GEMM on them within the bound."""
    rng = np.random.default_rng(36)
    M, N, K = 96, 320, 512
    xa = _bf16(rng.standard_normal((M, K)) * 3.0)
    xb = _bf16(rng.standard_normal((N, K)) * 0.25)
    QA, SA = _run_q8(xa, fa, ldq_pad=32, ldx_pad=8, lds_pad=3)
    QB, SB = _run_q8(xb, fb)
    for Q, S, x, f, rows in ((QA, SA, xa, fa, M), (QB, SB, xb, fb, N)):
        Qr, Sr = oracle_mod.quantize8(x, rows, K, ORACLE_FMT[f])
        assert np.array_equal(Q[:, :K], Qr) and np.array_equal(S[:, :K // 32], Sr), f
    assert (QA[:, K:] == 0xAB).all() and (SA[:, K // 32:] == 0xCD).all()
    p = inputs.Problem8("qsub", M, N, K, fa, fb, np.ascontiguousarray(QA[:, :K]), QB,
                        np.ascontiguousarray(SA[:, :K // 32]), SB, None, 1.0, 0.0, 0)
    Dref, sabs = oracle_full(oracle_mod, p)
    assert_within_bound(run8(Dev8(p)), Dref, sabs, 1.0, f"quantise -> {fa} x {fb} gemm")


@pytest.mark.parametrize("M,N,K,fa,fb", [(2304, 2600, 1024, "e4m3", "e2m3"),
                                         (300, 520, 512, "e2m1", "e5m2")])
def test_mxfp8_host_entry_matches_device_call(M, N, K, fa, fb):
    """Host buffers in and out through mxfp8_gemm_host (row panels x column
    halves at M, N >= 2048; one block below): with split_k = 1 every block
    runs the whole K in order, so D matches the device call bit for bit."""
    p = inputs.make_problem8("h8", M, N, K, M + N, fa, fb, "normal", 0.5, 0.5, 1.0)
    ref = run8(Dev8(p), split_k=1)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hA, hB, hSA, hSB = pin(p.A), pin(p.B), pin(p.SA), pin(p.SB)
    hC = pin(p.C.view(np.int16))
    hD = torch.zeros((M, N), dtype=torch.int16).pin_memory()
    arena_b = mx.mxfp8_gemm_host_arena_size(M, N, K, 1, True)
    arena = torch.empty(arena_b, dtype=torch.uint8, device="cuda")
    mx.mxfp8_gemm_host(hD, hC, hA, hB, hSA, hSB, ABI_FMT[fa], ABI_FMT[fb], p.alpha, p.beta,
                       M, N, K, 1, arena, arena_b)
    torch.cuda.synchronize()
    assert np.array_equal(hD.numpy().view(np.uint16), ref)
