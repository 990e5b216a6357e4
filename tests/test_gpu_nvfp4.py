"""NVFP4 GEMM (packed E2M1, one UE4M3 scale per 16 K) on the GPU through the
C ABI, element by element against the oracle (oracle.gemm_nv).

Bound, as for MXFP4: |D_gpu - D_ref| <= ulp_bf16(D_ref) + 2^-20 * sum|a_k b_k|.
The kernel is the CTA-pair kernel with kind::mxf4nvf4 MMAs, run for every
shape, after the scales are relaid into the caller's workspace.
"""
import numpy as np
import pytest

import block_scaled_mxfp4_gb300 as mx
from block_scaled_mxfp4_gb300 import inputs
from parity_util import assert_within_bound, bf16_bits_to_f64, d_to_bits, sample_pairs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_mxfp4_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mx.mxfp4_device_status(reset=True)
    yield
    assert mx.mxfp4_device_status() == 0, "a bounded wait timed out during the tests"


class DevNV:
    """An NVFP4 problem's operands on the GPU."""

    def __init__(self, p):
        self.p = p
        d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
        self.A, self.B, self.SA, self.SB = d(p.A), d(p.B), d(p.SA), d(p.SB)
        self.C = None
        if p.C is not None:
            self.C = d(np.ascontiguousarray(p.C).view(np.int16)).view(torch.bfloat16)


def run_nv(dev, alpha=None, beta=None, out=None, stream=None):
    p = dev.p
    alpha = p.alpha if alpha is None else alpha
    beta = p.beta if beta is None else beta
    D = out if out is not None else torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16,
                                               device="cuda")
    wsb = mx.nvfp4_gemm_workspace_size(p.M, p.N, p.K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    C = dev.C if beta != 0.0 else None
    mx.nvfp4_gemm(D, D.stride(0), C, 0 if C is None else C.stride(0), dev.A, dev.A.stride(0) * 2,
                  dev.B, dev.B.stride(0) * 2, dev.SA, dev.SA.stride(0), dev.SB, dev.SB.stride(0),
                  float(alpha), float(beta), p.M, p.N, p.K, ws, wsb, stream)
    torch.cuda.synchronize()
    return d_to_bits(D)


SHAPES = {
    # (M, N, K, alpha, beta, C sigma)
    "one-tile": (256, 256, 256, 1.0, 0.0, None),
    "alpha-beta": (512, 768, 512, 0.5, 0.75, 1.0),
    "ragged": (300, 520, 288, 1.0, 0.0, None),
    "ragged-k-tail": (260, 300, 160, -2.0, 1.0, 1.0),
    "many-tiles": (2304, 2304, 1024, 1.0, 0.0, None),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_nvfp4_matches_oracle(oracle_mod, name):
    M, N, K, alpha, beta, c_sigma = SHAPES[name]
    p = inputs.make_problem_nv(name, M, N, K, seed=M + N + K, alpha=alpha, beta=beta,
                               c_sigma=c_sigma)
    Dref, _, sabs, inexact = oracle_mod.gemm_nv(p.A, p.B, p.SA, p.SB, M, N, K, alpha=alpha,
                                                beta=beta, C=p.C)
    assert inexact == 0
    got = run_nv(DevNV(p))
    assert_within_bound(got, Dref, sabs, what=f"NVFP4 {name} {M}x{N}x{K}")


def test_nvfp4_large_sampled(oracle_mod):
    """8192^3 in the configuration the benchmark times, checked at tile edges
    and random positions."""
    M = N = K = 8192
    p = inputs.make_problem_nv("large-nv", M, N, K, seed=11, alpha=1.0, beta=0.0, c_sigma=None)
    got = run_nv(DevNV(p))
    pairs = sample_pairs(M, N, 1500, seed=12, tile_m=256, tile_n=256)
    Dref, _, sabs, inexact = oracle_mod.gemm_nv_sampled(p.A, p.B, p.SA, p.SB, M, N, K, pairs)
    assert inexact == 0
    assert_within_bound(got[pairs[:, 0], pairs[:, 1]], Dref, sabs, what="NVFP4 8192^3 sampled")


def test_nvfp4_scale_edge_codes(oracle_mod):
    """Scale bytes 0x00 (zero), 0x01 and 0x07 (subnormals), 0x08 (smallest
    normal) and 0x7E (448, the largest) in both operands."""
    M, N, K = 256, 512, 512
    p = inputs.make_problem_nv("edges", M, N, K, seed=5, alpha=1.0, beta=0.0, c_sigma=None)
    rng = np.random.default_rng(6)
    codes = np.array([0x00, 0x01, 0x07, 0x08, 0x7E, 0x38], dtype=np.uint8)
    p.SA[:] = codes[rng.integers(0, len(codes), p.SA.shape)]
    p.SB[:] = codes[rng.integers(0, len(codes), p.SB.shape)]
    Dref, _, sabs, inexact = oracle_mod.gemm_nv(p.A, p.B, p.SA, p.SB, M, N, K)
    assert inexact == 0
    got = run_nv(DevNV(p))
    assert_within_bound(got, Dref, sabs, what="NVFP4 scale edge codes")


def test_nvfp4_nan_scale_poisons_its_row_and_column(oracle_mod):
    """Scale byte 0x7F is NaN in UE4M3: A's row r and B's column c of D turn
    NaN, nothing else changes."""
    M, N, K = 512, 512, 512
    p = inputs.make_problem_nv("nan", M, N, K, seed=7, alpha=1.0, beta=1.0, c_sigma=1.0)
    r, c = 100, 301
    p.SA[r, 9] = 0x7F
    p.SB[c, K // 16 - 1] = 0x7F
    Dref, _, sabs, _ = oracle_mod.gemm_nv(p.A, p.B, p.SA, p.SB, M, N, K, alpha=1.0, beta=1.0,
                                          C=p.C)
    got = run_nv(DevNV(p))
    want_nan = np.zeros((M, N), dtype=bool)
    want_nan[r, :] = True
    want_nan[:, c] = True
    assert np.array_equal(np.isnan(bf16_bits_to_f64(Dref)), want_nan)
    assert np.array_equal(np.isnan(bf16_bits_to_f64(got)), want_nan)
    ok = ~want_nan
    assert_within_bound(got[ok], Dref[ok], sabs[ok], what="NVFP4 outside the NaN row / column")


def test_nvfp4_deterministic_and_ordered():
    """Bit-identical across calls, and a dependent chain (D2 reads D1 as C)
    enqueued without synchronisation gives the same bits as synchronised."""
    M, N, K = 1024, 1536, 1024
    p = inputs.make_problem_nv("chain", M, N, K, seed=9, alpha=1.0, beta=0.0, c_sigma=None)
    dev = DevNV(p)
    first = run_nv(dev)
    assert np.array_equal(run_nv(dev), first)
    wsb = mx.nvfp4_gemm_workspace_size(M, N, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def chain(sync):
        D1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        D2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        for D, C, beta in ((D1, None, 0.0), (D2, D1, 0.5)):
            mx.nvfp4_gemm(D, N, C, N if C is not None else 0, dev.A, K, dev.B, K, dev.SA, K // 16,
                          dev.SB, K // 16, 1.0, beta, M, N, K, ws, wsb)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return d_to_bits(D1), d_to_bits(D2)

    ref = chain(True)
    assert np.array_equal(ref[0], first)
    for _ in range(3):
        got = chain(False)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_nvfp4_strided_buffers(oracle_mod):
    """Row strides larger than the rows: A and B with 64 spare fp4 elements
    per row, scale rows with 8 spare bytes, C and D with 24 spare columns."""
    M, N, K = 384, 320, 512
    p = inputs.make_problem_nv("strided", M, N, K, seed=21, alpha=0.5, beta=1.0, c_sigma=1.0)
    Dref, _, sabs, inexact = oracle_mod.gemm_nv(p.A, p.B, p.SA, p.SB, M, N, K, alpha=0.5,
                                                beta=1.0, C=p.C)
    assert inexact == 0
    pad = lambda x, extra: np.concatenate([x, np.full((x.shape[0], extra), 0x5A, np.uint8)], 1)
    A = torch.from_numpy(pad(p.A, 32)).cuda()
    B = torch.from_numpy(pad(p.B, 32)).cuda()
    SA = torch.from_numpy(pad(p.SA, 8)).cuda()
    SB = torch.from_numpy(pad(p.SB, 8)).cuda()
    Cw = np.zeros((M, N + 24), dtype=np.uint16)
    Cw[:, :N] = p.C
    C = torch.from_numpy(Cw.view(np.int16)).cuda().view(torch.bfloat16)
    D = torch.full((M, N + 24), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = mx.nvfp4_gemm_workspace_size(M, N, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    mx.nvfp4_gemm(D, N + 24, C, N + 24, A, A.shape[1] * 2, B, B.shape[1] * 2, SA, SA.shape[1],
                  SB, SB.shape[1], 0.5, 1.0, M, N, K, ws, wsb)
    torch.cuda.synchronize()
    got = d_to_bits(D)
    assert_within_bound(got[:, :N], Dref, sabs, what="NVFP4 strided")
    assert np.isnan(bf16_bits_to_f64(got[:, N:])).all()          # padding columns untouched


def test_nvfp4_cuda_graph_replay():
    """nvfp4_gemm (relayout + dependent pair launch) captured in a CUDA graph
    replays to the eager bits and reads its inputs at replay time."""
    M, N, K = 1024, 768, 512
    p = inputs.make_problem_nv("graph", M, N, K, seed=31, alpha=1.0, beta=0.0, c_sigma=None)
    dev = DevNV(p)
    ref = run_nv(dev)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    wsb = mx.nvfp4_gemm_workspace_size(M, N, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.nvfp4_gemm(D, N, None, 0, dev.A, K, dev.B, K, dev.SA, K // 16, dev.SB, K // 16, 1.0,
                      0.0, M, N, K, ws, wsb, s)
    for _ in range(2):
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(d_to_bits(D), ref)
    dev.B.copy_(torch.roll(dev.B, 1, 0))
    dev.SB.copy_(torch.roll(dev.SB, 1, 0))
    ref2 = run_nv(dev)
    assert not np.array_equal(ref2, ref)
    D.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D), ref2)


# Skinny shapes (M <= 64) run the one-tile kernel (swap-AB, kind::mxf4nvf4,
# row-major scales by TMA, split-K summed in the tile's cluster).
SKINNY = {
    # (M, N, K, alpha, beta, C sigma)
    "decode": (1, 8192, 8192, 1.0, 0.0, None),
    "m8-ragged-n": (8, 3000, 2048, 0.5, 1.0, 0.1),
    "m33-ragged-k": (33, 1024, 4160, 1.0, 0.0, None),
    "m64": (64, 2048, 4096, 1.0, 1.0, 0.1),
}


@pytest.mark.parametrize("name", sorted(SKINNY))
def test_nvfp4_skinny_matches_oracle(oracle_mod, name):
    M, N, K, alpha, beta, c_sigma = SKINNY[name]
    p = inputs.make_problem_nv(name, M, N, K, seed=M + 3 * N + K, alpha=alpha, beta=beta,
                               c_sigma=c_sigma)
    plan = mx.mxfp4_plan_gemm(M, N, K, 0, 0)
    assert plan.swap_ab == 1
    Dref, _, sabs, inexact = oracle_mod.gemm_nv(p.A, p.B, p.SA, p.SB, M, N, K, alpha=alpha,
                                                beta=beta, C=p.C)
    assert inexact == 0
    dev = DevNV(p)
    # Scale rows padded to a multiple of 16 bytes (a K with a partial last
    # 256-K stage has K/16 % 16 != 0), as the one-tile path's TMA needs.
    width = (K // 16 + 15) // 16 * 16
    pad = lambda x: np.concatenate([x, np.full((x.shape[0], width - K // 16), 0x38, np.uint8)], 1)
    dev.SA = torch.from_numpy(pad(p.SA)).cuda()
    dev.SB = torch.from_numpy(pad(p.SB)).cuda()
    got = run_nv(dev)
    assert_within_bound(got, Dref, sabs, what=f"NVFP4 skinny {name} {M}x{N}x{K} "
                                              f"(split {plan.split_k})")
    assert np.array_equal(run_nv(dev), got)                     # deterministic


def test_nvfp4_skinny_scale_codes_and_nan(oracle_mod):
    """The one-tile path on the scale edge codes, and 0x7F poisoning exactly
    its row and column."""
    M, N, K = 16, 1536, 2048
    p = inputs.make_problem_nv("skinny-edges", M, N, K, seed=41, alpha=1.0, beta=0.0,
                               c_sigma=None)
    rng = np.random.default_rng(42)
    codes = np.array([0x00, 0x01, 0x07, 0x08, 0x7E, 0x38], dtype=np.uint8)
    p.SA[:] = codes[rng.integers(0, len(codes), p.SA.shape)]
    p.SB[:] = codes[rng.integers(0, len(codes), p.SB.shape)]
    r, c = 5, 777
    p.SA[r, 3] = 0x7F
    p.SB[c, 100] = 0x7F
    Dref, _, sabs, _ = oracle_mod.gemm_nv(p.A, p.B, p.SA, p.SB, M, N, K)
    got = run_nv(DevNV(p))
    want_nan = np.zeros((M, N), dtype=bool)
    want_nan[r, :] = True
    want_nan[:, c] = True
    assert np.array_equal(np.isnan(bf16_bits_to_f64(Dref)), want_nan)
    assert np.array_equal(np.isnan(bf16_bits_to_f64(got)), want_nan)
    ok = ~want_nan
    assert_within_bound(got[ok], Dref[ok], sabs[ok], what="NVFP4 skinny edge codes")


def test_nvfp4_skinny_misaligned_scales_take_the_pair_path(oracle_mod):
    """Scale rows that are not 16-byte aligned (ld_sa = K/16 + 4) cannot come
    by TMA: the call falls back to the pair kernel, same results."""
    M, N, K = 4, 1024, 1024
    p = inputs.make_problem_nv("skinny-odd", M, N, K, seed=43, alpha=1.0, beta=0.0, c_sigma=None)
    Dref, _, sabs, inexact = oracle_mod.gemm_nv(p.A, p.B, p.SA, p.SB, M, N, K)
    assert inexact == 0
    pad = lambda x: np.concatenate([x, np.full((x.shape[0], 4), 0x38, np.uint8)], 1)
    SA = torch.from_numpy(pad(p.SA)).cuda()
    SB = torch.from_numpy(pad(p.SB)).cuda()
    dev = DevNV(p)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = mx.nvfp4_gemm_workspace_size(M, N, K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    mx.nvfp4_gemm(D, N, None, 0, dev.A, K, dev.B, K, SA, SA.shape[1], SB, SB.shape[1], 1.0, 0.0,
                  M, N, K, ws, wsb)
    torch.cuda.synchronize()
    assert_within_bound(d_to_bits(D), Dref, sabs, what="NVFP4 skinny, unaligned scale rows")
