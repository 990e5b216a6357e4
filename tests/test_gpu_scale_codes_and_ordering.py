"""GPU parity on the E8M0 edge codes, and ordering of back-to-back calls.

E8M0 (page "asm_f4gemm -- driving aiter's gfx950 MXFP4 GEMM code objects",
section "Data layouts", subsection "A_scale / B_scale"): value 2^(e-127),
0xFF = NaN.  The page also says code 0 stands for 2^-126, against its own
formula; the oracle takes the formula (2^-127), and these tests show the
tensor cores do the same.  Scale pairs are chosen so that every product
stays in the normal fp32 range (each K block pairs a tiny scale with a huge
one, or two ordinary ones).

Ordering: every GEMM launch is a programmatic dependent of the work before
it on the stream and waits in-kernel before touching memory that work may
write.  A chain of calls enqueued with no synchronisation between them (each
reading the previous one's output as C, or A produced by the quantiser just
before) must give the same bits as the same calls with a synchronise after
each.
"""
import numpy as np
import pytest

import block_scaled_mxfp4_gb300 as mx
from block_scaled_mxfp4_gb300 import inputs
from parity_util import Dev, assert_within_bound, bf16_bits_to_f64, d_to_bits, run_gemm

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


# ------------------------------------------------------ E8M0 edge codes --

def edge_code_problem(M, N, K, seed):
    """Random E2M1 codes (all 16); the scale of K block kb is drawn by class
    kb % 4: A in {0, 1} with B in {253, 254}; A in {253, 254} with B in
    {0, 1}; A = 1 with B = 254; both ordinary (120..134).  So codes 0, 1, 253
    and 254 appear in both operands, and every product a_k * b_k is a normal
    fp32 number (2^(ea + eb - 254) in [2^-14, 2^14] times at most 36)."""
    rng = np.random.default_rng(seed)
    kb = K // 32
    A = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    SA = np.empty((M, kb), dtype=np.uint8)
    SB = np.empty((N, kb), dtype=np.uint8)
    for b in range(kb):
        c = b % 4
        if c == 0:
            SA[:, b] = rng.integers(0, 2, M)
            SB[:, b] = rng.integers(253, 255, N)
        elif c == 1:
            SA[:, b] = rng.integers(253, 255, M)
            SB[:, b] = rng.integers(0, 2, N)
        elif c == 2:
            SA[:, b] = 1
            SB[:, b] = 254
        else:
            SA[:, b] = rng.integers(120, 135, M)
            SB[:, b] = rng.integers(120, 135, N)
    C = inputs.f32_to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    return inputs.Problem("e8m0-edges", M, N, K, A, B, SA, SB, C, 0.75, 0.5, seed)


@pytest.mark.parametrize("M,N,K,split", [(128, 256, 256, 0), (16, 256, 512, 0),
                                         (1, 4096, 2048, 4), (96, 160, 1024, 2),
                                         (2304, 2304, 256, 0)],
                         ids=["one-tile", "swap", "decode-split", "split", "pair"])
def test_e8m0_edge_codes_match_oracle(oracle_mod, M, N, K, split):
    p = edge_code_problem(M, N, K, seed=M + N + K)
    for code in (0, 1, 253, 254):
        assert (p.SA == code).any() and (p.SB == code).any()
    if M >= 2304:
        assert mx.mxfp4_plan_gemm(M, N, K, 0, 0).pair == 1
    Dref, _, sabs, inexact = oracle_mod.gemm(p.A, p.B, p.SA, p.SB, M, N, K, alpha=p.alpha,
                                             beta=p.beta, C=p.C)
    assert inexact == 0
    got = run_gemm(Dev(p), split_k=split)
    assert_within_bound(got, Dref, sabs, what=f"E8M0 edge codes {M}x{N}x{K} split {split}")


@pytest.mark.parametrize("M,N,K,split", [(128, 256, 512, 0), (16, 512, 1024, 0),
                                         (1, 2048, 4096, 4), (2304, 2304, 512, 0)],
                         ids=["one-tile", "swap", "decode-split", "pair"])
def test_e8m0_nan_scale_poisons_its_row_and_column(oracle_mod, M, N, K, split):
    """Scale code 0xFF is NaN: a NaN scale of A's row r makes row r of D
    NaN, one of B's row c makes column c NaN, and nothing else changes."""
    p = inputs.make_problem("nan-scale", M, N, K, seed=M * 3 + N + K, values="codes",
                            alpha=1.0, beta=1.0, c_sigma=1.0)
    r, c = M // 2, N // 3 + 1
    p.SA[r, (K // 32) // 2] = 0xFF
    p.SB[c, K // 32 - 1] = 0xFF
    Dref, _, sabs, _ = oracle_mod.gemm(p.A, p.B, p.SA, p.SB, M, N, K, alpha=p.alpha,
                                       beta=p.beta, C=p.C)
    got = run_gemm(Dev(p), split_k=split)
    g, ref = bf16_bits_to_f64(got), bf16_bits_to_f64(Dref)
    want_nan = np.zeros((M, N), dtype=bool)
    want_nan[r, :] = True
    want_nan[:, c] = True
    assert np.array_equal(np.isnan(ref), want_nan)           # the oracle's reading
    assert np.array_equal(np.isnan(g), want_nan)
    ok = ~want_nan
    assert_within_bound(got[ok], Dref[ok], sabs[ok], what="outside the NaN row / column")


# --------------------------------------------- back-to-back call ordering --

CHAIN_SHAPES = {
    "decode-split": (1, 8192, 8192),
    "skinny-split": (48, 3072, 4096),
    "mid": (512, 1024, 2048),
    "relayout": (128, 40960, 512),
    "pair": (2304, 2304, 1024),
}


def _gemm(dev, D, C, beta, alpha, ws, wsb, flags, stream):
    p = dev.p
    mx.mxfp4_gemm_ex(D, D.stride(0), C, 0 if C is None else C.stride(0), dev.A, p.K, dev.B, p.K,
                     dev.SA, p.K // 32, dev.SB, p.K // 32, alpha, beta, p.M, p.N, p.K, 0, flags,
                     ws, wsb, stream)


@pytest.mark.parametrize("flags", [0, 1], ids=["plain", "b_static"])
@pytest.mark.parametrize("case", sorted(CHAIN_SHAPES))
def test_back_to_back_calls_see_the_previous_output(case, flags):
    """Three calls with no synchronisation between them: D1 = A.B^T;
    D2 = 0.5 A.B^T + 0.75 D1 (C = D1); then D1 <- A.B^T - D2 (C = D2, the
    output written over the first call's output).  The same workspace serves
    all three.  Bit-identical to the same calls synchronised one by one."""
    M, N, K = CHAIN_SHAPES[case]
    p = inputs.make_problem("chain", M, N, K, seed=M + 2 * N + K, values="normal", alpha=1.0,
                            beta=0.0, c_sigma=None)
    dev = Dev(p)
    s = torch.cuda.current_stream()
    wsb = mx.mxfp4_gemm_workspace_size(M, N, K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    plan = mx.mxfp4_plan_gemm(M, N, K, 0, 0)
    if case.endswith("split"):
        assert plan.split_k > 1
    if case == "relayout":
        assert plan.relayout_pass == 1 and plan.pair == 0
    if case == "pair":
        assert plan.pair == 1

    def chain(sync):
        D1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        D2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        steps = [lambda: _gemm(dev, D1, None, 0.0, 1.0, ws, wsb, flags, s),
                 lambda: _gemm(dev, D2, D1, 0.75, 0.5, ws, wsb, flags, s),
                 lambda: _gemm(dev, D1, D2, -1.0, 1.0, ws, wsb, flags, s)]
        for f in steps:
            f()
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return d_to_bits(D1), d_to_bits(D2)

    ref1, ref2 = chain(sync=True)
    for _ in range(3):
        got1, got2 = chain(sync=False)
        assert np.array_equal(got2, ref2)
        assert np.array_equal(got1, ref1)
    assert not np.isnan(bf16_bits_to_f64(ref1)).any()


def test_quantiser_then_gemm_without_sync():
    """A produced by mxfp4_quantize right before the GEMM on the same stream
    (no synchronisation): the GEMM reads the new A, not the old bytes."""
    M, N, K = 64, 4096, 4096
    rng = np.random.default_rng(71)
    X = torch.from_numpy(inputs.f32_to_bf16_bits(
        rng.standard_normal((M, K)).astype(np.float32)).view(np.int16)).cuda()
    p = inputs.make_problem("qchain", M, N, K, seed=72, values="normal", alpha=1.0, beta=0.0,
                            c_sigma=None)
    dev = Dev(p)
    Q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    S = torch.empty((M, K // 32), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    wsb = mx.mxfp4_gemm_workspace_size(M, N, K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")

    def run(sync):
        Q.fill_(0)
        S.fill_(0)
        torch.cuda.synchronize()
        mx.mxfp4_quantize(Q, K, S, K // 32, X, K, M, K)
        if sync:
            torch.cuda.synchronize()
        mx.mxfp4_gemm_ex(D, N, None, 0, Q, K, dev.B, K, S, K // 32, dev.SB, K // 32, 1.0, 0.0,
                         M, N, K, 0, mx.MXFP4_FLAG_B_STATIC, ws, wsb)
        torch.cuda.synchronize()
        return d_to_bits(D)

    ref = run(sync=True)
    assert not np.all(ref == 0)
    for _ in range(3):
        assert np.array_equal(run(sync=False), ref)


@pytest.mark.parametrize("name", ["decode", "skinny", "mid", "tiny"])
def test_b_static_flag_gives_the_same_bits(name):
    """MXFP4_FLAG_B_STATIC changes when B is read, not what is computed."""
    p = inputs.workload(name)
    dev = Dev(p)
    want = run_gemm(dev)
    D = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    C = dev.C if p.beta != 0.0 else None
    _gemm(dev, D, C, p.beta, p.alpha, ws, wsb, mx.MXFP4_FLAG_B_STATIC, None)
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D), want)
