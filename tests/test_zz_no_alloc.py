"""mxfp4_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Called through the C ABI on consecutive calls that reuse the shared scratch
array, it must agree with the CPU oracle element by element (the parity bound
every GPU test uses) and give exactly the bits of mxfp4_gemm, which runs the
same plan on a workspace the caller allocated.  It must refuse shapes whose
scratch need is larger than the array, and streams of another device.  This
file is collected last on purpose and must pass both alone in a fresh
process and after the other tests.
"""
import numpy as np
import pytest

import block_scaled_mxfp4_gb300 as mx
from block_scaled_mxfp4_gb300 import inputs
from parity_util import Dev, assert_within_bound, d_to_bits, run_gemm

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCRATCH_BYTES = 32 << 20        # MXFP4_NOALLOC_SCRATCH_BYTES in include/mxfp4_gemm.h


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_mxfp4_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_noalloc(dev, split_k):
    p = dev.p
    D = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = dev.C if p.beta != 0.0 else None
    mx.mxfp4_gemm_noalloc(D, D.stride(0), C, 0 if C is None else C.stride(0), dev.A,
                          dev.A.stride(0) * 2, dev.B, dev.B.stride(0) * 2, dev.SA,
                          dev.SA.stride(0), dev.SB, dev.SB.stride(0), p.alpha, p.beta,
                          p.M, p.N, p.K, split_k)
    torch.cuda.synchronize()
    return d_to_bits(D)


def test_header_declares_the_scratch_limit():
    text = open(mx.HEADER).read()
    assert "#define MXFP4_NOALLOC_SCRATCH_BYTES (32u << 20)" in text
    assert "mxfp4_gemm_noalloc" in mx.header_functions()


def test_noalloc_matches_mxfp4_gemm_on_consecutive_calls(oracle_mod):
    # Different problems back to back (each reuses scratch the one before
    # left behind), then the first again: sixteen splits keep fp32 partials
    # and tile counters in the scratch, the large one relays its scales into
    # it, the mid one needs none.
    cases = [
        (inputs.make_problem("na-skinny", 48, 3072, 4096, 21, "normal", 1.0, 1.0, 0.5), 16),
        (inputs.make_problem("na-mid", 256, 512, 1024, 22, "codes", 0.5, 0.5, 1.0), 0),
        (inputs.make_problem("na-big", 2304, 2304, 1024, 24, "codes", 1.0, 0.0, None), 0),
    ]
    cases.append(cases[0])
    for p, split in cases:
        dev = Dev(p)
        want = run_gemm(dev, split_k=split)           # existing entry point, torch workspace
        got = run_noalloc(dev, split)
        assert mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, split) <= SCRATCH_BYTES
        pairs = np.array([(m, n) for m in range(0, p.M, 7) for n in range(0, p.N, 13)])
        ref, _, sabs, inexact = oracle_mod.gemm_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K,
                                                        pairs, alpha=p.alpha, beta=p.beta, C=p.C)
        assert inexact == 0
        sel = (pairs[:, 0], pairs[:, 1])
        assert_within_bound(got[sel], ref, sabs, what=f"noalloc {p.name} against the oracle")
        assert np.array_equal(got, want), f"noalloc {p.name}: not the bits of mxfp4_gemm"
        assert not np.isnan((got.astype(np.uint32) << 16).view(np.float32)).any()


def test_noalloc_rejects_shapes_beyond_the_scratch():
    M = N = 2048
    K = 4096
    # Sixteen splits keep fp32 partials (up to eight reduce inside their cluster).
    assert mx.mxfp4_gemm_workspace_size(M, N, K, 16) > SCRATCH_BYTES
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((M, K // 2), dtype=torch.uint8, device="cuda")
    S = torch.full((M, K // 32), 127, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_gemm_noalloc(D, N, None, 0, A, K, A, K, S, K // 32, S, K // 32, 1.0, 0.0,
                              M, N, K, 16)
    assert e.value.status == -4                      # MXFP4_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(D).item() == 0        # nothing was enqueued


def test_noalloc_back_to_back_without_sync(oracle_mod):
    """Split-K calls enqueued with no synchronisation between them share the
    scratch; each waits for the one before it, so all give the same bits."""
    p = inputs.make_problem("na-chain", 16, 4096, 8192, 23, "normal", 1.0, 0.0, None)
    dev = Dev(p)
    assert mx.mxfp4_plan_gemm(p.M, p.N, p.K, 16, 0).split_k == 16
    assert mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, 16) > 0
    first = run_noalloc(dev, 16)
    outs = [torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(4)]
    for D in outs:
        mx.mxfp4_gemm_noalloc(D, p.N, None, 0, dev.A, p.K, dev.B, p.K, dev.SA, p.K // 32,
                              dev.SB, p.K // 32, p.alpha, p.beta, p.M, p.N, p.K, 16)
    torch.cuda.synchronize()
    for D in outs:
        assert np.array_equal(d_to_bits(D), first)
