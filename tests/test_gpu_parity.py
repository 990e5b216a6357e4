"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every comparison is element by element within the stated bound (see
parity_util).  Full comparisons at the sizes the oracle finishes in seconds;
at the full large / skinny sizes, sampled outputs (tile edges + random).
"""
import numpy as np
import pytest

import block_scaled_mxfp4_gb300 as mx
from block_scaled_mxfp4_gb300 import inputs
from parity_util import (Dev, assert_within_bound, bf16_bits_to_f64, d_to_bits, run_gemm,
                         sample_pairs)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="session", autouse=True)
def _built():
    from block_scaled_mxfp4_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mx.mxfp4_device_status(reset=True)
    yield
    assert mx.mxfp4_device_status() == 0, "a bounded wait timed out during the tests"


_PROBLEMS = {}


def problem(name):
    if name not in _PROBLEMS:
        _PROBLEMS[name] = inputs.identity_problem() if name == "identity" else inputs.workload(name)
    return _PROBLEMS[name]


def full_oracle(oracle_mod, p, alpha=None, beta=None):
    alpha = p.alpha if alpha is None else alpha
    beta = p.beta if beta is None else beta
    D, _, sabs, inexact = oracle_mod.gemm(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K, alpha=alpha,
                                          beta=beta, C=p.C)
    assert inexact == 0
    return D, sabs


# --------------------------------------------------------------- relayout --

def relayout_reference(S, rows, K):
    """tcgen05 scale layout written from its description: 512-byte atoms of
    128 rows x 4 blocks; row 32j + i, block b at byte 16i + 4j + b; atoms
    row-block major; rows padded to a multiple of 256, blocks to 8 per 256 K,
    with 0x7F."""
    kb = K // 32
    groups = 2 * (-(-K // 256))
    rblocks = 2 * (-(-rows // 256))
    out = np.full(rblocks * groups * 512, 0x7F, dtype=np.uint8)
    for rb in range(rblocks):
        for g in range(groups):
            base = (rb * groups + g) * 512
            for i in range(32):
                for j in range(4):
                    r = rb * 128 + 32 * j + i
                    for b in range(4):
                        k = g * 4 + b
                        if r < rows and k < kb:
                            out[base + 16 * i + 4 * j + b] = S[r, k]
    return out


@pytest.mark.parametrize("rows,K", [(1, 32), (128, 512), (300, 288), (64, 16384 // 8), (257, 1024)])
def test_scale_relayout_bytes(rows, K):
    rng = np.random.default_rng(rows * 7 + K)
    ld = K // 32 + 3
    S = rng.integers(0, 256, size=(rows, ld), dtype=np.uint8)
    src = torch.from_numpy(S).cuda()
    size = mx.mxfp4_scale_relayout_size(rows, K)
    dst = torch.zeros(size, dtype=torch.uint8, device="cuda")
    mx.mxfp4_scale_relayout(dst, src, rows, K, ld)
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    want = relayout_reference(S, rows, K)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("rows_a,rows_b,K", [(1, 8192, 1024), (300, 257, 288), (129, 64, 64)])
def test_scale_relayout2_bytes(rows_a, rows_b, K):
    """Both operands in one launch: each destination holds exactly what the
    single-operand relayout writes (different row strides, ragged rows)."""
    rng = np.random.default_rng(rows_a + 3 * rows_b + K)
    ld_a, ld_b = K // 32 + 1, K // 32 + 5
    Sa = rng.integers(0, 256, size=(rows_a, ld_a), dtype=np.uint8)
    Sb = rng.integers(0, 256, size=(rows_b, ld_b), dtype=np.uint8)
    da = torch.zeros(mx.mxfp4_scale_relayout_size(rows_a, K), dtype=torch.uint8, device="cuda")
    db = torch.zeros(mx.mxfp4_scale_relayout_size(rows_b, K), dtype=torch.uint8, device="cuda")
    mx.mxfp4_scale_relayout2(da, torch.from_numpy(Sa).cuda(), rows_a, ld_a,
                             db, torch.from_numpy(Sb).cuda(), rows_b, ld_b, K)
    torch.cuda.synchronize()
    assert np.array_equal(da.cpu().numpy(), relayout_reference(Sa, rows_a, K))
    assert np.array_equal(db.cpu().numpy(), relayout_reference(Sb, rows_b, K))


# ------------------------------------------------- scale placement probes --

def _ones_problem(M, N, K):
    A = np.full((M, K // 2), 0x22, dtype=np.uint8)        # every element 1.0
    B = np.full((N, K // 2), 0x22, dtype=np.uint8)
    SA = np.full((M, K // 32), 127, dtype=np.uint8)
    SB = np.full((N, K // 32), 127, dtype=np.uint8)
    return inputs.Problem("probe", M, N, K, A, B, SA, SB, None, 1.0, 0.0, 0)


@pytest.mark.parametrize("M,N", [(128, 256), (256, 128), (16, 256), (1, 200)])
def test_single_scale_probes(M, N):
    """One doubled scale at (row r, block kb) adds exactly 32 to the outputs
    of row r (A) or column r (B): pins which TMEM scale word feeds which row
    and K block, for the plain and the swapped mapping."""
    K = 512
    rows_a = sorted(r for r in {0, 1, 31, 32, 97, M - 1} if r < M)
    rows_b = sorted(r for r in {0, 5, 33, 64, 127, 128, 200, N - 1} if r < N)
    bad = []
    for which, rows in (("A", rows_a), ("B", rows_b)):
        for r in rows:
            for kb in (0, 1, 2, 3, 5, 8, 13, 15):
                p = _ones_problem(M, N, K)
                (p.SA if which == "A" else p.SB)[r, kb] = 128
                D = bf16_bits_to_f64(run_gemm(Dev(p)))
                want = np.full((M, N), float(K))
                if which == "A":
                    want[r, :] += 32
                else:
                    want[:, r] += 32
                if not np.array_equal(D, want):
                    wrong = np.argwhere(D != want)
                    bad.append((which, r, kb, len(wrong), wrong[:4].tolist(),
                                D[tuple(wrong[0])]))
    assert not bad, bad


# ------------------------------------------------------------ workloads --

def test_tiny_full(oracle_mod):
    p = problem("tiny")
    Dref, sabs = full_oracle(oracle_mod, p)
    assert_within_bound(run_gemm(Dev(p)), Dref, sabs, p.alpha, "tiny")


def test_identity_exact():
    p = problem("identity")
    D = bf16_bits_to_f64(run_gemm(Dev(p)))
    codes = inputs.unpack_fp4(p.A)
    vals = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    want = np.where(codes & 8, -vals[codes & 7], vals[codes & 7])[:, : p.N]
    assert np.array_equal(D, want)


def test_mid_full(oracle_mod):
    p = problem("mid")
    Dref, sabs = full_oracle(oracle_mod, p)
    dev = Dev(p)
    for split in (0, 1, 2, 4):
        assert_within_bound(run_gemm(dev, split_k=split), Dref, sabs, p.alpha, f"mid s={split}")


@pytest.mark.parametrize("split", [0, 1, 2, 4, 8, 16])
def test_decode_split_sweep(oracle_mod, split):
    p = problem("decode")
    if "decode_ref" not in _PROBLEMS:
        _PROBLEMS["decode_ref"] = full_oracle(oracle_mod, p)
    Dref, sabs = _PROBLEMS["decode_ref"]
    if "decode_dev" not in _PROBLEMS:
        _PROBLEMS["decode_dev"] = Dev(p)
    D = run_gemm(_PROBLEMS["decode_dev"], split_k=split)
    assert_within_bound(D, Dref, sabs, p.alpha, f"decode s={split}")


@pytest.mark.parametrize("split", [0, 1, 2, 4, 8])
def test_skinny_split_sweep(oracle_mod, split):
    p = problem("skinny")
    if "skinny_ref" not in _PROBLEMS:
        rows = [0, 1, 31, 32, 63]
        pairs = np.array([(m, n) for m in rows for n in range(p.N)], dtype=np.int64)
        pairs = np.unique(np.concatenate([pairs, sample_pairs(p.M, p.N, 3000, 4)]), axis=0)
        Dr, _, sabs, inexact = oracle_mod.gemm_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K, pairs,
                                                       alpha=p.alpha, beta=p.beta, C=p.C)
        assert inexact == 0
        _PROBLEMS["skinny_ref"] = (pairs, Dr, sabs)
        _PROBLEMS["skinny_dev"] = Dev(p)
    pairs, Dr, sabs = _PROBLEMS["skinny_ref"]
    D = run_gemm(_PROBLEMS["skinny_dev"], split_k=split)
    assert_within_bound(D[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, f"skinny s={split}")


def test_large_sampled(oracle_mod):
    p = problem("large")
    pairs = sample_pairs(p.M, p.N, 4000, 3)
    Dr, _, sabs, inexact = oracle_mod.gemm_sampled(p.A, p.B, p.SA, p.SB, p.M, p.N, p.K, pairs,
                                                   alpha=p.alpha, beta=p.beta, C=p.C)
    assert inexact == 0
    D = run_gemm(Dev(p))
    assert_within_bound(D[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, "large")
    assert not np.isnan(bf16_bits_to_f64(D)).any()


# ----------------------------------------------------------- edge cases --

EDGE_SHAPES = [
    (1, 16, 32), (7, 40, 96), (63, 200, 288), (65, 300, 256), (129, 520, 1024),
    (300, 2048, 1024), (1, 4096, 2048), (2, 129, 64), (200, 37, 160), (130, 130, 544),
    (5, 64, 128), (33, 100, 384), (257, 300, 384), (2000, 2600, 288),
]


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_edge_shapes(oracle_mod, M, N, K):
    p = inputs.make_problem("edge", M, N, K, seed=M * 131 + N * 7 + K, values="codes",
                            alpha=1.0, beta=1.0, c_sigma=1.0)
    Dref, sabs = full_oracle(oracle_mod, p)
    dev = Dev(p)
    for split in (0, 1, 3):
        assert_within_bound(run_gemm(dev, split_k=split), Dref, sabs, p.alpha,
                            f"{M}x{N}x{K} s={split}")


def test_alpha_beta_forms(oracle_mod):
    p = inputs.make_problem("ab", 96, 160, 256, seed=8, values="normal", alpha=1.0, beta=0.0,
                            c_sigma=1.0)
    dev = Dev(p)
    for alpha, beta in ((1.0, 0.0), (0.5, 0.5), (-2.0, 1.0), (0.0, 1.0), (1.0, -1.0)):
        Dref, sabs = full_oracle(oracle_mod, p, alpha=alpha, beta=beta)
        assert_within_bound(run_gemm(dev, alpha=alpha, beta=beta), Dref, sabs, alpha,
                            f"alpha={alpha} beta={beta}")
    # alpha = 0, beta = 1 returns C exactly.
    D = run_gemm(dev, alpha=0.0, beta=1.0)
    assert np.array_equal(bf16_bits_to_f64(D), bf16_bits_to_f64(p.C))


def test_beta_zero_ignores_nan_c():
    p = problem("tiny")
    dev = Dev(p)
    ref = run_gemm(dev)
    dev.C = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D = torch.empty((p.M, p.N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, 0), dtype=torch.uint8,
                     device="cuda")
    mx.mxfp4_gemm(D, p.N, dev.C, p.N, dev.A, p.K, dev.B, p.K, dev.SA, p.K // 32, dev.SB,
                  p.K // 32, 1.0, 0.0, p.M, p.N, p.K, 0, ws, ws.numel())
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D), ref)


def test_strides_and_in_place(oracle_mod):
    M, N, K = 130, 200, 512
    p = inputs.make_problem("strided", M, N, K, seed=12, values="normal", alpha=0.5, beta=1.0,
                            c_sigma=1.0)
    Dref, sabs = full_oracle(oracle_mod, p)
    pad_k, pad_s, pad_n = 64, 5, 24
    A = torch.zeros((M, (K + pad_k) // 2), dtype=torch.uint8, device="cuda")
    B = torch.zeros((N, (K + pad_k) // 2), dtype=torch.uint8, device="cuda")
    A[:, : K // 2] = torch.from_numpy(p.A).cuda()
    B[:, : K // 2] = torch.from_numpy(p.B).cuda()
    SA = torch.zeros((M, K // 32 + pad_s), dtype=torch.uint8, device="cuda")
    SB = torch.zeros((N, K // 32 + pad_s), dtype=torch.uint8, device="cuda")
    SA[:, : K // 32] = torch.from_numpy(p.SA).cuda()
    SB[:, : K // 32] = torch.from_numpy(p.SB).cuda()
    # D aliases C (in-place beta), both with a padded row stride.
    DC = torch.zeros((M, N + pad_n), dtype=torch.bfloat16, device="cuda")
    DC[:, :N] = torch.from_numpy(p.C.view(np.int16)).cuda().view(torch.bfloat16)
    ws = torch.empty(mx.mxfp4_gemm_workspace_size(M, N, K, 0), dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm(DC, N + pad_n, DC, N + pad_n, A, K + pad_k, B, K + pad_k, SA, K // 32 + pad_s,
                  SB, K // 32 + pad_s, p.alpha, p.beta, M, N, K, 0, ws, ws.numel())
    torch.cuda.synchronize()
    got = d_to_bits(DC[:, :N])
    assert_within_bound(got, Dref, sabs, p.alpha, "strided in-place")
    assert np.all(d_to_bits(DC[:, N:]) == 0)


def test_split_k_is_deterministic():
    p = problem("decode") if "decode" in _PROBLEMS else inputs.workload("decode")
    dev = Dev(p)
    a = run_gemm(dev, split_k=8)
    b = run_gemm(dev, split_k=8)
    assert np.array_equal(a, b)


def test_prepacked_and_host_entry_points_match():
    p = problem("mid")
    dev = Dev(p)
    ref = run_gemm(dev)
    M, N, K = p.M, p.N, p.K
    sfa = torch.empty(mx.mxfp4_scale_relayout_size(M, K), dtype=torch.uint8, device="cuda")
    sfb = torch.empty(mx.mxfp4_scale_relayout_size(N, K), dtype=torch.uint8, device="cuda")
    mx.mxfp4_scale_relayout(sfa, dev.SA, M, K, K // 32)
    mx.mxfp4_scale_relayout(sfb, dev.SB, N, K, K // 32)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    wsb = mx.mxfp4_gemm_prepacked_workspace_size(M, N, K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm_prepacked(D, N, dev.C, N, dev.A, K, dev.B, K, sfa, sfb, p.alpha, p.beta,
                            M, N, K, 0, ws, wsb)
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D), ref)
    # Host buffers in, host buffer out.
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hA, hB, hSA, hSB = pin(p.A), pin(p.B), pin(p.SA), pin(p.SB)
    hC = pin(p.C.view(np.int16))
    hD = torch.zeros((M, N), dtype=torch.int16).pin_memory()
    arena_b = mx.mxfp4_gemm_host_arena_size(M, N, K, 0, True)
    arena = torch.empty(arena_b, dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm_host(hD, hC, hA, hB, hSA, hSB, p.alpha, p.beta, M, N, K, 0, arena, arena_b)
    torch.cuda.synchronize()
    assert np.array_equal(hD.numpy().view(np.uint16), ref)


def test_host_entry_pipelined_panels(oracle_mod):
    """Host buffers with M >= 2048: the call copies B once, then pipelines row
    panels (copy in, GEMM, copy out on separate streams).  2304 rows make five
    panels of 512 / 256 rows; with split_k = 1 each panel runs the same kernel
    and K order as the whole matrix, so D matches the device call bit for bit."""
    M, N, K = 2304, 1024, 1024
    p = inputs.make_problem("panels", M, N, K, seed=21, values="normal", alpha=0.5, beta=0.5,
                            c_sigma=1.0)
    ref = run_gemm(Dev(p), split_k=1)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hA, hB, hSA, hSB = pin(p.A), pin(p.B), pin(p.SA), pin(p.SB)
    hC = pin(p.C.view(np.int16))
    hD = torch.zeros((M, N), dtype=torch.int16).pin_memory()
    arena_b = mx.mxfp4_gemm_host_arena_size(M, N, K, 1, True)
    arena = torch.empty(arena_b, dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm_host(hD, hC, hA, hB, hSA, hSB, p.alpha, p.beta, M, N, K, 1, arena, arena_b)
    torch.cuda.synchronize()
    got = hD.numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    pairs = sample_pairs(M, N, 2000, 21)
    Dr, _, sabs, inexact = oracle_mod.gemm_sampled(p.A, p.B, p.SA, p.SB, M, N, K, pairs,
                                                   alpha=p.alpha, beta=p.beta, C=p.C)
    assert inexact == 0
    assert_within_bound(got[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, "host panels")


def test_host_entry_column_blocks(oracle_mod):
    """M and N >= 2048: the host call also splits the columns in two blocks
    (1536 + a ragged 1064 here), so D returns in strided 2-D copies and the
    second half of B arrives after all of A.  With split_k = 1 every block runs
    the whole K in order, so D matches the device call bit for bit."""
    M, N, K = 2304, 2600, 1024
    p = inputs.make_problem("colblocks", M, N, K, seed=23, values="normal", alpha=0.5, beta=0.5,
                            c_sigma=1.0)
    ref = run_gemm(Dev(p), split_k=1)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hA, hB, hSA, hSB = pin(p.A), pin(p.B), pin(p.SA), pin(p.SB)
    hC = pin(p.C.view(np.int16))
    hD = torch.zeros((M, N), dtype=torch.int16).pin_memory()
    arena_b = mx.mxfp4_gemm_host_arena_size(M, N, K, 1, True)
    arena = torch.empty(arena_b, dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm_host(hD, hC, hA, hB, hSA, hSB, p.alpha, p.beta, M, N, K, 1, arena, arena_b)
    torch.cuda.synchronize()
    got = hD.numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    pairs = sample_pairs(M, N, 2000, 23)
    Dr, _, sabs, inexact = oracle_mod.gemm_sampled(p.A, p.B, p.SA, p.SB, M, N, K, pairs,
                                                   alpha=p.alpha, beta=p.beta, C=p.C)
    assert inexact == 0
    assert_within_bound(got[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, "host column blocks")
    # The heuristic's own split choice per block: within the bound everywhere.
    arena_b = mx.mxfp4_gemm_host_arena_size(M, N, K, 0, True)
    arena = torch.empty(arena_b, dtype=torch.uint8, device="cuda")
    hD.zero_()
    mx.mxfp4_gemm_host(hD, hC, hA, hB, hSA, hSB, p.alpha, p.beta, M, N, K, 0, arena, arena_b)
    torch.cuda.synchronize()
    got = hD.numpy().view(np.uint16)
    assert_within_bound(got[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, "host blocks, split 0")


def test_device_errors_are_reported():
    # Split-K keeps fp32 partials in the workspace: one byte short is an error.
    q = inputs.make_problem("ws16", 256, 512, 4096, 3, "normal", 1.0, 0.0, None)
    dq = Dev(q)
    Dq = torch.empty((q.M, q.N), dtype=torch.bfloat16, device="cuda")
    need = mx.mxfp4_gemm_workspace_size(q.M, q.N, q.K, 16)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_gemm(Dq, q.N, None, 0, dq.A, q.K, dq.B, q.K, dq.SA, q.K // 32, dq.SB,
                      q.K // 32, 1.0, 0.0, q.M, q.N, q.K, 16, ws, need - 1)
    assert e.value.status == -4
    p = problem("tiny")
    dev = Dev(p)
    D = torch.empty((p.M, p.N), dtype=torch.bfloat16, device="cuda")
    # Without split the GEMM needs no workspace at all.
    assert mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, 1) == 0
    mx.mxfp4_gemm(D, p.N, None, 0, dev.A, p.K, dev.B, p.K, dev.SA, p.K // 32, dev.SB,
                  p.K // 32, 1.0, 0.0, p.M, p.N, p.K, 1, None, 0)
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D), run_gemm(dev, split_k=1))


def test_bounded_wait_times_out_cleanly():
    """A wait nothing satisfies gives up after its limit, records
    MXFP4_ERR_TIMEOUT and returns; the context stays usable."""
    assert mx.mxfp4_device_status(reset=True) == 0
    mx.mxfp4_wait_timeout_probe(2_000_000)            # ~1 ms of SM cycles
    torch.cuda.synchronize()
    assert mx.mxfp4_device_status(reset=True) == -6
    assert mx.mxfp4_device_status() == 0
    p = problem("tiny")
    D = run_gemm(Dev(p))
    assert not np.isnan(bf16_bits_to_f64(D)).any()


# ------------------------------------------------------ CTA-pair kernel --
# The heuristic runs the CTA-pair kernel when the 256 x 256 tiles fill every
# SM pair at least once (76 tiles on 152 SMs): these shapes have 81 or more.

PAIR_SHAPES = [(2304, 2304, 512), (2300, 2100, 288), (2560, 2048, 1280), (2304, 2560, 1024)]


@pytest.mark.parametrize("which", ["A", "B"])
def test_pair_kernel_single_scale_probes(which):
    """Scale placement through the two-SM MMA: each CTA's scale-A rows and the
    full scale-B must reach the right accumulator rows / columns."""
    M = N = 2304
    K = 512
    assert mx.mxfp4_plan_gemm(M, N, K, 0, 0).pair == 1
    rows = [0, 31, 127, 128, 200, 255, 256, 1000, M - 1]
    bad = []
    for r in rows:
        for kb in (0, 3, 8, 15):
            p = _ones_problem(M, N, K)
            (p.SA if which == "A" else p.SB)[r, kb] = 128
            D = bf16_bits_to_f64(run_gemm(Dev(p)))
            want = np.full((M, N), float(K))
            if which == "A":
                want[r, :] += 32
            else:
                want[:, r] += 32
            if not np.array_equal(D, want):
                wrong = np.argwhere(D != want)
                bad.append((which, r, kb, len(wrong), wrong[:4].tolist(), D[tuple(wrong[0])]))
    assert not bad, bad


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
def test_pair_kernel_parity(oracle_mod, M, N, K):
    """Full comparison, ragged M / N (tiles past the edge), K with a partial
    last stage, alpha / beta with C."""
    p = inputs.make_problem("pair", M, N, K, seed=M + N + K, values="codes", alpha=0.5,
                            beta=1.0, c_sigma=1.0)
    plan = mx.mxfp4_plan_gemm(M, N, K, 0, 0)
    assert plan.pair == 1 and plan.tile_n == 256
    Dref, sabs = full_oracle(oracle_mod, p)
    assert_within_bound(run_gemm(Dev(p)), Dref, sabs, p.alpha, f"pair {M}x{N}x{K}")


def test_pair_kernel_many_tiles_sampled(oracle_mod):
    """More tiles than resident pairs (several tiles per pair, the
    accumulator reused), ragged in M and N, checked on sampled outputs."""
    M, N, K = 4400, 4700, 1024
    p = inputs.make_problem("pair_many", M, N, K, seed=17, values="codes", alpha=1.0, beta=0.5,
                            c_sigma=1.0)
    plan = mx.mxfp4_plan_gemm(M, N, K, 0, 0)
    assert plan.pair == 1 and plan.waves > 1
    pairs = sample_pairs(M, N, 3000, 5, tile_m=256, tile_n=256)
    Dr, _, sabs, inexact = oracle_mod.gemm_sampled(p.A, p.B, p.SA, p.SB, M, N, K, pairs,
                                                   alpha=p.alpha, beta=p.beta, C=p.C)
    assert inexact == 0
    D = run_gemm(Dev(p))
    assert_within_bound(D[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, f"pair {M}x{N}x{K}")
    assert not np.isnan(bf16_bits_to_f64(D)).any()


# ------------------------------------------------------ split-K reduce --

@pytest.mark.parametrize("split", [2, 10])
def test_splitk_for_large_grids(oracle_mod, split):
    """A wide grid (over 1000 output tiles), each tile's splits summed inside
    the tile's cluster (2 splits) or by the CTA that finishes the tile last
    (10 splits, fp32 partials in the workspace); every tile completes (same
    bound, sampled)."""
    M, N, K = 4224, 8192, 2560
    if "wide" not in _PROBLEMS:
        p = inputs.make_problem("wide", M, N, K, seed=9, values="normal", alpha=1.0, beta=0.0,
                                c_sigma=None)
        pairs = sample_pairs(M, N, 3000, 11)
        Dr, _, sabs, inexact = oracle_mod.gemm_sampled(p.A, p.B, p.SA, p.SB, M, N, K, pairs,
                                                       alpha=p.alpha, beta=p.beta, C=p.C)
        assert inexact == 0
        _PROBLEMS["wide"] = (p, Dev(p), pairs, Dr, sabs)
    p, dev, pairs, Dr, sabs = _PROBLEMS["wide"]
    plan = mx.mxfp4_plan_gemm(M, N, K, split, 0)
    assert plan.split_k == split and plan.grid_x * plan.grid_y > 1024
    assert (plan.workspace_bytes > 0) == (split > 8)
    D = run_gemm(dev, split_k=split)
    assert_within_bound(D[pairs[:, 0], pairs[:, 1]], Dr, sabs, p.alpha, f"wide s={split}")


@pytest.mark.parametrize("kernel", ["auto", "pair"])
def test_d_only_16_byte_aligned(oracle_mod, kernel):
    """D whose rows are 16- but not 32-byte aligned (base offset 8 elements,
    ldd % 16 == 8): the epilogues fall back from 32- to 16-byte stores."""
    M, N, K = (384, 512, 512) if kernel == "auto" else (2304, 2304, 256)
    assert mx.mxfp4_plan_gemm(M, N, K, 0, 0).pair == (kernel == "pair")
    p = inputs.make_problem("d16", M, N, K, seed=31, values="codes", alpha=1.0, beta=1.0,
                            c_sigma=1.0)
    Dref, sabs = full_oracle(oracle_mod, p)
    dev = Dev(p)
    ldd = N + 24
    buf = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    D = buf[:, 8:8 + N]
    assert D.data_ptr() % 32 == 16
    wsb = mx.mxfp4_gemm_workspace_size(M, N, K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm(D, ldd, dev.C, N, dev.A, K, dev.B, K, dev.SA, K // 32, dev.SB, K // 32,
                  p.alpha, p.beta, M, N, K, 0, ws, wsb)
    torch.cuda.synchronize()
    assert_within_bound(d_to_bits(D.contiguous()), Dref, sabs, p.alpha, f"d16 {kernel}")
    assert torch.isnan(buf[:, :8].float()).all() and torch.isnan(buf[:, 8 + N:].float()).all()


# ------------------------------------------------------------- quantiser --

def _quantize_gpu(Xbits, rows, K, ldx=None, ldq=None, lds=None):
    ldx = ldx or K
    ldq = ldq or K
    lds = lds or K // 32
    Xp = np.zeros((rows, ldx), dtype=np.uint16)
    Xp[:, :K] = Xbits
    X = torch.from_numpy(Xp.view(np.int16)).cuda()
    Q = torch.full((rows, ldq // 2), 0xA5, dtype=torch.uint8, device="cuda")
    S = torch.full((rows, lds), 0x5A, dtype=torch.uint8, device="cuda")
    mx.mxfp4_quantize(Q, ldq, S, lds, X, ldx, rows, K)
    torch.cuda.synchronize()
    return Q.cpu().numpy(), S.cpu().numpy()


def _bf16(x):
    return inputs.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


@pytest.mark.parametrize("rows,K", [(1, 32), (37, 96), (128, 1024), (5, 4128), (300, 512)])
def test_quantize_matches_oracle(oracle_mod, rows, K):
    """Codes and scales bit for bit against the oracle on rows whose
    magnitudes span 2^-60 .. 2^60."""
    rng = np.random.default_rng(rows * 1000 + K)
    x = rng.standard_normal((rows, K)) * np.ldexp(1.0, rng.integers(-60, 60, size=(rows, 1)))
    bits = _bf16(x)
    Qw, Sw = oracle_mod.quantize(bits, rows, K)
    Qg, Sg = _quantize_gpu(bits, rows, K)
    assert np.array_equal(Sg, Sw)
    assert np.array_equal(Qg, Qw)


def test_quantize_special_blocks(oracle_mod):
    """All-zero and negative-zero blocks, every rounding tie, saturation at
    the block maximum, bf16 subnormals and values near the bf16 maximum."""
    K = 32 * 12
    x = np.zeros((4, K), dtype=np.float64)
    x[0, 32:64] = -0.0
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -2.5, -5.0, 6.0])
    x[0, 64:64 + ties.size] = ties                               # scale 0: ties as they stand
    x[0, 96:96 + ties.size] = ties * 2.0 ** 20                   # same ties at another scale
    x[1, :32] = np.linspace(-11.9, 11.9, 32)                     # max in [6, 12): saturates
    x[1, 32:64] = np.ldexp(1.0, -133) * np.arange(1, 33)         # bf16 subnormals
    x[1, 64:96] = 3.0e38 * np.linspace(-1, 1, 32)                # near the bf16 maximum
    x[2] = np.where(np.arange(K) % 2, -1e-30, 1e-30)             # tiny against nothing
    x[3] = np.random.default_rng(4).standard_normal(K) * 0.01
    x[3, ::7] = -0.0
    bits = _bf16(x)
    Qw, Sw = oracle_mod.quantize(bits, 4, K)
    Qg, Sg = _quantize_gpu(bits, 4, K)
    assert np.array_equal(Sg, Sw)
    assert np.array_equal(Qg, Qw)


def test_quantize_strided_leaves_padding(oracle_mod):
    rows, K = 9, 256
    x = np.random.default_rng(6).standard_normal((rows, K))
    bits = _bf16(x)
    Qw, Sw = oracle_mod.quantize(bits, rows, K)
    Qg, Sg = _quantize_gpu(bits, rows, K, ldx=K + 24, ldq=K + 64, lds=K // 32 + 5)
    assert np.array_equal(Qg[:, :K // 2], Qw) and np.array_equal(Sg[:, :K // 32], Sw)
    assert (Qg[:, K // 2:] == 0xA5).all() and (Sg[:, K // 32:] == 0x5A).all()


def test_quantize_then_gemm(oracle_mod):
    """bf16 activations and weights through the quantiser, then the GEMM:
    equal to the oracle GEMM on the oracle-quantised operands."""
    M, N, K = 96, 320, 1024
    rng = np.random.default_rng(12)
    xa, xb = _bf16(rng.standard_normal((M, K))), _bf16(rng.standard_normal((N, K)))
    QA, SA = _quantize_gpu(xa, M, K)
    QB, SB = _quantize_gpu(xb, N, K)
    QAo, SAo = oracle_mod.quantize(xa, M, K)
    QBo, SBo = oracle_mod.quantize(xb, N, K)
    assert np.array_equal(QA, QAo) and np.array_equal(SB, SBo)
    p = inputs.Problem("qgemm", M, N, K, QA, QB, SA, SB, None, 1.0, 0.0, 12)
    Dref, sabs = full_oracle(oracle_mod, p)
    assert_within_bound(run_gemm(Dev(p)), Dref, sabs, 1.0, "quantised operands")


# ---------------------------------------------------------- CUDA graphs --

def _gemm_call(dev, D, ws, wsb, split, stream):
    p = dev.p
    C = dev.C if p.beta != 0.0 else None
    mx.mxfp4_gemm(D, D.stride(0), C, 0 if C is None else C.stride(0), dev.A, dev.A.stride(0) * 2,
                  dev.B, dev.B.stride(0) * 2, dev.SA, dev.SA.stride(0), dev.SB, dev.SB.stride(0),
                  float(p.alpha), float(p.beta), p.M, p.N, p.K, split, ws if wsb else None, wsb,
                  stream)


@pytest.mark.parametrize("case", ["decode", "mid", "pair", "split16"])
def test_cuda_graph_capture_and_replay(case):
    """mxfp4_gemm captured into a CUDA graph (dependent launches, cluster
    launches and both split-K reductions included) replays to the eager
    result, and reads its inputs at replay time.  split16 keeps its partials
    and per-tile counters in the workspace: the replays show that each call
    leaves the counters ready for the next one."""
    split = 0
    if case == "pair":
        p = inputs.make_problem("gpair", 2048, 4096, 2048, 41, "normal", 1.0, 0.0, None)
        assert mx.mxfp4_plan_gemm(p.M, p.N, p.K, 0, 0).pair == 1
    elif case == "split16":
        p = problem("decode")
        split = 16
        assert mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, split) > 0
    else:
        p = problem(case)
    dev = Dev(p)
    wsb = mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, split)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    D = torch.empty((p.M, p.N), dtype=torch.bfloat16, device="cuda")
    ref = run_gemm(dev, split_k=split)                    # eager; also the first-use setup
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _gemm_call(dev, D, ws, wsb, split, s)
    for _ in range(3):
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(d_to_bits(D), ref)
    # New B values, same buffers: the replay sees them.
    dev.B.copy_(torch.roll(dev.B, 1, 0))
    ref2 = run_gemm(dev, split_k=split)
    D.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D), ref2)


def test_cuda_graph_host_entry_and_mxfp8():
    """The pipelined host-buffer calls (copy streams forked from and joined
    to the captured stream) and mxfp8_gemm, captured and replayed."""
    M, N, K = 2304, 1024, 1024
    p = inputs.make_problem("ghost", M, N, K, seed=43, values="normal", alpha=1.0, beta=0.0,
                            c_sigma=None)
    ref = run_gemm(Dev(p), split_k=1)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hA, hB, hSA, hSB = pin(p.A), pin(p.B), pin(p.SA), pin(p.SB)
    hD = torch.zeros((M, N), dtype=torch.int16).pin_memory()
    arena_b = mx.mxfp4_gemm_host_arena_size(M, N, K, 1, False)
    arena = torch.empty(arena_b, dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm_host(hD, None, hA, hB, hSA, hSB, 1.0, 0.0, M, N, K, 1, arena, arena_b)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.mxfp4_gemm_host(hD, None, hA, hB, hSA, hSB, 1.0, 0.0, M, N, K, 1, arena, arena_b, s)
    hD.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(hD.numpy().view(np.uint16), ref)

    # The same pipeline on the byte forms (mxfp8_gemm_host), E2M3 x E4M3.
    q = inputs.make_problem8("gh8", M, N, K, 45, "e2m3", "e4m3", "normal", 1.0, 0.0, None)
    qA, qB, qSA, qSB = pin(q.A), pin(q.B), pin(q.SA), pin(q.SB)
    arena8_b = mx.mxfp8_gemm_host_arena_size(M, N, K, 1, False)
    arena8 = torch.empty(arena8_b, dtype=torch.uint8, device="cuda")
    hcall = lambda st: mx.mxfp8_gemm_host(hD, None, qA, qB, qSA, qSB, mx.MXFP6_E2M3,
                                          mx.MXFP8_E4M3, 1.0, 0.0, M, N, K, 1, arena8, arena8_b,
                                          st)
    hcall(None)
    torch.cuda.synchronize()
    ref8 = hD.numpy().copy()
    gh = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gh, stream=s):
        hcall(s)
    hD.zero_()
    gh.replay()
    torch.cuda.synchronize()
    assert np.array_equal(hD.numpy(), ref8)

    q = inputs.make_problem8("g8", 300, 520, 1024, 44, "e4m3", "e5m2", "normal", 1.0, 0.0, None)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    A8, B8, SA8, SB8 = d(q.A), d(q.B), d(q.SA), d(q.SB)
    D8 = torch.empty((q.M, q.N), dtype=torch.bfloat16, device="cuda")
    wsb = mx.mxfp8_gemm_workspace_size(q.M, q.N, q.K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    call = lambda st: mx.mxfp8_gemm(D8, q.N, None, 0, A8, q.K, B8, q.K, SA8, q.K // 32, SB8,
                                    q.K // 32, mx.MXFP8_E4M3, mx.MXFP8_E5M2, 1.0, 0.0, q.M, q.N,
                                    q.K, 0, ws if wsb else None, wsb, st)
    call(None)
    torch.cuda.synchronize()
    ref8 = d_to_bits(D8)
    g8 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g8, stream=s):
        call(s)
    D8.fill_(float("nan"))
    g8.replay()
    torch.cuda.synchronize()
    assert np.array_equal(d_to_bits(D8), ref8)


@pytest.mark.parametrize("M,N,K", [(100, 65535 * 256, 64), (1 << 22, 1024, 64)],
                         ids=["grid-y-65535", "D-beyond-2^31-elements"])
def test_maximum_sizes_sampled(oracle_mod, M, N, K):
    """The largest one-tile grid (65535 tile columns of 256) and an output of
    more than 2^31 elements (64-bit row offsets, pair kernel), checked on
    sampled outputs that include the first and last rows and columns."""
    rng = np.random.default_rng(M + N)
    A = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    SA = rng.integers(120, 135, size=(M, K // 32), dtype=np.uint8)
    SB = rng.integers(120, 135, size=(N, K // 32), dtype=np.uint8)
    d = lambda x: torch.from_numpy(x).cuda()
    dA, dB, dSA, dSB = d(A), d(B), d(SA), d(SB)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    wsb = mx.mxfp4_gemm_workspace_size(M, N, K, 0)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    mx.mxfp4_gemm(D, N, None, 0, dA, K, dB, K, dSA, K // 32, dSB, K // 32, 1.0, 0.0,
                  M, N, K, 0, ws, wsb)
    torch.cuda.synchronize()
    pairs = np.concatenate([sample_pairs(M, N, 600, 7),
                            np.array([[M - 1, N - 1], [M - 1, 0], [0, N - 1]], dtype=np.int64)])
    idx = torch.from_numpy(pairs).cuda()
    got = D[idx[:, 0], idx[:, 1]].view(torch.int16).cpu().numpy().view(np.uint16)
    del D
    torch.cuda.empty_cache()
    Dr, _, sabs, inexact = oracle_mod.gemm_sampled(A, B, SA, SB, M, N, K, pairs)
    assert inexact == 0
    assert_within_bound(got, Dr, sabs, 1.0, f"maximum sizes {M}x{N}x{K}")
