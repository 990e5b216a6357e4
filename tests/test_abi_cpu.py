"""Host-side checks of the C ABI that need no GPU.

The library loads, exports every function the public header declares, and
its host logic (plan heuristic, workspace sizes, argument validation that
returns before any device call) behaves as documented.
"""
import ctypes
import os
import subprocess

import pytest

import block_scaled_mxfp4_gb300 as mx
from block_scaled_mxfp4_gb300 import build as mxbuild


@pytest.fixture(scope="module")
def L():
    mxbuild.build()
    return mx.lib()


def test_library_exports_every_header_symbol(L):
    names = mx.header_functions()
    assert len(names) >= 14
    out = subprocess.run(["nm", "-D", "--defined-only", mx.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, n
        assert getattr(L, n) is not None


def test_library_is_sm103a_only():
    # One -gencode, no PTX for other targets.
    assert mxbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version_and_strerror(L):
    assert mx.mxfp4_version() == 10000
    for code in range(-7, 1):
        s = mx.mxfp4_strerror(code)
        assert s and s != "unknown status"
    assert mx.mxfp4_strerror(-99) == "unknown status"


def _a256(x):
    return -(-x // 256) * 256


def splitk_ws(tiles, split, part_cols):
    """Split-K workspace: up to 8 splits reduce inside each tile's cluster and
    need none; more keep one 8-byte counter per tile, then one 128-row fp32
    partial slot of part_cols columns (rounded up to 4) per (tile, split),
    each part 256-byte aligned."""
    if split <= 8:
        return 0
    return _a256(tiles * 8) + _a256(tiles * split * 128 * (-(-part_cols // 4) * 4) * 4)


WORKLOADS = {"tiny": (128, 256, 512), "decode": (1, 8192, 8192), "mid": (512, 1024, 2048),
             "large": (8192, 8192, 8192), "skinny": (64, 7168, 16384)}


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_plan_invariants(L, name):
    M, N, K = WORKLOADS[name]
    for split in range(0, 17):
        p = mx.mxfp4_plan_gemm(M, N, K, split, 152)
        kt = -(-K // p.tile_k)
        assert p.tile_m == (256 if p.pair else 128) and p.tile_k == 256
        assert p.split_k >= 1 and p.split_k <= 16
        assert p.k_tiles_per_split * (p.split_k - 1) < kt <= p.k_tiles_per_split * p.split_k
        P, Q = (N, M) if p.swap_ab else (M, N)
        tiles = -(-P // 128) * -(-Q // p.tile_n)
        if split == 0:
            # Automatic split: none when the tiles fill half a wave, else as
            # many as fill the resident CTA slots with >= 8 K stages each.
            slots = 152 * (2 if p.swap_ab else 1)
            if p.pair:
                # 256 x 256 tiles filling all 76 SM pairs at least once.
                assert not p.swap_ab and M >= 256 and N >= 256
                assert -(-M // 256) * -(-N // 256) >= 76
                assert (p.tile_m, p.tile_n, p.split_k, p.ctas) == (256, 256, 1, 152)
                continue
            want = 1 if 2 * tiles >= slots else max(1, min(slots // tiles, kt // 8, 16, kt))
            per = -(-kt // want)
            assert p.split_k == -(-kt // per)
            assert p.grid_z == p.split_k
            continue
        assert p.split_k <= split
        assert p.grid_x == -(-P // 128) and p.grid_y == -(-Q // p.tile_n)
        assert p.grid_z == p.split_k
        assert p.workspace_bytes == splitk_ws(tiles, p.split_k, min(Q, p.tile_n))
    # Skinny M swaps; large uses the pair kernel.
    p = mx.mxfp4_plan_gemm(M, N, K, 0, 152)
    assert p.swap_ab == (1 if M <= 64 else 0)
    if name == "large":
        assert (p.pair, p.tile_m, p.tile_n, p.split_k) == (1, 256, 256, 1)
    else:
        assert p.pair == 0
    if name in ("decode", "skinny"):
        assert p.split_k == {"decode": 4, "skinny": 5}[name]


def test_plan_ignores_the_environment(L, monkeypatch):
    """The plan is a function of the shape alone: the variables that once
    switched kernels for tuning have no effect."""
    shapes = [(8192, 8192, 8192), (1, 8192, 8192), (64, 7168, 16384), (512, 1024, 2048)]
    before = [mx.mxfp4_plan_gemm(*s, 0, 152).as_dict() for s in shapes]
    for var, val in [("MXFP4_KERNEL", "persistent"), ("MXFP4_KERNEL", "gemv"),
                     ("MXFP4_PAIR_N", "192"), ("MXFP4_PAIR_CLUSTER", "2"),
                     ("MXFP4_PAIR_KS", "512"), ("MXFP4_SPLIT_REDUCE", "cluster"),
                     ("MXFP4_TILE", "128:6")]:
        monkeypatch.setenv(var, val)
    assert [mx.mxfp4_plan_gemm(*s, 0, 152).as_dict() for s in shapes] == before


def test_no_multicast_loads_in_the_library():
    """No TMA load with cluster multicast anywhere in the library sources
    (the pair kernel's commit may arrive on both CTAs' barriers)."""
    import glob
    import re
    csrc = os.path.join(os.path.dirname(mx.library_path()), "csrc")
    for path in glob.glob(os.path.join(csrc, "*")):
        text = open(path).read()
        for m in re.finditer(r"multicast::cluster", text):
            line = text[text.rfind("\n", 0, m.start()) + 1:text.find("\n", m.start())]
            assert "tcgen05.commit" in line, (path, line)
        assert "cp.async.bulk.tensor" not in text or \
            not re.search(r"cp\.async\.bulk\.tensor[^;\"]*multicast", text), path


def test_plan_heuristic_prefers_fewer_waves(L):
    # 8192^2 output: 128x256 tiles need 14 waves on 152 SMs, 128x128 need 27.
    assert mx.mxfp4_plan_gemm(8192, 8192, 8192, 1, 152).tile_n == 256
    # 512x1024: both fit in one wave; 128x128 fills more SMs.
    assert mx.mxfp4_plan_gemm(512, 1024, 2048, 0, 152).tile_n == 128
    # Deterministic.
    a = mx.mxfp4_plan_gemm(300, 2048, 1024, 0, 152).as_dict()
    b = mx.mxfp4_plan_gemm(300, 2048, 1024, 0, 152).as_dict()
    assert a == b


def test_sizes(L):
    assert mx.mxfp4_scale_relayout_size(1, 32) == 2 * 2 * 512
    assert mx.mxfp4_scale_relayout_size(256, 512) == 2 * 4 * 512
    assert mx.mxfp4_scale_relayout_size(257, 512) == 4 * 4 * 512
    assert mx.mxfp4_scale_relayout_size(0, 512) == 0
    assert mx.mxfp4_scale_relayout_size(5, 48) == 0
    assert mx.mxfp4_gemm_workspace_size(0, 1, 32, 0) == 0
    assert mx.mxfp4_gemm_workspace_size(1, 1, 32, 17) == 0
    # The decode and skinny shapes split K four and five ways: the splits of a
    # tile reduce inside their cluster, so no workspace.
    assert mx.mxfp4_gemm_workspace_size(1, 8192, 8192, 4) == 0
    p = mx.mxfp4_plan_gemm(1, 8192, 8192, 0, 152)
    assert p.split_k == 4 and p.workspace_bytes == 0
    p = mx.mxfp4_plan_gemm(64, 7168, 16384, 0, 152)
    assert p.split_k == 5 and p.workspace_bytes == 0
    # Sixteen splits of decode: 64 counters and 16 x 64 partial slots of 128
    # rows x 4 columns (M = 1, rounded up to a chunk of 4).
    assert mx.mxfp4_gemm_workspace_size(1, 8192, 8192, 16) == 512 + 16 * 64 * 128 * 16
    # The large shape relays its scales out first: workspace = both relaid buffers.
    p = mx.mxfp4_plan_gemm(8192, 8192, 8192, 1, 0)
    assert p.relayout_pass == 1
    assert mx.mxfp4_gemm_workspace_size(8192, 8192, 8192, 1) == \
        2 * mx.mxfp4_scale_relayout_size(8192, 8192)
    assert mx.mxfp4_plan_gemm(1, 8192, 8192, 0, 0).relayout_pass == 0
    assert mx.mxfp4_gemm_workspace_size(128, 256, 512, 1) == 0
    assert mx.mxfp4_gemm_host_arena_size(8192, 8192, 8192, 1, False) > 0


def _call_gemm(L, **kw):
    args = dict(D=0x1000, ldd=256, C=None, ldc=0, A=0x2000, lda=512, B=0x3000, ldb=512,
                SA=0x4000, ld_sa=16, SB=0x5000, ld_sb=16, alpha=1.0, beta=0.0, M=128, N=256,
                K=512, split=0, ws=0x10000, wsb=1 << 30, stream=None)
    args.update(kw)
    return L.mxfp4_gemm(args["D"], args["ldd"], args["C"], args["ldc"], args["A"], args["lda"],
                        args["B"], args["ldb"], args["SA"], args["ld_sa"], args["SB"],
                        args["ld_sb"], args["alpha"], args["beta"], args["M"], args["N"],
                        args["K"], args["split"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=None), -1), (dict(A=None), -1), (dict(B=None), -1),
    (dict(SA=None), -1), (dict(SB=None), -1),
    (dict(M=0), -1), (dict(N=0), -1), (dict(K=0), -1), (dict(K=48, lda=64, ldb=64), -1),
    (dict(lda=256), -1), (dict(ldb=500), -1), (dict(ldd=255), -1),
    (dict(ld_sa=15), -1), (dict(ld_sb=1), -1),
    (dict(beta=1.0), -1), (dict(beta=1.0, C=0x6000, ldc=100), -1),
    (dict(split=17), -1), (dict(split=-1), -1),
    (dict(lda=528), -3), (dict(ldb=520), -3), (dict(A=0x2008), -3), (dict(B=0x3004), -3),
    # Split K keeps fp32 partials in the workspace (K = 4096: 16 stages).
    (dict(ws=None, split=16, K=4096, lda=4096, ldb=4096, ld_sa=128, ld_sb=128), -4),
    (dict(ws=0x10010), -3),
    (dict(wsb=1000, split=16, K=4096, lda=4096, ldb=4096, ld_sa=128, ld_sb=128), -4),
])
def test_gemm_argument_validation(L, kw, status):
    # These return before any device call, so they run without a GPU.
    assert _call_gemm(L, **kw) == status


def _call_gemm8(L, **kw):
    args = dict(D=0x1000, ldd=256, C=None, ldc=0, A=0x2000, lda=512, B=0x3000, ldb=512,
                SA=0x4000, ld_sa=16, SB=0x5000, ld_sb=16, fa=0, fb=1, alpha=1.0, beta=0.0,
                M=128, N=256, K=512, split=0, ws=0x10000, wsb=1 << 30, stream=None)
    args.update(kw)
    return L.mxfp8_gemm(args["D"], args["ldd"], args["C"], args["ldc"], args["A"], args["lda"],
                        args["B"], args["ldb"], args["SA"], args["ld_sa"], args["SB"],
                        args["ld_sb"], args["fa"], args["fb"], args["alpha"], args["beta"],
                        args["M"], args["N"], args["K"], args["split"], args["ws"], args["wsb"],
                        args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=None), -1), (dict(A=None), -1), (dict(SA=None), -1),
    (dict(fa=2), -1), (dict(fb=-1), -1),
    (dict(M=0), -1), (dict(K=48, lda=64, ldb=64), -1), (dict(K=0), -1),
    (dict(lda=500), -1), (dict(ldb=256), -1), (dict(ld_sa=15), -1),
    (dict(beta=1.0), -1), (dict(split=17), -1),
    (dict(lda=520), -3), (dict(ldb=536), -3), (dict(A=0x2008), -3),
    (dict(ws=None, split=16, K=2048, lda=2048, ldb=2048, ld_sa=64, ld_sb=64), -4),
    (dict(ws=0x10010), -3),
])
def test_mxfp8_argument_validation(L, kw, status):
    # lda / ldb count 8-bit elements (bytes): >= K and a multiple of 16.
    assert _call_gemm8(L, **kw) == status


def _call_gemm_nv(L, **kw):
    args = dict(D=0x1000, ldd=256, C=None, ldc=0, A=0x2000, lda=512, B=0x3000, ldb=512,
                SA=0x4000, ld_sa=32, SB=0x5000, ld_sb=32, alpha=1.0, beta=0.0, M=128, N=256,
                K=512, ws=0x10000, wsb=1 << 30, stream=None)
    args.update(kw)
    return L.nvfp4_gemm(args["D"], args["ldd"], args["C"], args["ldc"], args["A"], args["lda"],
                        args["B"], args["ldb"], args["SA"], args["ld_sa"], args["SB"],
                        args["ld_sb"], args["alpha"], args["beta"], args["M"], args["N"],
                        args["K"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=None), -1), (dict(A=None), -1), (dict(SA=None), -1), (dict(SB=None), -1),
    (dict(M=0), -1), (dict(K=48), -1), (dict(K=0), -1),
    (dict(ld_sa=31), -1), (dict(ld_sb=16), -1),          # one scale per 16 K: 32 per row
    (dict(beta=1.0), -1), (dict(lda=520), -3), (dict(A=0x2008), -3),
    (dict(ws=None), -4), (dict(wsb=1024), -4), (dict(ws=0x10010), -3),
])
def test_nvfp4_argument_validation(L, kw, status):
    # These return before any device call, so they run without a GPU.
    assert _call_gemm_nv(L, **kw) == status


def test_nvfp4_workspace_size():
    # Two relaid scale buffers: row blocks (even count) x four 512-byte atoms
    # per 256 K, each buffer rounded up to 256 bytes.
    assert mx.nvfp4_gemm_workspace_size(256, 256, 256) == 2 * (2 * 4 * 512)
    assert mx.nvfp4_gemm_workspace_size(257, 256, 288) == 4 * 8 * 512 + 2 * 8 * 512
    assert mx.nvfp4_gemm_workspace_size(8192, 8192, 8192) == 2 * (64 * 128 * 512)
    assert mx.nvfp4_gemm_workspace_size(0, 256, 256) == 0
    assert mx.nvfp4_gemm_workspace_size(256, 256, 48) == 0


def test_mxfp8_prepacked_validates_before_device(L):
    f = L.mxfp8_gemm_prepacked
    ok = (0x1000, 256, None, 0, 0x2000, 512, 0x3000, 512, 0x4000, 0x5000, 0, 1, 1.0, 0.0, 128, 256,
          512, 0, 0x10000, 1 << 30, None)
    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    for bad in (2, 6, -1):                        # format codes other than 0, 1, 3, 4, 5
        assert call(a10=bad) == -1
        assert call(a11=bad) == -1
    assert call(a8=None) == -1                    # relaid scale A
    assert call(a8=0x4008) == -3                  # relaid scales 16-byte aligned
    assert call(a5=520) == -3                     # lda % 16
    assert call(a16=48, a5=64, a7=64) == -1       # K % 32


def test_mxfp8_quantize_validates_before_device(L):
    q = L.mxfp8_quantize
    assert q(0x1000, 64, 0x2000, 2, 0x3000, 64, 4, 64, 2, None) == -1   # format
    assert q(0x1000, 64, 0x2000, 2, 0x3000, 64, 4, 48, 0, None) == -1   # K % 32
    assert q(0x1000, 32, 0x2000, 2, 0x3000, 64, 4, 64, 0, None) == -1   # ldq < K
    assert q(0x1000, 64, 0x2000, 1, 0x3000, 64, 4, 64, 1, None) == -1   # lds < K/32
    assert q(None, 64, 0x2000, 2, 0x3000, 64, 4, 64, 0, None) == -1
    assert q(0x1000, 72, 0x2000, 2, 0x3000, 72, 4, 64, 0, None) == -3   # ldq % 16
    assert q(0x1008, 64, 0x2000, 2, 0x3000, 64, 4, 64, 0, None) == -3   # Q alignment
    assert q(0x1000, 64, 0x2000, 2, 0x3008, 64, 4, 64, 0, None) == -3   # X alignment


def test_mxfp8_plan(L):
    p = mx.mxfp8_plan_gemm(8192, 8192, 8192, 0, 152)
    assert (p.tile_m, p.tile_n, p.tile_k, p.stages, p.pair) == (128, 256, 128, 4, 0)
    assert p.relayout_pass == 1
    # The plan of an fp4 GEMM whose rows hold as many bytes (K doubled).
    for M, N, K in [(1, 8192, 8192), (64, 7168, 16384), (512, 1024, 2048), (300, 520, 1024)]:
        a = mx.mxfp8_plan_gemm(M, N, K, 0, 152).as_dict()
        monkey = mx.mxfp4_plan_gemm(M, N, 2 * K, 0, 152).as_dict()
        a.pop("tile_k"), monkey.pop("tile_k")
        if not monkey["pair"]:
            assert a == monkey, (M, N, K)
    # The pair kernel is MXFP4-only.
    assert mx.mxfp8_plan_gemm(8192, 8192, 8192, 0, 152).pair == 0
    with pytest.raises(mx.Mxfp4Error):
        mx.mxfp8_plan_gemm(128, 256, 48, 0, 152)
    assert mx.mxfp8_gemm_workspace_size(128, 256, 512, 1) == 0
    assert mx.mxfp8_gemm_workspace_size(8192, 8192, 8192, 0) == \
        2 * mx.mxfp4_scale_relayout_size(8192, 8192)


def test_other_entry_points_validate_before_device(L):
    assert L.mxfp4_scale_relayout(None, 0x1000, 4, 64, 2, None) == -1
    assert L.mxfp4_scale_relayout(0x1000, 0x2000, 4, 48, 2, None) == -1
    assert L.mxfp4_scale_relayout(0x1000, 0x2000, 4, 64, 1, None) == -1
    assert L.mxfp4_scale_relayout(0x1008, 0x2000, 4, 64, 2, None) == -3
    ex = L.mxfp4_gemm_ex
    good = (0x1000, 256, None, 0, 0x2000, 512, 0x3000, 512, 0x4000, 16, 0x5000, 16, 1.0, 0.0,
            128, 256, 512, 0)
    assert ex(*good, 2, 0x10000, 1 << 30, None) == -1          # unknown flag bit
    assert ex(*good, 0x80000000, 0x10000, 1 << 30, None) == -1
    assert ex(None, *good[1:], 1, 0x10000, 1 << 30, None) == -1
    qz = L.mxfp4_quantize
    assert qz(None, 64, 0x2000, 2, 0x3000, 64, 4, 64, None) == -1
    assert qz(0x1000, 64, 0x2000, 2, 0x3000, 64, 4, 48, None) == -1      # K % 32
    assert qz(0x1000, 32, 0x2000, 2, 0x3000, 64, 4, 64, None) == -1      # ldq < K
    assert qz(0x1000, 64, 0x2000, 1, 0x3000, 64, 4, 64, None) == -1      # lds < K/32
    assert qz(0x1000, 64, 0x2000, 2, 0x3000, 64, 0, 64, None) == -1      # rows
    assert qz(0x1000, 64, 0x2000, 2, 0x3008, 64, 4, 64, None) == -3      # X alignment
    assert qz(0x1000, 64, 0x2000, 2, 0x3000, 68, 4, 64, None) == -3      # ldx % 8
    assert qz(0x1000, 80, 0x2000, 2, 0x3000, 64, 4, 64, None) == -3      # ldq % 32
    r2 = L.mxfp4_scale_relayout2
    assert r2(None, 0x2000, 4, 2, 0x3000, 0x4000, 4, 2, 64, None) == -1
    assert r2(0x1000, 0x2000, 4, 2, 0x3000, 0x4000, 0, 2, 64, None) == -1
    assert r2(0x1000, 0x2000, 4, 2, 0x3000, 0x4000, 4, 1, 64, None) == -1
    assert r2(0x1000, 0x2000, 4, 2, 0x3000, 0x4000, 4, 2, 48, None) == -1
    assert r2(0x1000, 0x2000, 4, 2, 0x3008, 0x4000, 4, 2, 64, None) == -3
    assert L.mxfp4_gemm_prepacked(0x1000, 256, None, 0, 0x2000, 512, 0x3000, 512, None, 0x5000,
                                  1.0, 0.0, 128, 256, 512, 0, None, 0, None) == -1
    assert L.mxfp4_gemm_prepacked(0x1000, 256, None, 0, 0x2000, 512, 0x3000, 512, 0x4008, 0x5000,
                                  1.0, 0.0, 128, 256, 512, 0, None, 0, None) == -3
    assert L.mxfp4_gemm_host(None, None, 1, 1, 1, 1, 1.0, 0.0, 1, 1, 32, 0, 0x1000, 1 << 20,
                             None) == -1
    assert L.mxfp4_gemm_host(1, None, 1, 1, 1, 1, 1.0, 1.0, 1, 1, 32, 0, 0x1000, 1 << 20,
                             None) == -1
    assert L.mxfp4_gemm_host(1, None, 1, 1, 1, 1, 1.0, 0.0, 1, 1, 32, 0, 0x1000, 16, None) == -4
    assert L.mxfp4_wait_timeout_probe(0, None) == -1
    assert L.mxfp4_device_status(None, 0) == -1
    plan = mx.Plan()
    assert L.mxfp4_plan_gemm(1, 1, 33, 0, 152, ctypes.byref(plan)) == -1
    assert L.mxfp4_plan_gemm(1, 1, 32, 0, 152, None) == -1


def test_no_device_reports_cuda_error_not_crash(L):
    # With arguments valid, the first device query fails cleanly on a machine
    # without a GPU (and succeeds on one), never crashes.
    if os.environ.get("CUDA_VISIBLE_DEVICES", None) is None:
        try:
            import torch
            has_gpu = torch.cuda.is_available()
        except Exception:
            has_gpu = False
        if has_gpu:
            pytest.skip("a GPU is visible")
    st = ctypes.c_int(123)
    assert L.mxfp4_device_status(ctypes.byref(st), 0) in (-5, -7)


def test_plan_respects_the_grid_limit():
    """The one-tile launch puts tile columns on grid.y (<= 65535): the plan
    takes a wider tile when the narrower one would exceed it, rejects the
    shape when no tile fits, and the persistent pair kernel has no such limit."""
    p = mx.mxfp4_plan_gemm(100, 65535 * 256, 64, 0, 152)
    assert p.tile_n == 256 and p.grid_y == 65535 and p.pair == 0
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_plan_gemm(100, 65535 * 256 + 1, 64, 0, 152)
    assert e.value.status == -2                       # MXFP4_ERR_UNSUPPORTED_SHAPE
    q = mx.mxfp4_plan_gemm(300, 65535 * 256 + 1, 256, 0, 152)
    assert q.pair == 1 and q.grid_y == 1


def test_mxfp8_host_entry_validates_before_device(L):
    """mxfp8_gemm_host checks pointers, C with beta, the formats and the
    arena size before touching a device; its arena holds one byte per
    element of A and B (twice the MXFP4 operand bytes)."""
    f = L.mxfp8_gemm_host
    base = [1, None, 1, 1, 1, 1, 0, 0, 1.0, 0.0, 1, 1, 32, 0, 0x1000, 1 << 20, None]
    def call(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a0=None) == -1                       # D_host
    assert call(a9=1.0) == -1                        # beta != 0 without C
    for bad in (2, 6, -1):
        assert call(a6=bad) == -1 and call(a7=bad) == -1
    assert call(a15=16) == -4                        # arena too small
    assert call(a14=0x1008) == -3                    # arena alignment
    M, N, K = 4096, 3072, 2048
    a8 = mx.mxfp8_gemm_host_arena_size(M, N, K, 1, False)
    a4 = mx.mxfp4_gemm_host_arena_size(M, N, K, 1, False)
    assert a8 - a4 >= (M + N) * K // 2
    assert mx.mxfp8_gemm_host_arena_size(M, N, 33, 1, False) == 0
