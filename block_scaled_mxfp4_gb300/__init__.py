"""Python binding of the GB300 block-scaled MXFP4 GEMM C ABI (include/mxfp4_gemm.h).

    D[M,N] (bf16) = alpha * A[M,K] (mxfp4) * B[N,K]^T (mxfp4) + beta * C[M,N]

The functions named like the C entry points marshal arguments only (torch
tensors or raw integer pointers -> void*, the current torch stream by
default); every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the compiled library is missing, loading fails.
``gemm`` is a convenience wrapper that allocates D and the workspace with
torch and calls ``mxfp4_gemm``.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

__all__ = [
    "Mxfp4Error", "lib", "library_path", "header_functions",
    "mxfp4_gemm", "mxfp4_gemm_ex", "mxfp4_gemm_prepacked", "mxfp4_gemm_noalloc",
    "mxfp4_gemm_host", "MXFP4_FLAG_B_STATIC",
    "mxfp4_scale_relayout", "mxfp4_scale_relayout2", "mxfp4_quantize",
    "mxfp4_plan_gemm", "mxfp4_gemm_workspace_size", "mxfp4_gemm_prepacked_workspace_size",
    "mxfp4_scale_relayout_size", "mxfp4_gemm_host_arena_size", "mxfp4_device_status",
    "mxfp4_wait_timeout_probe", "mxfp4_set_wait_limit",
    "mxfp4_strerror", "mxfp4_version",
    "mxfp8_gemm", "mxfp8_gemm_prepacked", "mxfp8_plan_gemm", "mxfp8_gemm_workspace_size",
    "mxfp8_gemm_prepacked_workspace_size", "mxfp8_quantize", "mxfp8_gemm_host",
    "mxfp8_gemm_host_arena_size", "nvfp4_gemm", "nvfp4_gemm_workspace_size",
    "MXFP8_E4M3", "MXFP8_E5M2", "MXFP6_E2M3", "MXFP6_E3M2", "MXFP4_E2M1_PADDED",
    "gemm", "Plan",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
HEADER = os.path.join(_ROOT, "include", "mxfp4_gemm.h")
_LIB_NAME = "libmxfp4_gb300.so"

MXFP4_OK = 0
MXFP4_FLAG_B_STATIC = 1
MXFP8_E4M3, MXFP8_E5M2, MXFP6_E2M3, MXFP6_E3M2, MXFP4_E2M1_PADDED = 0, 1, 3, 4, 5
STATUS_NAMES = {0: "MXFP4_OK", -1: "MXFP4_ERR_INVALID_ARG", -2: "MXFP4_ERR_UNSUPPORTED_SHAPE",
                -3: "MXFP4_ERR_MISALIGNED", -4: "MXFP4_ERR_WORKSPACE", -5: "MXFP4_ERR_CUDA",
                -6: "MXFP4_ERR_TIMEOUT", -7: "MXFP4_ERR_ARCH"}


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status})")


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


class Plan(ctypes.Structure):
    _fields_ = [("swap_ab", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("tile_k", ctypes.c_int), ("stages", ctypes.c_int), ("split_k", ctypes.c_int),
                ("k_tiles_per_split", ctypes.c_int), ("grid_x", ctypes.c_int),
                ("grid_y", ctypes.c_int), ("grid_z", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t), ("relayout_pass", ctypes.c_int),
                ("pair", ctypes.c_int), ("ctas", ctypes.c_int), ("waves", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_lib = None


def lib() -> ctypes.CDLL:
    """Load the compiled library (build it first with block_scaled_mxfp4_gb300.build)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: the CUDA library must be built "
                              "(python -m block_scaled_mxfp4_gb300.build); there is no fallback")
        L = ctypes.CDLL(path)
        vp, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_float, ctypes.c_size_t)
        sigs = {
            "mxfp4_plan_gemm": (i32, [i32, i32, i32, i32, i32, ctypes.POINTER(Plan)]),
            "mxfp4_gemm_workspace_size": (sz, [i32, i32, i32, i32]),
            "mxfp4_gemm_prepacked_workspace_size": (sz, [i32, i32, i32, i32]),
            "mxfp4_scale_relayout_size": (sz, [i32, i32]),
            "mxfp4_gemm_host_arena_size": (sz, [i32, i32, i32, i32, i32]),
            "mxfp4_scale_relayout": (i32, [vp, vp, i32, i32, i64, vp]),
            "mxfp4_scale_relayout2": (i32, [vp, vp, i32, i64, vp, vp, i32, i64, i32, vp]),
            "mxfp4_quantize": (i32, [vp, i64, vp, i64, vp, i64, i32, i32, vp]),
            "mxfp4_gemm": (i32, [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                 f32, f32, i32, i32, i32, i32, vp, sz, vp]),
            "mxfp4_gemm_ex": (i32, [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                    f32, f32, i32, i32, i32, i32, ctypes.c_uint, vp, sz, vp]),
            "mxfp8_gemm": (i32, [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                 i32, i32, f32, f32, i32, i32, i32, i32, vp, sz, vp]),
            "mxfp8_gemm_prepacked": (i32, [vp, i64, vp, i64, vp, i64, vp, i64, vp, vp, i32, i32,
                                           f32, f32, i32, i32, i32, i32, vp, sz, vp]),
            "mxfp8_gemm_prepacked_workspace_size": (sz, [i32, i32, i32, i32]),
            "mxfp8_plan_gemm": (i32, [i32, i32, i32, i32, i32, ctypes.POINTER(Plan)]),
            "mxfp8_quantize": (i32, [vp, i64, vp, i64, vp, i64, i32, i32, i32, vp]),
            "mxfp8_gemm_workspace_size": (sz, [i32, i32, i32, i32]),
            "nvfp4_gemm": (i32, [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                 f32, f32, i32, i32, i32, vp, sz, vp]),
            "nvfp4_gemm_workspace_size": (sz, [i32, i32, i32]),
            "mxfp4_gemm_prepacked": (i32, [vp, i64, vp, i64, vp, i64, vp, i64, vp, vp,
                                           f32, f32, i32, i32, i32, i32, vp, sz, vp]),
            "mxfp4_gemm_noalloc": (i32, [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                         f32, f32, i32, i32, i32, i32, vp]),
            "mxfp4_gemm_host": (i32, [vp, vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32,
                                      vp, sz, vp]),
            "mxfp8_gemm_host": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, f32, f32, i32, i32, i32,
                                      i32, vp, sz, vp]),
            "mxfp8_gemm_host_arena_size": (sz, [i32, i32, i32, i32, i32]),
            "mxfp4_device_status": (i32, [ctypes.POINTER(ctypes.c_int), i32]),
            "mxfp4_wait_timeout_probe": (i32, [ctypes.c_longlong, vp]),
            "mxfp4_set_wait_limit": (None, [ctypes.c_longlong]),
            "mxfp4_strerror": (ctypes.c_char_p, [i32]),
            "mxfp4_version": (i32, []),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions(path: str = HEADER):
    """Names of the functions declared in the public header."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp4_\w+)\s*\(", text)))


def _p(x) -> Optional[int]:
    """Tensor / integer / None -> raw pointer value."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):                      # numpy array
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> int:
    if status != MXFP4_OK:
        raise Mxfp4Error(status, where)
    return status


def mxfp4_plan_gemm(M, N, K, split_k=0, num_sms=0) -> Plan:
    plan = Plan()
    _check(lib().mxfp4_plan_gemm(M, N, K, split_k, num_sms, ctypes.byref(plan)), "mxfp4_plan_gemm")
    return plan


def mxfp4_gemm_workspace_size(M, N, K, split_k=0) -> int:
    return lib().mxfp4_gemm_workspace_size(M, N, K, split_k)


def mxfp4_gemm_prepacked_workspace_size(M, N, K, split_k=0) -> int:
    return lib().mxfp4_gemm_prepacked_workspace_size(M, N, K, split_k)


def mxfp4_scale_relayout_size(rows, K) -> int:
    return lib().mxfp4_scale_relayout_size(rows, K)


def mxfp4_gemm_host_arena_size(M, N, K, split_k=0, with_c=False) -> int:
    return lib().mxfp4_gemm_host_arena_size(M, N, K, split_k, int(bool(with_c)))


def mxfp4_scale_relayout(dst, src, rows, K, ld_src, stream=None):
    return _check(lib().mxfp4_scale_relayout(_p(dst), _p(src), rows, K, ld_src, _stream(stream)),
                  "mxfp4_scale_relayout")


def mxfp4_scale_relayout2(dst_a, src_a, rows_a, ld_a, dst_b, src_b, rows_b, ld_b, K, stream=None):
    return _check(lib().mxfp4_scale_relayout2(_p(dst_a), _p(src_a), rows_a, ld_a, _p(dst_b),
                                              _p(src_b), rows_b, ld_b, K, _stream(stream)),
                  "mxfp4_scale_relayout2")


def mxfp4_quantize(Q, ldq, S, lds, X, ldx, rows, K, stream=None):
    return _check(lib().mxfp4_quantize(_p(Q), ldq, _p(S), lds, _p(X), ldx, rows, K,
                                       _stream(stream)), "mxfp4_quantize")


def mxfp4_gemm(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha, beta,
               M, N, K, split_k, workspace, workspace_bytes, stream=None):
    return _check(lib().mxfp4_gemm(_p(D), ldd, _p(C), ldc, _p(A), lda, _p(B), ldb, _p(scaleA),
                                   ld_sa, _p(scaleB), ld_sb, alpha, beta, M, N, K, split_k,
                                   _p(workspace), workspace_bytes, _stream(stream)), "mxfp4_gemm")


def mxfp4_gemm_ex(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha, beta,
                  M, N, K, split_k, flags, workspace, workspace_bytes, stream=None):
    """mxfp4_gemm with flags (MXFP4_FLAG_B_STATIC: the work before this call
    on the stream does not write B or scaleB, so B may be loaded early)."""
    return _check(lib().mxfp4_gemm_ex(_p(D), ldd, _p(C), ldc, _p(A), lda, _p(B), ldb, _p(scaleA),
                                      ld_sa, _p(scaleB), ld_sb, alpha, beta, M, N, K, split_k,
                                      flags, _p(workspace), workspace_bytes, _stream(stream)),
                  "mxfp4_gemm_ex")


def mxfp8_gemm(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, fmt_a, fmt_b,
               alpha, beta, M, N, K, split_k, workspace, workspace_bytes, stream=None):
    """MXFP8 / MXFP6 GEMM (A, B: one byte per element, lda / ldb in elements)."""
    return _check(lib().mxfp8_gemm(_p(D), ldd, _p(C), ldc, _p(A), lda, _p(B), ldb, _p(scaleA),
                                   ld_sa, _p(scaleB), ld_sb, fmt_a, fmt_b, alpha, beta, M, N, K,
                                   split_k, _p(workspace), workspace_bytes, _stream(stream)),
                  "mxfp8_gemm")


def mxfp8_gemm_prepacked(D, ldd, C, ldc, A, lda, B, ldb, scaleA_relaid, scaleB_relaid, fmt_a,
                         fmt_b, alpha, beta, M, N, K, split_k, workspace, workspace_bytes,
                         stream=None):
    """MXFP8 GEMM on scales relaid by mxfp4_scale_relayout (with this K)."""
    return _check(lib().mxfp8_gemm_prepacked(_p(D), ldd, _p(C), ldc, _p(A), lda, _p(B), ldb,
                                             _p(scaleA_relaid), _p(scaleB_relaid), fmt_a, fmt_b,
                                             alpha, beta, M, N, K, split_k, _p(workspace),
                                             workspace_bytes, _stream(stream)),
                  "mxfp8_gemm_prepacked")


def nvfp4_gemm(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha, beta, M, N,
               K, workspace, workspace_bytes, stream=None):
    """NVFP4 GEMM: packed E2M1 A, B; one UE4M3 scale per 16 K (ld_sa, ld_sb >= K/16)."""
    return _check(lib().nvfp4_gemm(_p(D), ldd, _p(C), ldc, _p(A), lda, _p(B), ldb, _p(scaleA),
                                   ld_sa, _p(scaleB), ld_sb, alpha, beta, M, N, K,
                                   _p(workspace), workspace_bytes, _stream(stream)),
                  "nvfp4_gemm")


def nvfp4_gemm_workspace_size(M, N, K) -> int:
    return lib().nvfp4_gemm_workspace_size(M, N, K)


def mxfp8_quantize(Q, ldq, S, lds, X, ldx, rows, K, fmt, stream=None):
    """bf16 rows -> E4M3 / E5M2 codes (one per byte) + E8M0 scales."""
    return _check(lib().mxfp8_quantize(_p(Q), ldq, _p(S), lds, _p(X), ldx, rows, K, fmt,
                                       _stream(stream)), "mxfp8_quantize")


def mxfp8_gemm_prepacked_workspace_size(M, N, K, split_k=0) -> int:
    return lib().mxfp8_gemm_prepacked_workspace_size(M, N, K, split_k)


def mxfp8_plan_gemm(M, N, K, split_k=0, num_sms=0) -> Plan:
    plan = Plan()
    _check(lib().mxfp8_plan_gemm(M, N, K, split_k, num_sms, ctypes.byref(plan)), "mxfp8_plan_gemm")
    return plan


def mxfp8_gemm_workspace_size(M, N, K, split_k=0) -> int:
    return lib().mxfp8_gemm_workspace_size(M, N, K, split_k)


def mxfp4_gemm_noalloc(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha,
                       beta, M, N, K, split_k, stream=None):
    """mxfp4_gemm without a workspace argument, for callers that cannot
    allocate device memory: scratch comes from a fixed array in the library's
    device image (MXFP4_NOALLOC_SCRATCH_BYTES).  Calls that overlap on the GPU
    share that array and must be serialised by the caller."""
    return _check(lib().mxfp4_gemm_noalloc(_p(D), ldd, _p(C), ldc, _p(A), lda, _p(B), ldb,
                                           _p(scaleA), ld_sa, _p(scaleB), ld_sb, alpha, beta,
                                           M, N, K, split_k, _stream(stream)),
                  "mxfp4_gemm_noalloc")


def mxfp4_gemm_prepacked(D, ldd, C, ldc, A, lda, B, ldb, scaleA_relaid, scaleB_relaid, alpha,
                         beta, M, N, K, split_k, workspace, workspace_bytes, stream=None):
    return _check(lib().mxfp4_gemm_prepacked(_p(D), ldd, _p(C), ldc, _p(A), lda, _p(B), ldb,
                                             _p(scaleA_relaid), _p(scaleB_relaid), alpha, beta,
                                             M, N, K, split_k, _p(workspace), workspace_bytes,
                                             _stream(stream)), "mxfp4_gemm_prepacked")


def mxfp8_gemm_host(D_host, C_host, A_host, B_host, scaleA_host, scaleB_host, fmt_a, fmt_b,
                    alpha, beta, M, N, K, split_k, device_arena, arena_bytes, stream=None):
    """mxfp4_gemm_host for the byte forms of mxfp8_gemm (host arrays in and out)."""
    return _check(lib().mxfp8_gemm_host(_p(D_host), _p(C_host), _p(A_host), _p(B_host),
                                        _p(scaleA_host), _p(scaleB_host), fmt_a, fmt_b, alpha,
                                        beta, M, N, K, split_k, _p(device_arena), arena_bytes,
                                        _stream(stream)), "mxfp8_gemm_host")


def mxfp8_gemm_host_arena_size(M, N, K, split_k=0, with_c=False) -> int:
    return lib().mxfp8_gemm_host_arena_size(M, N, K, split_k, int(bool(with_c)))


def mxfp4_gemm_host(D_host, C_host, A_host, B_host, scaleA_host, scaleB_host, alpha, beta,
                    M, N, K, split_k, device_arena, arena_bytes, stream=None):
    return _check(lib().mxfp4_gemm_host(_p(D_host), _p(C_host), _p(A_host), _p(B_host),
                                        _p(scaleA_host), _p(scaleB_host), alpha, beta, M, N, K,
                                        split_k, _p(device_arena), arena_bytes, _stream(stream)),
                  "mxfp4_gemm_host")


def mxfp4_device_status(reset=False) -> int:
    st = ctypes.c_int(0)
    _check(lib().mxfp4_device_status(ctypes.byref(st), int(bool(reset))), "mxfp4_device_status")
    return st.value


def mxfp4_wait_timeout_probe(limit_cycles, stream=None):
    return _check(lib().mxfp4_wait_timeout_probe(limit_cycles, _stream(stream)),
                  "mxfp4_wait_timeout_probe")


def mxfp4_set_wait_limit(cycles):
    lib().mxfp4_set_wait_limit(cycles)


def mxfp4_strerror(status) -> str:
    return lib().mxfp4_strerror(status).decode()


def mxfp4_version() -> int:
    return lib().mxfp4_version()


def gemm(A, B, SA, SB, alpha=1.0, beta=0.0, C=None, split_k=0, out=None, workspace=None,
         stream=None):
    """D = alpha * A . B^T + beta * C on device tensors.

    A [M, K/2], B [N, K/2] uint8 (packed E2M1), SA [M, K/32], SB [N, K/32]
    uint8 (E8M0), C [M, N] bfloat16 or None.  Returns D [M, N] bfloat16.
    """
    import torch
    M, N, K = A.shape[0], B.shape[0], A.shape[1] * 2
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    need = mxfp4_gemm_workspace_size(M, N, K, split_k)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=A.device)
    mxfp4_gemm(out, out.stride(0), C, 0 if C is None else C.stride(0), A, A.stride(0) * 2,
               B, B.stride(0) * 2, SA, SA.stride(0), SB, SB.stride(0), float(alpha),
               float(beta), M, N, K, split_k, workspace, workspace.numel(), stream)
    return out
