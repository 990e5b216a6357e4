"""Shared helpers of the GPU parity tests: device upload, C-ABI calls and the
element-wise bound against the oracle.

Bound (per output element, as the target states it):
    |D_gpu - D_ref| <= ulp_bf16(D_ref) + 2^-20 * sum_k |a_k b_k|
with ulp_bf16(x) = 2^(max(floor(log2|x|), -126) - 7) and ulp_bf16(0) = 2^-133,
and a_k, b_k the scaled inputs.  The first term is one bf16 rounding of the
output; the second covers fp32 accumulation order inside the tensor cores
and the split-K partial sums.  alpha does not enter it.
"""
import numpy as np

import block_scaled_mxfp4_gb300 as mx


def bf16_bits_to_f64(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, E = np.frexp(a)
    e = np.maximum(E - 1, -126)
    u = np.ldexp(1.0, (e - 7).astype(np.int32))
    return np.where(a == 0, 2.0 ** -133, u)


def error_ratio(d_gpu_bits, d_ref_bits, sabs, alpha=None):
    g = bf16_bits_to_f64(d_gpu_bits)
    r = bf16_bits_to_f64(d_ref_bits)
    bound = ulp_bf16(r) + 2.0 ** -20 * np.asarray(sabs)
    err = np.abs(g - r)
    ratio = err / bound
    ratio[np.isnan(g) | np.isnan(r)] = np.inf
    return ratio


def assert_within_bound(d_gpu_bits, d_ref_bits, sabs, alpha=None, what=""):
    ratio = error_ratio(d_gpu_bits, d_ref_bits, sabs, alpha)
    worst = float(ratio.max()) if ratio.size else 0.0
    if not worst <= 1.0:
        idx = np.argwhere(ratio > 1.0)
        sample = idx[:12].tolist()
        g = bf16_bits_to_f64(d_gpu_bits)
        r = bf16_bits_to_f64(d_ref_bits)
        details = [(tuple(i), float(g[tuple(i)]), float(r[tuple(i)])) for i in sample]
        raise AssertionError(f"{what}: {len(idx)} of {ratio.size} outside the bound, "
                             f"max ratio {worst:.3g}; first (index, gpu, ref): {details}")
    return worst


class Dev:
    """A problem's operands on the GPU."""

    def __init__(self, p, device="cuda"):
        import torch
        self.p = p
        self.A = torch.from_numpy(np.ascontiguousarray(p.A)).to(device)
        self.B = torch.from_numpy(np.ascontiguousarray(p.B)).to(device)
        self.SA = torch.from_numpy(np.ascontiguousarray(p.SA)).to(device)
        self.SB = torch.from_numpy(np.ascontiguousarray(p.SB)).to(device)
        self.C = None
        if p.C is not None:
            self.C = torch.from_numpy(np.ascontiguousarray(p.C).view(np.int16)).to(device) \
                .view(torch.bfloat16)


def d_to_bits(D):
    import torch
    return D.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_gemm(dev, split_k=0, alpha=None, beta=None, out=None):
    """mxfp4_gemm through the C ABI on the current stream; returns D bits."""
    import torch
    p = dev.p
    alpha = p.alpha if alpha is None else alpha
    beta = p.beta if beta is None else beta
    D = out if out is not None else torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16,
                                               device=dev.A.device)
    ws_bytes = mx.mxfp4_gemm_workspace_size(p.M, p.N, p.K, split_k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev.A.device)
    C = dev.C if beta != 0.0 else None
    mx.mxfp4_gemm(D, D.stride(0), C, 0 if C is None else C.stride(0), dev.A, dev.A.stride(0) * 2,
                  dev.B, dev.B.stride(0) * 2, dev.SA, dev.SA.stride(0), dev.SB, dev.SB.stride(0),
                  float(alpha), float(beta), p.M, p.N, p.K, split_k, ws, ws_bytes)
    torch.cuda.synchronize()
    return d_to_bits(D)


def sample_pairs(M, N, count, seed, tile_m=128, tile_n=256):
    """Random (m, n) pairs plus the corners of every tile edge that exists."""
    rng = np.random.default_rng(seed)
    ms = {0, M - 1}
    for t in range(0, M, tile_m):
        ms.update({t, min(M - 1, t + tile_m - 1)})
    ns = {0, N - 1}
    for t in range(0, N, tile_n):
        ns.update({t, min(N - 1, t + 31), min(N - 1, t + tile_n - 1)})
    ms_l, ns_l = sorted(ms), sorted(ns)
    edge = [(m, n) for m in ms_l[:: max(1, len(ms_l) // 16)] for n in ns_l[:: max(1, len(ns_l) // 16)]]
    rnd = np.stack([rng.integers(0, M, count), rng.integers(0, N, count)], axis=1)
    pairs = np.concatenate([np.array(edge, dtype=np.int64).reshape(-1, 2), rnd.astype(np.int64)])
    return np.unique(pairs, axis=0)
