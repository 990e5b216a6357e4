"""Run the prepacked MXFP4 GEMM on one seeded random shape (for profilers).

    python -m block_scaled_mxfp4_gb300.run_shape M N K [--calls C] [--seed S]

Draws random fp4x2 codes for A [M, K/2] and B [N, K/2] and E8M0 scales in
[120, 127] on the current CUDA device, relays the scales out once with
mxfp4_scale_relayout, then makes C calls of mxfp4_gemm_prepacked (alpha 1,
beta 0) with the heuristic's plan, synchronising after the last.  Nothing is
checked: this only gives a profiler a short program with a known number of
GEMM launches.
"""
import argparse

import torch

from . import (mxfp4_gemm_prepacked, mxfp4_gemm_prepacked_workspace_size, mxfp4_plan_gemm,
               mxfp4_scale_relayout, mxfp4_scale_relayout_size)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("M", type=int)
    ap.add_argument("N", type=int)
    ap.add_argument("K", type=int)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)
    M, N, K = args.M, args.N, args.K
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(args.seed)
    A = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev, generator=g)
    B = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=g)
    SA = torch.randint(120, 128, (M, K // 32), dtype=torch.uint8, device=dev, generator=g)
    SB = torch.randint(120, 128, (N, K // 32), dtype=torch.uint8, device=dev, generator=g)
    sfa = torch.empty(mxfp4_scale_relayout_size(M, K), dtype=torch.uint8, device=dev)
    sfb = torch.empty(mxfp4_scale_relayout_size(N, K), dtype=torch.uint8, device=dev)
    mxfp4_scale_relayout(sfa, SA, M, K, K // 32)
    mxfp4_scale_relayout(sfb, SB, N, K, K // 32)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    wsb = mxfp4_gemm_prepacked_workspace_size(M, N, K, 0)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    plan = mxfp4_plan_gemm(M, N, K, 0, 0)
    for _ in range(args.calls):
        mxfp4_gemm_prepacked(D, N, None, N, A, K, B, K, sfa, sfb, 1.0, 0.0, M, N, K, 0,
                             ws if wsb else None, wsb)
    torch.cuda.synchronize()
    print(f"{M}x{N}x{K}: {args.calls} calls, plan {plan.as_dict()}")


if __name__ == "__main__":
    main()
