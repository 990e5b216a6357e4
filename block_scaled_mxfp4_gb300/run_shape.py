"""Run the GEMM on one seeded random shape (for profilers).

    python -m block_scaled_mxfp4_gb300.run_shape M N K [--calls C] [--seed S]
                                                 [--format mxfp4|e4m3|e5m2|e2m3|e3m2|e2m1]

mxfp4 (default): random fp4x2 codes for A [M, K/2] and B [N, K/2] and E8M0
scales in [120, 127] on the current CUDA device; the scales are relaid once
with mxfp4_scale_relayout, then C calls of mxfp4_gemm_prepacked follow.
e4m3 / e5m2: random 8-bit codes (the format's NaN codes avoided) for A
[M, K] and B [N, K]; e2m3 / e3m2 / e2m1: random bytes (every byte is a valid
padded 6- or 4-bit group: the codes cover all values and the padding is not
read); then C calls of mxfp8_gemm with row-major scales (each call relays
them itself when its plan asks for it).  alpha 1, beta 0, the
heuristic's plan, a synchronise after the last call.  Nothing is checked:
this only gives a profiler a short program with a known number of GEMM
launches.
"""
import argparse

import torch

from . import (MXFP4_E2M1_PADDED, MXFP6_E2M3, MXFP6_E3M2, MXFP8_E4M3, MXFP8_E5M2,
               mxfp4_gemm_prepacked, mxfp4_gemm_prepacked_workspace_size,
               mxfp4_plan_gemm, mxfp4_scale_relayout, mxfp4_scale_relayout_size, mxfp8_gemm,
               mxfp8_gemm_workspace_size, mxfp8_plan_gemm)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("M", type=int)
    ap.add_argument("N", type=int)
    ap.add_argument("K", type=int)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--format", choices=["mxfp4", "e4m3", "e5m2", "e2m3", "e3m2", "e2m1"],
                    default="mxfp4")
    args = ap.parse_args(argv)
    M, N, K = args.M, args.N, args.K
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(args.seed)
    if args.format != "mxfp4":
        fmt = {"e4m3": MXFP8_E4M3, "e5m2": MXFP8_E5M2, "e2m3": MXFP6_E2M3, "e3m2": MXFP6_E3M2,
               "e2m1": MXFP4_E2M1_PADDED}[args.format]
        # 8-bit: codes with exponent fields below the top (no NaN or infinity
        # codes); the padded 6- and 4-bit forms have no special codes at all.
        top = 0x70 if args.format in ("e4m3", "e5m2") else 256
        A = torch.randint(0, top, (M, K), dtype=torch.uint8, device=dev, generator=g)
        B = torch.randint(0, top, (N, K), dtype=torch.uint8, device=dev, generator=g)
        SA = torch.randint(120, 128, (M, K // 32), dtype=torch.uint8, device=dev, generator=g)
        SB = torch.randint(120, 128, (N, K // 32), dtype=torch.uint8, device=dev, generator=g)
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsb = mxfp8_gemm_workspace_size(M, N, K, 0)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        plan = mxfp8_plan_gemm(M, N, K, 0, 0)
        for _ in range(args.calls):
            mxfp8_gemm(D, N, None, N, A, K, B, K, SA, K // 32, SB, K // 32, fmt, fmt, 1.0, 0.0,
                       M, N, K, 0, ws if wsb else None, wsb)
        torch.cuda.synchronize()
        print(f"{M}x{N}x{K} {args.format}: {args.calls} calls, plan {plan.as_dict()}")
        return
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
