"""Critical Newton depth K*(T): the smallest fixed K whose Newton result agrees
with the sequential unroll within tau (FAQs "What is critical Newton depth
(K*)?"; numerics contract "Four echelons / 2. Lab campaign").

Both trajectories come from this library's CUDA kernels on the same batch,
as verify_agreement does.  Run as a module for a sweep over T on synthetic
diag-GRU inputs:

    python -m nonlinear_rnn_gb300.kstar [--d-h 64] [--batch 4] [--kmax 6] [--picard 0]
"""
from __future__ import annotations

import argparse
import json

import torch

from ._binding import (default_agreement_atol, input_projection, newton_forward, params_tensor,
                       sequential_forward)


def agreement_sweep(preact, params, K_values=range(0, 7), cu_seqlens=None, picard_iters=0,
                    algo="auto"):
    """[(K, max_abs(H_newton(K) - H_sequential), residual)] for each K."""
    Hs = sequential_forward(preact, params, cu_seqlens=cu_seqlens).float()
    out = []
    for K in K_values:
        H, rho = newton_forward(preact, params, cu_seqlens=cu_seqlens, K=int(K), algo=algo,
                                check=False, picard_iters=picard_iters)
        err = float((H.float() - Hs).abs().max().item()) if H.numel() else 0.0
        out.append((int(K), err, float(rho.item())))
    return out


def k_star(rows, atol):
    """Smallest K of a sweep with max-abs <= atol (None if none)."""
    for K, err, _ in rows:
        if err <= atol:
            return K
    return None


def main(argv=None):
    import synthetic as syn   # seeded synthetic inputs (shapes and draws only)

    ap = argparse.ArgumentParser()
    ap.add_argument("--d-h", type=int, default=64)
    ap.add_argument("--d-in", type=int, default=64)
    ap.add_argument("--batch", type=int, default=4)
    ap.add_argument("--kmax", type=int, default=6)
    ap.add_argument("--picard", type=int, default=0)
    ap.add_argument("--T", type=int, nargs="*",
                    default=[64, 256, 1024, 4096, 16384, 65536, 131072])
    args = ap.parse_args(argv)
    for T in args.T:
        w = syn.Workload(f"kstar T{T}", args.batch, T, args.d_in, args.d_h, args.kmax, "f32",
                         seed=100 + T % 97)
        inp = syn.make_inputs(w)
        x = torch.from_numpy(inp["x"]).cuda()
        P = input_projection(x, torch.from_numpy(inp["W_x"]).cuda())
        prm = params_tensor(inp["params"], w.d_h, "cuda")
        rows = agreement_sweep(P, prm, range(0, args.kmax + 1), picard_iters=args.picard)
        tau = default_agreement_atol(torch.float32)
        print(json.dumps({"T": T, "B": w.B, "d_h": w.d_h, "picard_iters": args.picard,
                          "tau": tau, "K_star": k_star(rows, tau),
                          "max_abs": {K: e for K, e, _ in rows},
                          "residual": {K: r for K, _, r in rows}}), flush=True)


if __name__ == "__main__":
    main()
