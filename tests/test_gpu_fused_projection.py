"""Newton forward with the input projection fused into the Newton kernel
(bf16): against the oracle run on the float64 projection rounded to bf16,
and against the unfused pipeline (projection kernel + Newton kernel)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu

CASES = [dict(B=2, T=300, d_in=136, d_h=40, lens=None),      # ragged T, d_h, d_in tails
         dict(B=1, T=None, d_in=64, d_h=32, lens=[130, 1, 0, 300, 77]),
         dict(B=3, T=1000, d_in=512, d_h=96, lens=None),
         dict(B=1, T=64, d_in=8, d_h=8, lens=None),          # one 32-wide slice, mostly zero-filled
         dict(B=2, T=129, d_in=40, d_h=72, lens=None),       # a 32-wide slice and a tail of 8
         dict(B=1, T=200, d_in=1024, d_h=32, lens=None)]     # 32 slices through the 2-stage ring


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_projection_newton_matches_oracle(case):
    import nonlinear_rnn_gb300 as nr
    cfg = CASES[case]
    cu = syn.cu_from_lengths(cfg["lens"]) if cfg["lens"] else None
    T = int(cu[-1]) if cu is not None else cfg["T"]
    w = syn.small_workload(B=cfg["B"], T=T, d_in=cfg["d_in"], d_h=cfg["d_h"], dtype="bf16",
                           seed=95 + case)
    inp = syn.make_inputs(w)
    x, W, prm = inp["x"], inp["W_x"], inp["params"]
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    Wd = torch.from_numpy(W).cuda().to(torch.bfloat16)
    H, rho = nr.newton_forward_x(xd, Wd, prm, cu_seqlens=cu, K=3, check=False)
    # oracle on the float64 projection rounded to bf16 (a 1-ulp difference in
    # a rounded preactivation moves H by far less than the bf16 band)
    P = syn.round_bf16(oracle.input_projection(x, W).astype(np.float32))
    Href, rho_ref = oracle.newton(P, prm, 3, cu_seqlens=cu)
    assert np.max(np.abs(H.float().cpu().numpy() - Href)) <= 5e-2
    # same as the two-kernel pipeline up to the projection's accumulation order
    Pd = nr.input_projection(xd, Wd)
    H2, rho2 = nr.newton_forward(Pd, prm, cu_seqlens=cu, K=3, algo="fused", check=False)
    assert (H.float() - H2.float()).abs().max().item() <= 2e-2
    assert abs(rho.item() - rho2.item()) <= 2e-2


def test_fused_projection_rejects_fp32():
    import nonlinear_rnn_gb300 as nr
    x = torch.zeros((1, 8, 8), device="cuda")
    W = torch.zeros((24, 8), device="cuda")
    with pytest.raises(TypeError):
        nr.newton_forward_x(x, W, np.zeros((6, 8), np.float32), K=1)
