"""Backward (adjoint) pass on the GPU against the oracle's adjoint (itself
pinned by finite differences of the unroll)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dtype)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


CASES = [dict(B=3, T=300, d_h=40, lens=None), dict(B=1, T=None, d_h=24, lens=[130, 1, 0, 300, 77, 256]),
         dict(B=2, T=1000, d_h=64, lens=None)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_backward_matches_oracle(dtype, case):
    import nonlinear_rnn_gb300 as nr
    cfg = CASES[case]
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    cu = syn.cu_from_lengths(cfg["lens"]) if cfg["lens"] else None
    T = int(cu[-1]) if cu is not None else cfg["T"]
    w = syn.small_workload(B=cfg["B"], T=T, d_h=cfg["d_h"], dtype=dtype, seed=80 + case)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    H = oracle.sequential(P, prm, cu_seqlens=cu).astype(np.float32)
    gH = np.random.default_rng(81 + case).normal(size=H.shape).astype(np.float32)
    if dtype == "bf16":
        H, gH = syn.round_bf16(H), syn.round_bf16(gH)
    gP_ref, gprm_ref = oracle.backward(P, prm, H, gH, cu_seqlens=cu)
    gP, gprm = nr.newton_backward(dev(P, tdt), prm, dev(H, tdt), dev(gH, tdt), cu_seqlens=cu)
    scale = max(1.0, float(np.max(np.abs(gP_ref))))
    tol = 2e-5 if dtype == "f32" else 2e-2          # bf16: gP stored in bf16
    assert np.max(np.abs(host(gP) - gP_ref)) <= tol * scale
    # parameter gradients: sums over B*T terms
    rel = np.max(np.abs(gprm.cpu().numpy() - gprm_ref)) / max(1.0, float(np.max(np.abs(gprm_ref))))
    assert rel <= (1e-4 if dtype == "f32" else 1e-2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,d_h", [(1, 1 << 20, 8), (1, 128, 8192)])
def test_backward_extreme_shapes(dtype, B, T, d_h):
    """One reverse look-back chain of 16384 chunks (T = 2^20, 8 units: every
    resident CTA in one column), and 256 unit tiles of two chunks each
    (d_h = 8192), against the oracle's adjoint."""
    import nonlinear_rnn_gb300 as nr
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w = syn.small_workload(B=B, T=T, d_h=d_h, dtype=dtype, seed=90 + d_h)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Pd = dev(P, tdt)
    Pq = host(Pd)
    H = oracle.sequential(Pq, prm).astype(np.float32)
    gH = np.random.default_rng(91 + d_h).normal(size=H.shape).astype(np.float32)
    Hd, gHd = dev(H, tdt), dev(gH, tdt)
    gP_ref, gprm_ref = oracle.backward(Pq, prm, host(Hd), host(gHd))
    gP, gprm = nr.newton_backward(Pd, prm, Hd, gHd)
    scale = max(1.0, float(np.max(np.abs(gP_ref))))
    tol = 2e-5 if dtype == "f32" else 2e-2
    assert np.max(np.abs(host(gP) - gP_ref)) <= tol * scale
    rel = np.max(np.abs(gprm.cpu().numpy() - gprm_ref)) / max(1.0, float(np.max(np.abs(gprm_ref))))
    assert rel <= (1e-4 if dtype == "f32" else 1e-2)
