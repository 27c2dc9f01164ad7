"""The five workloads at full size, in the launch configuration bench.py times
(algo auto) and with the per-iteration algorithm, checked against the oracle
on sampled hidden units (units are independent, so the oracle computes those
columns exactly at full T).  The preactivation buffer is drawn directly on the
GPU; the host regenerates the sampled columns bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 5e-2}


@pytest.mark.parametrize("algo", ["auto", "per_iter"])
@pytest.mark.parametrize("wl", range(5))
def test_workload_full_size_sampled_units(wl, algo):
    import nonlinear_rnn_gb300 as nr
    w = syn.WORKLOADS[wl]
    P = syn.preact_uniform_torch(w, device="cuda")
    inp = syn.make_inputs(w, with_x=False)
    prm = inp["params"]
    cu = inp["cu_seqlens"]
    H, rho = nr.newton_forward(P, prm, cu_seqlens=cu, K=w.K, algo=algo, check=False)
    units = np.unique(np.concatenate([[0, w.d_h - 1], np.linspace(1, w.d_h - 2, 6).astype(int)]))
    rows = np.arange(w.B)
    Pc = syn.preact_uniform_columns(w, units, rows)
    # the device buffer holds exactly these values
    assert torch.equal(P[:, :, torch.as_tensor(units, device="cuda")].float().cpu(),
                       torch.from_numpy(Pc[:, :, :len(units)]))
    Href, rho_ref = oracle.newton(Pc, oracle.pack_params(prm)[:, units], w.K, cu_seqlens=cu,
                                  threads=8)
    Hg = H[:, :, torch.as_tensor(units, device="cuda")].double().cpu().numpy()
    err = float(np.max(np.abs(Hg - Href)))
    assert err <= TOL[w.dtype], err
    # the GPU residual covers every unit, the oracle's only the sample
    assert rho.item() >= rho_ref - TOL[w.dtype]
    assert np.isfinite(rho.item())


@pytest.mark.parametrize("wl", range(5))
def test_workload_agrees_with_sequential_unroll_at_measured_k_star(wl):
    """Against the float64 sequential unroll (the pages' agreement claim), with
    the Newton depth raised to the measured K* = 4 for this init: within tau
    (1e-4 fp32; 5e-2 bf16) on sampled units of every workload at full size."""
    import nonlinear_rnn_gb300 as nr
    w = syn.WORKLOADS[wl]
    K = 4
    P = syn.preact_uniform_torch(w, device="cuda")
    inp = syn.make_inputs(w, with_x=False)
    cu = inp["cu_seqlens"]
    H, _ = nr.newton_forward(P, inp["params"], cu_seqlens=cu, K=K, check=False)
    units = np.array([0, w.d_h // 2, w.d_h - 1])
    Pc = syn.preact_uniform_columns(w, units)
    Hs = oracle.sequential(Pc, oracle.pack_params(inp["params"])[:, units], cu_seqlens=cu,
                           threads=3)
    Hg = H[:, :, torch.as_tensor(units, device="cuda")].double().cpu().numpy()
    assert float(np.max(np.abs(Hg - Hs))) <= TOL[w.dtype]
