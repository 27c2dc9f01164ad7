"""Picard warm start, Newton from a given iterate and the K* sweep, on the GPU
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nr():
    import nonlinear_rnn_gb300 as m
    return m


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dtype)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("sweeps", [0, 1, 2, 5])
@pytest.mark.parametrize("ragged", [False, True])
def test_picard_matches_oracle(nr, dtype, sweeps, ragged):
    # d_h = 24 and 40: a thread's units (2 fp32 or 4 bf16) end the tile part way
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    if ragged:
        cu = syn.cu_from_lengths([100, 1, 0, 200, 129])
        w = syn.small_workload(B=1, T=int(cu[-1]), d_h=24, seed=41)
    else:
        cu = None
        w = syn.small_workload(B=2, T=300, d_h=40, seed=42)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Pd = dev(P, tdt)
    G = nr.picard(Pd, prm, sweeps, cu_seqlens=cu)
    # the oracle on the stored preactivations; bf16 stores each sweep's G
    # rounded (a few bf16 units in the last place after five sweeps)
    ref = oracle.picard(host(Pd), prm, sweeps, cu_seqlens=cu)
    assert np.max(np.abs(host(G) - ref)) <= (1e-6 if dtype == "f32" else 2e-2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ["fused", "per_iter"])
@pytest.mark.parametrize("K", [0, 1, 3])
def test_newton_from_initial_iterate_matches_oracle(nr, dtype, algo, K):
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w = syn.small_workload(B=2, T=400, d_h=40, dtype=dtype, seed=43 + K)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    H0 = oracle.picard(P, prm, 3).astype(np.float32)
    if dtype == "bf16":
        H0 = syn.round_bf16(H0)
    Href, rho_ref = oracle.newton_init(P, prm, K, H0)
    H, rho = nr.newton_forward(dev(P, tdt), prm, K=K, algo=algo, check=False,
                               H_init=dev(H0, tdt))
    tol = 2e-5 if dtype == "f32" else 5e-2
    assert np.max(np.abs(host(H) - Href)) <= tol
    assert abs(rho.item() - rho_ref) <= tol


def test_picard_warm_start_then_newton(nr):
    lens = [300, 5, 0, 500]
    cu = syn.cu_from_lengths(lens)
    w = syn.small_workload(B=1, T=int(cu[-1]), d_h=16, seed=44)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    G = nr.picard(dev(P), prm, 2, cu_seqlens=cu)
    Href, _ = oracle.newton_init(P, prm, 2, host(G), cu_seqlens=cu)
    H, _ = nr.newton_forward(dev(P), prm, cu_seqlens=cu, K=2, picard_iters=2, check=False)
    assert np.max(np.abs(host(H) - Href)) <= 2e-5


def test_initial_iterate_must_not_alias_output(nr):
    w = syn.small_workload(B=1, T=200, d_h=8, seed=45)
    P = dev(syn.direct_preact(w))
    H = torch.zeros((1, 200, 8), device="cuda")
    with pytest.raises(ValueError):
        nr.newton_forward(P, syn.make_params(w), K=2, H_init=H, out=H)


def test_kstar_sweep_matches_oracle(nr):
    from nonlinear_rnn_gb300 import kstar
    w = syn.small_workload(B=2, T=600, d_h=16, seed=46)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    rows = kstar.agreement_sweep(dev(P), prm, range(0, 6))
    Hs = oracle.sequential(P, prm)
    for K, err, rho in rows:
        Hn, rho_ref = oracle.newton(P, prm, K)
        assert abs(err - np.max(np.abs(Hn - Hs))) <= 2e-5
        assert abs(rho - rho_ref) <= 2e-5
    ks = kstar.k_star(rows, 1e-4)
    assert ks is not None and rows[ks][1] <= 1e-4 and (ks == 0 or rows[ks - 1][1] > 1e-4)
