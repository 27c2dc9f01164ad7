"""Seeded random shapes through every Newton form against the float64 oracle:
batch rows or packs (with and without room for segment-aligned chunks),
ragged unit tiles and time chunks, fused and per-iteration, f32 and bf16,
K from 1 to 5.  Sizes stay small enough for the oracle to finish in
seconds."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}
N_CASES = 24


def _case(i):
    rng = np.random.default_rng(5000 + i)
    dtype = ("f32", "bf16")[i % 2]
    algo = ("fused", "per_iter")[(i // 2) % 2]
    K = int(rng.integers(1, 6))
    d_h = int(8 * rng.integers(1, 26))                       # 8 .. 200
    if i % 3 == 0:                                           # a pack
        S = int(rng.integers(2, 7))
        lens = rng.integers(0, 900, size=S)
        lens[rng.integers(0, S)] = int(rng.integers(1, 3))   # a very short segment
        B, T = 1, int(lens.sum())
        if T == 0:
            lens[0], T = 1, 1
        cu = syn.cu_from_lengths(lens)
    else:
        B, T, cu = int(rng.integers(1, 5)), int(rng.integers(1, 2200)), None
    return dict(dtype=dtype, algo=algo, K=K, d_h=d_h, B=B, T=T, cu=cu, seed=6000 + i)


@pytest.fixture(scope="module")
def nr():
    import nonlinear_rnn_gb300 as m
    return m


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_oracle(nr, i):
    c = _case(i)
    w = syn.small_workload(B=c["B"], T=c["T"], d_h=c["d_h"], dtype=c["dtype"], seed=c["seed"])
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    tdt = TDT[c["dtype"]]
    Pd = torch.from_numpy(np.ascontiguousarray(P, dtype=np.float32)).cuda().to(tdt)
    # the values as stored are what both sides read
    Pq = Pd.float().cpu().numpy().astype(np.float64)
    Href, rho_ref = oracle.newton(Pq, prm, c["K"], cu_seqlens=c["cu"])
    S = 0 if c["cu"] is None else len(c["cu"]) - 1
    ws = torch.empty(nr.workspace_bytes(c["B"], c["T"], c["d_h"], tdt, c["K"], c["algo"], num_segments=S),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((c["B"], c["T"], c["d_h"]), float("nan"), dtype=tdt, device="cuda")
    H, rho = nr.newton_forward(Pd, prm, cu_seqlens=c["cu"], K=c["K"], algo=c["algo"], check=False,
                               out=out, workspace=ws)
    assert not torch.isnan(H).any(), c
    err = float(np.max(np.abs(H.float().cpu().numpy() - Href)))
    tol = 2e-5 if c["dtype"] == "f32" else 5e-2
    assert err <= tol, (c, err)
    assert abs(rho.item() - rho_ref) <= tol, (c, rho.item(), rho_ref)


def test_random_packs_with_room_for_segment_aligned_chunks(nr):
    """Long packs of few segments (at most one per 8 chunks) on segment-aligned
    chunks, against the oracle."""
    for i in range(4):
        rng = np.random.default_rng(7000 + i)
        S = int(rng.integers(2, 6))
        lens = rng.integers(64 * 8, 64 * 40, size=S)
        cu = syn.cu_from_lengths(lens)
        N, d_h, K = int(cu[-1]), int(8 * rng.integers(2, 12)), int(rng.integers(1, 4))
        algo = ("fused", "per_iter")[i % 2]
        w = syn.small_workload(B=1, T=N, d_h=d_h, seed=7100 + i)
        P = syn.direct_preact(w)
        prm = syn.make_params(w)
        ws = torch.empty(nr.workspace_bytes(1, N, d_h, torch.float32, K, algo, num_segments=S),
                         dtype=torch.uint8, device="cuda")
        assert ws.numel() > nr.workspace_bytes(1, N, d_h, torch.float32, K, algo)
        H, rho = nr.newton_forward(torch.from_numpy(P).cuda(), prm, cu_seqlens=cu, K=K, algo=algo,
                                   check=False, workspace=ws)
        Href, rho_ref = oracle.newton(P, prm, K, cu_seqlens=cu)
        assert float(np.max(np.abs(H.double().cpu().numpy() - Href))) <= 2e-5
        assert abs(rho.item() - rho_ref) <= 2e-5


@pytest.mark.parametrize("i", range(6))
def test_random_backward_matches_oracle(nr, i):
    """The adjoint scan on random shapes (batch rows, packs with and without
    room for segment-aligned chunks) against the oracle's adjoint."""
    rng = np.random.default_rng(8000 + i)
    dtype = ("f32", "bf16")[i % 2]
    tdt = TDT[dtype]
    d_h = int(8 * rng.integers(1, 16))
    if i >= 2:
        S = int(rng.integers(2, 5))
        lens = rng.integers(1, 64 * (12 if i >= 4 else 3), size=S)
        cu = syn.cu_from_lengths(lens)
        B, T = 1, int(cu[-1])
    else:
        cu, B, T = None, int(rng.integers(1, 4)), int(rng.integers(1, 1500))
    w = syn.small_workload(B=B, T=T, d_h=d_h, dtype=dtype, seed=8100 + i)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Pd = torch.from_numpy(np.ascontiguousarray(P, dtype=np.float32)).cuda().to(tdt)
    Pq = Pd.float().cpu().numpy().astype(np.float64)
    H = oracle.sequential(Pq, prm, cu_seqlens=cu).astype(np.float32)
    gH = rng.normal(size=H.shape).astype(np.float32)
    Hd = torch.from_numpy(H).cuda().to(tdt)
    gHd = torch.from_numpy(gH).cuda().to(tdt)
    Hq = Hd.float().cpu().numpy().astype(np.float64)
    gHq = gHd.float().cpu().numpy().astype(np.float64)
    gP_ref, gprm_ref = oracle.backward(Pq, prm, Hq, gHq, cu_seqlens=cu)
    gP, gprm = nr.newton_backward(Pd, prm, Hd, gHd, cu_seqlens=cu)
    scale = max(1.0, float(np.max(np.abs(gP_ref))))
    tol = 2e-5 if dtype == "f32" else 2e-2
    assert float(np.max(np.abs(gP.float().cpu().numpy() - gP_ref))) <= tol * scale
    rel = np.max(np.abs(gprm.cpu().numpy() - gprm_ref)) / max(1.0, float(np.max(np.abs(gprm_ref))))
    assert rel <= (1e-4 if dtype == "f32" else 1e-2)
