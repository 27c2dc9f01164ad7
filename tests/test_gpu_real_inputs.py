"""The five workloads at full size on the inputs their configurations define:
x ~ N(0, 1), W_x ~ U(+-1/sqrt(d_in)), P = x W_x^T on the tensor cores
(nrnn_input_projection), then the Newton forward at the configuration's K in
the launch configuration bench.py times.

Two checks per workload, both against the float64 oracle on inputs it builds
itself from the same seeded x and W_x (nothing the CUDA path computed feeds
the oracle):
  * the projection on at least 4096 sampled rows of P (all 3 d_h columns)
    against a float64 matmul, in the projection's band relative to
    sum_k |x_k| |W_k| (shapes_layout, "W_x ... caller strides");
  * H on sampled hidden units against oracle Newton at the same K, whose
    preactivations are the float64 projection of those units' W_x rows
    rounded to the storage type (FAQs, "Does parallel Newton match
    sequential unroll?": tau = 1e-4 fp32, 5e-2 bf16 storage).
The projection's own rounding differences reach H through the recurrence,
which contracts them: they stay far inside tau."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 5e-2}
# f32: split-TF32 products (error of order 2^-21 of sum |x||W|) with fp32 sums;
# bf16: exact products, fp32 sums, one rounding of the output to bf16
PROJ_BAND = {"f32": 1e-5, "bf16": 8e-3}


def _storage(a, dtype):
    a = np.asarray(a, dtype=np.float32)
    return syn.round_bf16(a) if dtype == "bf16" else a


def _sample_units(d_h):
    return np.unique(np.concatenate([[0, d_h - 1], np.linspace(1, d_h - 2, 6).astype(int)]))


@pytest.mark.parametrize("wl", range(5))
def test_workload_real_inputs_full_size(wl):
    import nonlinear_rnn_gb300 as nr
    w = syn.WORKLOADS[wl]
    inp = syn.make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x = torch.from_numpy(inp["x"]).cuda().to(tdt)
    W = torch.from_numpy(inp["W_x"]).cuda().to(tdt)
    P = nr.input_projection(x, W)
    assert P.shape == (w.B, w.T, 3 * w.d_h)

    # the projection on sampled rows, every column
    n_rows = w.B * w.T
    rng = np.random.default_rng(1000 + wl)
    ridx = np.unique(np.concatenate([[0, n_rows - 1],
                                     rng.choice(n_rows, min(n_rows, 4096), replace=False)]))
    assert len(ridx) >= min(n_rows, 4096)
    xs = inp["x"].reshape(-1, w.d_in)[ridx]
    ref = oracle.input_projection(xs, inp["W_x"])
    Pg = P.reshape(-1, 3 * w.d_h)[torch.as_tensor(ridx, device="cuda")].double().cpu().numpy()
    scale = np.abs(xs).astype(np.float64) @ np.abs(inp["W_x"]).astype(np.float64).T
    rel = float(np.max(np.abs(Pg - ref) / (scale + 1e-30)))
    assert rel <= PROJ_BAND[w.dtype], rel

    # the Newton forward at the configuration's K on sampled units
    cu = inp["cu_seqlens"]
    H, rho = nr.newton_forward(P, inp["params"], cu_seqlens=cu, K=w.K, check=False)
    units = _sample_units(w.d_h)
    cols = np.concatenate([units, w.d_h + units, 2 * w.d_h + units])
    Pc = _storage(oracle.input_projection(inp["x"], inp["W_x"][cols]), w.dtype)
    Href, rho_ref = oracle.newton(Pc, oracle.pack_params(inp["params"])[:, units], w.K,
                                  cu_seqlens=cu, threads=8)
    Hg = H[:, :, torch.as_tensor(units, device="cuda")].double().cpu().numpy()
    err = float(np.max(np.abs(Hg - Href)))
    assert err <= TOL[w.dtype], err
    # the GPU residual covers every unit, the oracle's only the sample
    assert np.isfinite(rho.item()) and rho.item() >= rho_ref - TOL[w.dtype]


def _small(dtype, seed, T=700, d_h=48):
    w = syn.small_workload(B=2, T=T, d_h=d_h, dtype=dtype, seed=seed)
    return w, syn.direct_preact(w), syn.make_params(w)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 6])
def test_verify_agreement_reports_the_oracles_max_abs(dtype, K):
    """verify_agreement (numerics contract, "Four echelons / 3. Opt-in oracle")
    runs Newton and the sequential unroll on the GPU and reports their max-abs
    difference; it must equal the float64 oracle's |Newton_K - unroll| up to
    the two GPU paths' own errors, and `ok` must follow the band."""
    import nonlinear_rnn_gb300 as nr
    w, P, prm = _small(dtype, seed=400 + K)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rep = nr.verify_agreement(torch.from_numpy(P).cuda().to(tdt), prm, K=K)
    Hn, _ = oracle.newton(P, prm, K)
    Hs = oracle.sequential(P, prm)
    want = float(np.max(np.abs(Hn - Hs)))
    # implementation error of each GPU path: fp32 a few 1e-6; bf16 storage
    # rounds H to bf16 (half a step is 2^-9 of |h| < 1)
    slack = 4e-5 if dtype == "f32" else 1.5e-2
    assert abs(rep.max_abs - want) <= slack, (rep.max_abs, want)
    assert rep.atol == (1e-4 if dtype == "f32" else 5e-2)
    assert rep.ok == (rep.max_abs <= rep.atol)
    assert rep.K == K and np.isfinite(rep.residual)
    d = rep.to_dict()
    assert d["max_abs"] == rep.max_abs and d["ok"] == rep.ok


def test_verify_agreement_raise_on_fail():
    import nonlinear_rnn_gb300 as nr
    w, P, prm = _small("f32", seed=431)
    Pd = torch.from_numpy(P).cuda()
    # one iteration from H = 0 is far from the unroll on this input
    Hn, _ = oracle.newton(P, prm, 1)
    assert np.max(np.abs(Hn - oracle.sequential(P, prm))) > 1e-2
    with pytest.raises(nr.AgreementError):
        nr.verify_agreement(Pd, prm, K=1, raise_on_fail=True)
    # K = T reproduces the unroll exactly (iteration k fixes step k); K is at
    # most 64, so on a 64-step sequence
    w64, P64, prm64 = _small("f32", seed=432, T=64)
    rep = nr.verify_agreement(torch.from_numpy(P64).cuda(), prm64, K=w64.T, raise_on_fail=True)
    assert rep.ok and rep.max_abs <= 2e-5
    # a caller's band replaces the default
    rep = nr.verify_agreement(Pd, prm, K=1, atol=10.0, raise_on_fail=True)
    assert rep.ok and rep.atol == 10.0
