"""GPU parity of the CUDA path (called through the C ABI via the binding)
against the float64 oracle, element by element on the same seeded inputs.

Bars: fp32 storage max-abs <= 1e-4 (the pages' agreement tau); bf16 storage
(fp32 math) <= 5e-2; head masks bit-exact.  The oracle runs the same
algorithm (K Newton iterations) in float64, so these bars bound the
implementation error; the method error (Newton at K vs the unroll) is
measured separately in test_gpu_workloads.py."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
TOL = {"f32": 1e-4, "bf16": 5e-2}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def nr():
    import nonlinear_rnn_gb300 as m
    return m


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dtype)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def nan_out(B, T, d_h, dtype):
    return torch.full((B, T, d_h), float("nan"), dtype=dtype, device="cuda")


@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_golden_tiny(nr, algo):
    with open(os.path.join(HERE, "golden", "tiny_newton.json")) as fh:
        g = json.load(fh)
    P = np.array(g["P"], dtype=np.float32)
    prm = {k: np.array(v, dtype=np.float32) for k, v in g["params"].items()}
    for K, v in g["newton"].items():
        H, rho = nr.newton_forward(dev(P), prm, K=int(K), algo=algo, check=False)
        np.testing.assert_allclose(host(H), np.array(v["H"]), atol=2e-6)
        assert abs(rho.item() - v["rho"]) < 2e-6
    cu = np.array(g["pack"]["cu_seqlens"], dtype=np.int32)
    H, _ = nr.newton_forward(dev(P[:1]), prm, cu_seqlens=cu, K=3, algo=algo, check=False)
    np.testing.assert_allclose(host(H), np.array(g["pack"]["newton3"]), atol=2e-6)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ["fused", "per_iter"])
@pytest.mark.parametrize("K", [1, 2, 3, 6])
def test_newton_matches_oracle_small(nr, dtype, algo, K):
    # 3 rows x 300 steps (several full time tiles + a ragged tail) x 40 units
    # (one full 32-unit tile + a ragged 8)
    w = syn.small_workload(B=3, T=300, d_h=40, dtype=dtype, seed=20 + K)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Href, rho_ref = oracle.newton(P, prm, K)
    out = nan_out(w.B, w.T, w.d_h, TDT[dtype])
    H, rho = nr.newton_forward(dev(P, TDT[dtype]), prm, K=K, algo=algo, check=False, out=out)
    err = np.max(np.abs(host(H) - Href))
    assert not torch.isnan(H).any()
    assert err <= TOL[dtype], err
    if dtype == "f32":
        assert err <= 2e-5, err          # implementation error well inside tau
        assert abs(rho.item() - rho_ref) <= 2e-5
    else:
        assert abs(rho.item() - rho_ref) <= 5e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_one_column_of_16384_chunks(nr, dtype, algo):
    # B = 1, T = 2^20, d_h = 8: a single look-back chain of 16384 chunks, so that
    # every resident CTA belongs to the same column (the deepest chains the
    # look-back meets), and 24 of each tile's 32 unit lanes idle
    w = syn.small_workload(B=1, T=1 << 20, d_h=8, dtype=dtype, seed=31)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Pd = dev(P, TDT[dtype])
    Href, rho_ref = oracle.newton(host(Pd), prm, 2)
    out = nan_out(w.B, w.T, w.d_h, TDT[dtype])
    H, rho = nr.newton_forward(Pd, prm, K=2, algo=algo, check=False, out=out)
    assert not torch.isnan(H).any()
    err = float(np.max(np.abs(host(H) - Href)))
    assert err <= (2e-5 if dtype == "f32" else 5e-2), err
    assert abs(rho.item() - rho_ref) <= (2e-5 if dtype == "f32" else 5e-2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_256_unit_tiles(nr, dtype, algo):
    # d_h = 8192 (256 unit tiles) over T = 200 (four chunks, the last ragged):
    # many short columns, and a preactivation row of 24576 values
    w = syn.small_workload(B=1, T=200, d_h=8192, dtype=dtype, seed=34)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Pd = dev(P, TDT[dtype])
    Href, rho_ref = oracle.newton(host(Pd), prm, 3)
    out = nan_out(w.B, w.T, w.d_h, TDT[dtype])
    H, rho = nr.newton_forward(Pd, prm, K=3, algo=algo, check=False, out=out)
    assert not torch.isnan(H).any()
    err = float(np.max(np.abs(host(H) - Href)))
    assert err <= (2e-5 if dtype == "f32" else 5e-2), err
    assert abs(rho.item() - rho_ref) <= (2e-5 if dtype == "f32" else 5e-2)


@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_forwards_on_two_streams_at_once(nr, algo):
    # two forwards with their own workspaces in flight together on two
    # streams (the look-back waits only on CTAs of its own grid that have
    # started): each equals the same forward run alone, up to the order in
    # which a chunk's carry was composed (an inclusive prefix, or aggregates
    # and an earlier inclusive: the same value up to rounding)
    shapes = [dict(B=4, T=5000, d_h=96, seed=51), dict(B=1, T=40000, d_h=40, seed=52)]
    Ps, prms, refs = [], [], []
    for sh in shapes:
        w = syn.small_workload(B=sh["B"], T=sh["T"], d_h=sh["d_h"], seed=sh["seed"])
        P, prm = dev(syn.direct_preact(w)), syn.make_params(w)
        H, rho = nr.newton_forward(P, prm, K=3, algo=algo, check=False)
        Ps.append(P), prms.append(prm), refs.append((H.clone(), rho.item()))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        outs = []
        for P, prm, st in zip(Ps, prms, streams):
            with torch.cuda.stream(st):
                outs.append(nr.newton_forward(P, prm, K=3, algo=algo, check=False))
        torch.cuda.synchronize()
        for (H, rho), (Hr, rr) in zip(outs, refs):
            assert (H - Hr).abs().max().item() <= 1e-5
            assert abs(rho.item() - rr) <= 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_and_per_iteration_agree(nr, dtype):
    w = syn.small_workload(B=2, T=1000, d_h=64, dtype=dtype, seed=5)
    P = dev(syn.direct_preact(w), TDT[dtype])
    prm = syn.make_params(w)
    Ha, ra = nr.newton_forward(P, prm, K=3, algo="fused", check=False)
    Hb, rb = nr.newton_forward(P, prm, K=3, algo="per_iter", check=False)
    tol = 1e-5 if dtype == "f32" else 2e-2
    assert (Ha.float() - Hb.float()).abs().max().item() <= tol


def test_newton_K0_is_zero_state_residual(nr):
    w = syn.small_workload(B=2, T=200, d_h=16, seed=7)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    _, rho_ref = oracle.newton(P, prm, 0)
    H, rho = nr.newton_forward(dev(P), prm, K=0, check=False, out=nan_out(2, 200, 16, torch.float32))
    assert torch.count_nonzero(H).item() == 0
    assert abs(rho.item() - rho_ref) < 1e-6


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sequential_matches_oracle(nr, dtype):
    w = syn.small_workload(B=3, T=700, d_h=48, dtype=dtype, seed=9)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Href = oracle.sequential(P, prm)
    H = nr.sequential_forward(dev(P, TDT[dtype]), prm, out=nan_out(3, 700, 48, TDT[dtype]))
    err = np.max(np.abs(host(H) - Href))
    assert err <= (1e-5 if dtype == "f32" else 4e-3), err


RAGGED = [
    [1, 5, 127, 128, 129, 300, 2, 40],
    [0, 128, 0, 0, 128, 1, 1, 1, 256, 0],
    [500],
    [3] * 90,
]


@pytest.mark.parametrize("lens", RAGGED)
@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_ragged_pack_matches_oracle(nr, lens, algo):
    cu = syn.cu_from_lengths(lens)
    N = int(cu[-1])
    w = syn.small_workload(B=1, T=N, d_h=24, seed=len(lens))
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    for K in (1, 3):
        Href, rho_ref = oracle.newton(P, prm, K, cu_seqlens=cu)
        H, rho = nr.newton_forward(dev(P), prm, cu_seqlens=cu, K=K, algo=algo, check=False)
        assert np.max(np.abs(host(H) - Href)) <= 2e-5
        assert abs(rho.item() - rho_ref) <= 2e-5
    Hs = nr.sequential_forward(dev(P), prm, cu_seqlens=cu)
    assert np.max(np.abs(host(Hs) - oracle.sequential(P, prm, cu_seqlens=cu))) <= 1e-5


def test_segment_head_value_is_first_step_of_cell(nr):
    """After any K >= 1 the first token of each segment is f(0, P) of that token."""
    lens = [7, 200, 1, 64]
    cu = syn.cu_from_lengths(lens)
    w = syn.small_workload(B=1, T=int(cu[-1]), d_h=8, seed=3)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Hs = oracle.sequential(P, prm, cu_seqlens=cu)
    for K in (1, 2):
        H, _ = nr.newton_forward(dev(P), prm, cu_seqlens=cu, K=K, check=False)
        heads = cu[:-1][np.diff(cu) > 0]
        np.testing.assert_allclose(host(H)[0, heads], Hs[0, heads], atol=1e-6)


def _heads_np(cu, N):
    m = np.zeros(N, np.uint8)
    if N:
        m[0] = 1
    for i in range(len(cu) - 1):
        if cu[i] < cu[i + 1]:
            m[cu[i]] = 1
    return m


def test_head_mask_bit_exact(nr):
    rng = np.random.default_rng(0)
    cases = [[0, 128, 128, 256, 1000], [0, 1, 2, 3, 4, 5, 6], [0, 0, 0, 5000]]
    for _ in range(5):
        lens = rng.integers(0, 700, size=rng.integers(1, 60))
        cases.append(list(syn.cu_from_lengths(lens)))
    cases.append(list(syn.cu_from_lengths(syn.segment_lengths(4, 64, 262144, 256, 8192))))
    for cu in cases:
        cu = np.asarray(cu, np.int32)
        N = int(cu[-1])
        if N == 0:
            continue
        m = nr.head_mask(cu, N).cpu().numpy()
        np.testing.assert_array_equal(m, _heads_np(cu, N))


def test_residual_entry_point(nr):
    w = syn.small_workload(B=2, T=300, d_h=16, seed=12)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Hs = oracle.sequential(P, prm)
    assert nr.residual(dev(P), prm, dev(Hs)).item() < 2e-6
    G = np.zeros_like(Hs)
    G[1, 17, 3] = 0.5
    ref = oracle.residual(P, prm, G)
    assert abs(nr.residual(dev(P), prm, dev(G)).item() - ref) < 1e-6


def test_divergence_gate(nr):
    w = syn.small_workload(B=1, T=64, d_h=8, seed=1)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    with pytest.raises(nr.NewtonDivergenceError) as ei:
        nr.newton_forward(dev(P), prm, K=0, residual_fail=1e-3)
    assert ei.value.residual > 1e-3 and ei.value.H is not None
    P2 = P.copy()
    P2[0, 10, 3] = np.nan
    with pytest.raises(nr.NewtonDivergenceError) as ei:
        nr.newton_forward(dev(P2), prm, K=3)
    assert math.isinf(ei.value.residual)
    H, rho = nr.newton_forward(dev(P), prm, K=12)        # converged: passes the gate
    assert rho.item() < 1e-5


def test_noncontiguous_preact_is_copied(nr):
    w = syn.small_workload(B=2, T=400, d_h=16, seed=2)
    P = dev(syn.direct_preact(w))
    prm = syn.make_params(w)
    view = P[:, ::2]
    assert not view.is_contiguous()
    Ha, _ = nr.newton_forward(view, prm, K=3, check=False)
    Hb, _ = nr.newton_forward(view.contiguous(), prm, K=3, check=False)
    assert torch.equal(Ha, Hb)


def test_empty_inputs(nr):
    prm = syn.make_params(syn.small_workload(d_h=8))
    for shape in [(0, 10, 24), (2, 0, 24)]:
        P = torch.zeros(shape, device="cuda")
        H, rho = nr.newton_forward(P, prm, K=3)
        assert H.shape == (shape[0], shape[1], 8) and rho.item() == 0.0
        assert nr.sequential_forward(P, prm).shape == (shape[0], shape[1], 8)


def test_bounded_wait_gives_up_and_context_survives(nr):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert nr.bounded_wait(flag, 50_000_000) == 2          # nobody sets it: gives up
    flag.fill_(1)
    assert nr.bounded_wait(flag, 50_000_000) == 1
    assert torch.ones(4, device="cuda").sum().item() == 4.0  # context still usable


PROJ_SHAPES = [(1000, 136, 72), (128, 8, 16), (4097, 512, 256), (300, 1024, 344), (2000, 64, 40)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", PROJ_SHAPES)
def test_input_projection_matches_oracle(nr, dtype, shape):
    # ragged rows (M), gate columns (N = 3 d_h) and d_in (K) against the tiles
    rows, d_in, d_h = shape
    rng = np.random.default_rng(rows + d_in)
    x = rng.normal(size=(rows, d_in)).astype(np.float32)
    W = rng.uniform(-1, 1, size=(3 * d_h, d_in)).astype(np.float32) / math.sqrt(d_in)
    if dtype == "bf16":
        x, W = syn.round_bf16(x), syn.round_bf16(W)
    ref = oracle.input_projection(x, W)
    out = torch.full((rows, 3 * d_h), float("nan"), dtype=TDT[dtype], device="cuda")
    P = nr.input_projection(dev(x, TDT[dtype]), dev(W, TDT[dtype]), out=out)
    assert not torch.isnan(P).any()
    scale = np.abs(x) @ np.abs(W).T
    rel = np.max(np.abs(host(P) - ref) / (scale + 1e-30))
    # f32: split-TF32 tensor-core products (three TF32 terms, error of order
    # 2^-21 of sum |x||W|) with fp32 sums, checked against the 1e-5 relative
    # band of the projection; bf16: exact products, fp32 sums, one bf16 rounding
    assert rel <= (1e-5 if dtype == "f32" else 8e-3), rel


@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_lookback_timeout_is_reported_and_context_survives(nr, algo):
    """A tile that never publishes makes its successors' bounded waits run out:
    the call terminates, reports NRNN_ERR_TIMEOUT, and the next call is correct."""
    w = syn.small_workload(B=1, T=1000, d_h=16, seed=90)    # one column of chunks
    assert nr.lookback_form(1, 1000, 16, torch.float32, algo) == "plain"
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    old_limit = nr.set_wait_limit_ns(2_000_000)               # 2 ms
    try:
        nr.debug_withhold_publish(2)                          # chunk 2 of the column
        with pytest.raises(nr.NrnnError) as ei:
            nr.newton_forward(dev(P), prm, K=2, algo=algo)
        assert ei.value.status == -6
    finally:
        nr.debug_withhold_publish(-1)
        nr.set_wait_limit_ns(old_limit)
    Href, _ = oracle.newton(P, prm, 2)
    H, _ = nr.newton_forward(dev(P), prm, K=2, algo=algo)
    assert np.max(np.abs(host(H) - Href)) <= 2e-5


@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_lookback_timeout_in_the_early_form(nr, algo):
    """320 columns (10 rows x 32 unit tiles) leave at most 4 chunks of a column
    resident, so the launcher takes the early look-back form, which reads the
    nearest predecessors' slots before the CTA barrier: a tile that withholds
    its publish still makes its successors' bounded waits run out, the call
    reports NRNN_ERR_TIMEOUT, and the next call is correct."""
    w = syn.small_workload(B=10, T=256, d_h=1024, seed=91)   # 4 chunks per column
    assert nr.lookback_form(10, 256, 1024, torch.float32, algo) == "early"
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    n_ut, n_chunks = 1024 // 32, 4
    old_limit = nr.set_wait_limit_ns(2_000_000)               # 2 ms
    try:
        nr.debug_withhold_publish((3 * n_ut + 5) * n_chunks + 1)   # row 3, unit tile 5, chunk 1
        with pytest.raises(nr.NrnnError) as ei:
            nr.newton_forward(dev(P), prm, K=2, algo=algo)
        assert ei.value.status == -6
    finally:
        nr.debug_withhold_publish(-1)
        nr.set_wait_limit_ns(old_limit)
    units = np.array([0, 5 * 32 + 7, 1023])
    Pc, pc = oracle.columns(P, prm, units)
    Href, _ = oracle.newton(Pc, pc, 2)
    H, _ = nr.newton_forward(dev(P), prm, K=2, algo=algo)
    assert np.max(np.abs(host(H)[:, :, units] - Href)) <= 2e-5


def test_probe_xu_rates(nr):
    # special-function throughput per SM clock: a power-of-two rate on every
    # NVIDIA part so far; ex2 at least as fast as rcp
    ex2, rcp, tanh = nr.probe_xu_rates()
    assert 4.0 < ex2 < 80.0 and 2.0 < rcp < 80.0 and 2.0 < tanh < 80.0
    assert ex2 >= 0.9 * rcp
