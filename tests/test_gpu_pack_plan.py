"""Segment-aligned chunks of a cu_seqlens pack: the chunk plan the Newton
kernels take, and the forward over it, against the float64 oracle and against
the same forward on chunks of the pack's time axis."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}
TOL = {"f32": 2e-5, "bf16": 5e-2}
# empty, length-1, exactly one chunk, one row short of and past a chunk,
# long segments; 9 segments over 4621 rows = 73 chunks (>= 8 x 9)
EDGE_LENGTHS = [1, 0, 64, 63, 65, 128, 1000, 2000, 1300]


@pytest.fixture(scope="module")
def nr():
    import nonlinear_rnn_gb300 as m
    return m


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dtype)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def expected_chunks(cu):
    """Every (segment, chunk) of a pack: first row, segment end, chunk index
    in the segment, index of the chunk in segment order."""
    out, g = {}, 0
    for s in range(len(cu) - 1):
        n = -(-(int(cu[s + 1]) - int(cu[s])) // 64)
        for j in range(n):
            out[(s, j)] = (int(cu[s]) + 64 * j, int(cu[s + 1]), j, g)
            g += 1
    return out


@pytest.mark.parametrize("lengths", [
    EDGE_LENGTHS,
    list(syn.segment_lengths(7, 64, 262144, 256, 8192)),     # the ragged workload's pack
    [4096] * 16,                                              # equal lengths
])
def test_plan_holds_every_chunk_in_level_order(nr, lengths):
    cu = syn.cu_from_lengths(lengths)
    N = int(cu[-1])
    plan = nr.pack_plan(cu, N).numpy()
    want = expected_chunks(cu)
    assert len(plan) == len(want)
    seg_of_row = np.searchsorted(cu, plan[:, 0], side="right") - 1
    got = {(int(s), int(e[2])): tuple(int(v) for v in e) for s, e in zip(seg_of_row, plan)}
    assert got == want                                    # each chunk once, fields exact
    chunks = -(-np.diff(cu) // 64)
    level = plan[:, 2]
    assert np.all(np.diff(level) >= 0)                    # by chunk index within the segment
    for j in np.unique(level):
        n_seg = chunks[seg_of_row[level == j]]
        assert np.all(np.diff(n_seg) <= 0)                # segments of most chunks first
    pos = {k: i for i, k in enumerate((int(s), int(e[2])) for s, e in zip(seg_of_row, plan))}
    assert all(pos[(s, j - 1)] < pos[(s, j)] for (s, j) in want if j > 0)


def _pair(nr, P, prm, cu, K, algo, dtype):
    """The forward with a workspace sized for the pack (segment-aligned chunks)
    and one sized for the time axis (nrnn_newton_workspace_bytes)."""
    Pd = dev(P, TDT[dtype])
    N, d_h = P.shape[1], P.shape[2] // 3
    ws_pack = torch.empty(nr.workspace_bytes(1, N, d_h, TDT[dtype], K, algo, num_segments=len(cu) - 1),
                          dtype=torch.uint8, device="cuda")
    ws_plain = torch.empty(nr.workspace_bytes(1, N, d_h, TDT[dtype], K, algo), dtype=torch.uint8,
                           device="cuda")
    assert ws_pack.numel() > ws_plain.numel()
    out = torch.full((1, N, d_h), float("nan"), dtype=TDT[dtype], device="cuda")
    Ha, ra = nr.newton_forward(Pd, prm, cu_seqlens=cu, K=K, algo=algo, check=False, out=out,
                               workspace=ws_pack)
    Hb, rb = nr.newton_forward(Pd, prm, cu_seqlens=cu, K=K, algo=algo, check=False,
                               workspace=ws_plain)
    return Ha, ra, Hb, rb


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ["fused", "per_iter"])
@pytest.mark.parametrize("K", [1, 3])
def test_segment_aligned_pack_matches_oracle(nr, dtype, algo, K):
    cu = syn.cu_from_lengths(EDGE_LENGTHS)
    w = syn.small_workload(B=1, T=int(cu[-1]), d_h=40, dtype=dtype, seed=95 + K)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Href, rho_ref = oracle.newton(P, prm, K, cu_seqlens=cu)
    Ha, ra, Hb, rb = _pair(nr, P, prm, cu, K, algo, dtype)
    assert not torch.isnan(Ha).any()                     # every row of every segment written
    assert np.max(np.abs(host(Ha) - Href)) <= TOL[dtype]
    assert abs(ra.item() - rho_ref) <= TOL[dtype]
    # the same values as on time-axis chunks, up to the look-back's grouping
    assert np.max(np.abs(host(Ha) - host(Hb))) <= (1e-5 if dtype == "f32" else 2e-2)


def test_segment_aligned_pack_warm_start(nr):
    """Picard sweeps, then Newton from their result (fused kernel with an
    initial iterate) on segment-aligned chunks."""
    cu = syn.cu_from_lengths(EDGE_LENGTHS)
    w = syn.small_workload(B=1, T=int(cu[-1]), d_h=24, seed=99)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    H, rho = nr.newton_forward(dev(P), prm, cu_seqlens=cu, K=2, picard_iters=2, check=False)
    H0 = oracle.picard(P, prm, 2, cu_seqlens=cu)
    Href, rho_ref = oracle.newton_init(P, prm, 2, H0, cu_seqlens=cu)
    assert np.max(np.abs(host(H) - Href)) <= 2e-5
    assert abs(rho.item() - rho_ref) <= 2e-5


def test_ragged_workload_pack_on_sampled_units(nr):
    """The ragged workload's full pack (N = 262144, 64 segments, d_h = 512)
    on segment-aligned chunks, sampled units against the oracle."""
    w = syn.WORKLOADS[4]
    cu = syn.make_inputs(w, with_x=False)["cu_seqlens"]
    P = syn.preact_uniform_torch(w, device="cuda")
    prm = syn.make_params(w)
    ws = torch.empty(nr.workspace_bytes(1, w.T, w.d_h, P.dtype, w.K, "fused", num_segments=len(cu) - 1),
                     dtype=torch.uint8, device="cuda")
    H, rho = nr.newton_forward(P, prm, cu_seqlens=cu, K=w.K, check=False, workspace=ws)
    units = np.array([0, 31, 32, 200, 511])
    Pc = syn.preact_uniform_columns(w, units)
    Href, _ = oracle.newton(Pc, oracle.pack_params(prm)[:, units], w.K, cu_seqlens=cu, threads=8)
    err = np.max(np.abs(H[:, :, torch.as_tensor(units, device="cuda")].double().cpu().numpy() - Href))
    assert err <= 1e-4, err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_on_segment_aligned_pack(nr, dtype):
    """The adjoint scan on segment-aligned chunks (each chain from the segment's
    end; a segment's short last chunk stores dL/dP row by row) against the
    oracle's adjoint and against the same call on time-axis chunks."""
    cu = syn.cu_from_lengths(EDGE_LENGTHS)
    N, d_h = int(cu[-1]), 40
    tdt = TDT[dtype]
    w = syn.small_workload(B=1, T=N, d_h=d_h, dtype=dtype, seed=97)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    H = oracle.sequential(P, prm, cu_seqlens=cu).astype(np.float32)
    gH = np.random.default_rng(98).normal(size=H.shape).astype(np.float32)
    if dtype == "bf16":
        H, gH = syn.round_bf16(H), syn.round_bf16(gH)
    gP_ref, gprm_ref = oracle.backward(P, prm, H, gH, cu_seqlens=cu)
    ws_pack = torch.empty(nr.workspace_bytes(1, N, d_h, tdt, 1, "fused", num_segments=len(cu) - 1),
                          dtype=torch.uint8, device="cuda")
    ws_plain = torch.empty(nr.workspace_bytes(1, N, d_h, tdt, 1, "fused"), dtype=torch.uint8,
                           device="cuda")
    assert ws_pack.numel() > ws_plain.numel()
    args = (dev(P, tdt), prm, dev(H, tdt), dev(gH, tdt))
    gP, gprm = nr.newton_backward(*args, cu_seqlens=cu, workspace=ws_pack)
    gP2, _ = nr.newton_backward(*args, cu_seqlens=cu, workspace=ws_plain)
    scale = max(1.0, float(np.max(np.abs(gP_ref))))
    tol = 2e-5 if dtype == "f32" else 2e-2
    assert np.max(np.abs(host(gP) - gP_ref)) <= tol * scale
    assert np.max(np.abs(host(gP) - host(gP2))) <= tol * scale
    rel = np.max(np.abs(gprm.cpu().numpy() - gprm_ref)) / max(1.0, float(np.max(np.abs(gprm_ref))))
    assert rel <= (1e-4 if dtype == "f32" else 1e-2)


@pytest.mark.parametrize("lengths", [EDGE_LENGTHS, list(syn.segment_lengths(7, 64, 262144, 256, 8192))])
def test_reverse_plan_order(nr, lengths):
    """The backward's plan: every chunk once, ordered by the number of chunks
    of its segment after it, within that by the segment's chunk count, and
    each chunk after the chunk that follows it in time."""
    cu = syn.cu_from_lengths(lengths)
    plan = nr.pack_plan(cu, int(cu[-1]), reverse=True).numpy()
    want = expected_chunks(cu)
    seg = np.searchsorted(cu, plan[:, 0], side="right") - 1
    got = {(int(s), int(e[2])): tuple(int(v) for v in e) for s, e in zip(seg, plan)}
    assert got == want
    chunks = -(-np.diff(cu) // 64)
    after = chunks[seg] - 1 - plan[:, 2]
    assert np.all(np.diff(after) >= 0)
    for r in np.unique(after):
        assert np.all(np.diff(chunks[seg[after == r]]) <= 0)
    pos = {(int(s), int(e[2])): i for i, (s, e) in enumerate(zip(seg, plan))}
    assert all(pos[(s, j + 1)] < pos[(s, j)] for (s, j) in want if (s, j + 1) in want)


@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_lookback_timeout_on_segment_aligned_chunks(nr, algo):
    """A withheld chunk of a segment-aligned pack (the first chunk of the
    2000-row segment, index 23 in segment order) makes the later chunks of its
    chain give up their bounded waits: the call reports NRNN_ERR_TIMEOUT, and
    the next call is correct."""
    cu = syn.cu_from_lengths(EDGE_LENGTHS)
    N, d_h = int(cu[-1]), 16
    w = syn.small_workload(B=1, T=N, d_h=d_h, seed=96)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    ws = torch.empty(nr.workspace_bytes(1, N, d_h, torch.float32, 2, algo, num_segments=len(cu) - 1),
                     dtype=torch.uint8, device="cuda")
    chunks = -(-np.diff(cu) // 64)
    assert int(chunks[:7].sum()) == 23 and chunks[7] > 1
    old_limit = nr.set_wait_limit_ns(2_000_000)               # 2 ms
    try:
        nr.debug_withhold_publish(23)
        with pytest.raises(nr.NrnnError) as ei:
            nr.newton_forward(dev(P), prm, cu_seqlens=cu, K=2, algo=algo, workspace=ws)
        assert ei.value.status == -6
    finally:
        nr.debug_withhold_publish(-1)
        nr.set_wait_limit_ns(old_limit)
    Href, _ = oracle.newton(P, prm, 2, cu_seqlens=cu)
    H, _ = nr.newton_forward(dev(P), prm, cu_seqlens=cu, K=2, algo=algo, workspace=ws)
    assert np.max(np.abs(host(H) - Href)) <= 2e-5


@pytest.mark.parametrize("algo", ["fused", "per_iter"])
def test_long_pack_whose_plan_takes_its_own_kernel(nr, algo):
    """A pack of 400000 rows and 8 segments: 6250 chunks, so the plan needs
    more shared memory than the clear kernel's blocks should reserve and is
    built by a kernel of its own; the forward on it against the oracle."""
    lens = syn.segment_lengths(11, 8, 400000, 20000, 80000)
    cu = syn.cu_from_lengths(lens)
    N = int(cu[-1])
    assert N == 400000
    w = syn.small_workload(B=1, T=N, d_h=16, seed=101)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    ws = torch.empty(nr.workspace_bytes(1, N, 16, torch.float32, 2, algo, num_segments=8),
                     dtype=torch.uint8, device="cuda")
    assert ws.numel() > nr.workspace_bytes(1, N, 16, torch.float32, 2, algo)
    H, rho = nr.newton_forward(dev(P), prm, cu_seqlens=cu, K=2, algo=algo, check=False, workspace=ws)
    Href, rho_ref = oracle.newton(P, prm, 2, cu_seqlens=cu)
    assert np.max(np.abs(host(H) - Href)) <= 2e-5
    assert abs(rho.item() - rho_ref) <= 2e-5
    plan = nr.pack_plan(cu, N).numpy()
    assert len(plan) == int(sum(-(-int(l) // 64) for l in lens))
