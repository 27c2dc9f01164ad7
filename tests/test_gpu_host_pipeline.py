"""The host-buffer Newton forward (nrnn_newton_forward_host): blocks of rows or
of whole segments streamed through the device forward with overlapped copies,
against the float64 oracle and against the device entry point."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
TOL = {"f32": 2e-5, "bf16": 5e-2}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def nr():
    import nonlinear_rnn_gb300 as m
    return m


def host_tensor(a, dtype, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dtype)
    return t.pin_memory() if pinned else t


def as_f64(t):
    return t.float().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows_per_block", [1, 2, 0])
def test_row_blocks_match_oracle_and_device_call(nr, dtype, rows_per_block):
    w = syn.small_workload(B=5, T=300, d_h=40, seed=61)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Pq = as_f64(host_tensor(P, TDT[dtype]))              # the values as stored
    tpb = rows_per_block * w.T                            # 0: the default split
    H, rho = nr.newton_forward_host(host_tensor(P, TDT[dtype]), prm, K=3, tokens_per_block=tpb)
    Href, rho_ref = oracle.newton(Pq, prm, 3)
    assert H.device.type == "cpu" and H.dtype == TDT[dtype]
    assert np.max(np.abs(as_f64(H) - Href)) <= TOL[dtype]
    Hd, rd = nr.newton_forward(host_tensor(P, TDT[dtype]).cuda(), prm, K=3)
    assert np.max(np.abs(as_f64(H) - Hd.float().cpu().numpy())) <= (1e-5 if dtype == "f32" else 2e-2)
    assert abs(rho - rd.item()) <= (1e-5 if dtype == "f32" else 2e-2)
    assert abs(rho - rho_ref) <= TOL[dtype]


@pytest.mark.parametrize("tokens_per_block", [1, 300, 0])
def test_segment_blocks_of_a_pack(nr, tokens_per_block):
    cu = syn.cu_from_lengths([100, 1, 0, 250, 129, 64, 0, 300, 7])
    w = syn.small_workload(B=1, T=int(cu[-1]), d_h=24, seed=62)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    H, rho = nr.newton_forward_host(host_tensor(P, torch.float32), prm, cu_seqlens=cu, K=3,
                                    tokens_per_block=tokens_per_block)
    Href, rho_ref = oracle.newton(P, prm, 3, cu_seqlens=cu)
    assert np.max(np.abs(as_f64(H) - Href)) <= TOL["f32"]
    assert abs(rho - rho_ref) <= TOL["f32"]


def test_pageable_memory_k0_and_empty(nr):
    w = syn.small_workload(B=3, T=200, d_h=16, seed=63)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    H, rho = nr.newton_forward_host(host_tensor(P, torch.float32, pinned=False), prm, K=2,
                                    out=torch.empty((3, 200, 16)), tokens_per_block=200)
    Href, _ = oracle.newton(P, prm, 2)
    assert np.max(np.abs(as_f64(H) - Href)) <= TOL["f32"]
    H0, r0 = nr.newton_forward_host(host_tensor(P, torch.float32), prm, K=0, check=False)
    assert np.all(as_f64(H0) == 0.0)
    assert abs(r0 - oracle.residual(P, prm, np.zeros_like(Href))) <= 1e-6
    He, re = nr.newton_forward_host(torch.empty((2, 0, 48)), np.zeros((6, 16)), K=3)
    assert He.shape == (2, 0, 16) and re == 0.0


def test_divergence_and_staging_errors(nr):
    w = syn.small_workload(B=2, T=100, d_h=8, seed=64)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    P2 = P.copy()
    P2[1, 40, 3] = np.nan
    with pytest.raises(nr.NewtonDivergenceError) as ei:
        nr.newton_forward_host(host_tensor(P2, torch.float32), prm, K=3, tokens_per_block=100)
    assert math.isinf(ei.value.residual)
    need = nr.host_staging_bytes(2, 100, 8, torch.float32, 3, tokens_per_block=100)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    lib = nr.load()
    Ph = host_tensor(P, torch.float32)
    with pytest.raises(nr.NrnnError) as ei2:
        Hh = torch.empty((2, 100, 8)).pin_memory()
        prm_d = nr.params_tensor(prm, 8, "cuda")
        rho = ctypes.c_float(0)
        st = lib.nrnn_newton_forward_host(ctypes.c_void_p(Ph.data_ptr()), 0, ctypes.c_void_p(prm_d.data_ptr()),
                                          2, 100, 8, None, 0, 3, 1.0, ctypes.c_void_p(Hh.data_ptr()),
                                          ctypes.byref(rho), ctypes.c_void_p(small.data_ptr()),
                                          small.numel(), 100, None)
        nr._binding._raise(st, "newton_forward_host")
    assert ei2.value.status == -7


def _x_case(dtype, B, T, d_in, d_h, seed, cu=None):
    w = syn.small_workload(B=B, T=T, d_in=d_in, d_h=d_h, dtype=dtype, seed=seed)
    inp = syn.make_inputs(w)
    P = oracle.input_projection(inp["x"], inp["W_x"])
    if dtype == "bf16":
        P = syn.round_bf16(P.astype(np.float32))    # the projection stores bf16
    return inp, P


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows_per_block", [1, 3, 0])
def test_x_input_row_blocks_match_oracle_and_device_calls(nr, dtype, rows_per_block):
    B, T, d_in, d_h = 5, 260, 64, 72
    inp, Pref = _x_case(dtype, B, T, d_in, d_h, seed=65)
    prm = inp["params"]
    xh = host_tensor(inp["x"], TDT[dtype])
    Wd = torch.from_numpy(inp["W_x"]).to(TDT[dtype]).cuda()
    H, rho = nr.newton_forward_x_host(xh, Wd, prm, K=3, tokens_per_block=rows_per_block * T)
    assert H.device.type == "cpu" and H.dtype == TDT[dtype] and H.shape == (B, T, d_h)
    Href, rho_ref = oracle.newton(Pref, prm, 3)
    assert np.max(np.abs(as_f64(H) - Href)) <= TOL[dtype]
    assert abs(rho - rho_ref) <= TOL[dtype]
    # the device entry points on the same values: projection, then the forward
    Pd = nr.input_projection(xh.cuda(), Wd)
    Hd, rd = nr.newton_forward(Pd, prm, K=3)
    assert np.max(np.abs(as_f64(H) - Hd.float().cpu().numpy())) <= (1e-5 if dtype == "f32" else 2e-2)
    assert abs(rho - rd.item()) <= (1e-5 if dtype == "f32" else 2e-2)


@pytest.mark.parametrize("tokens_per_block", [1, 400, 0])
def test_x_input_segment_blocks_of_a_pack(nr, tokens_per_block):
    cu = syn.cu_from_lengths([100, 1, 0, 250, 129, 64, 0, 300, 7])
    inp, Pref = _x_case("f32", 1, int(cu[-1]), 24, 40, seed=66)
    H, rho = nr.newton_forward_x_host(host_tensor(inp["x"], torch.float32),
                                      torch.from_numpy(inp["W_x"]).cuda(), inp["params"],
                                      cu_seqlens=cu, K=3, tokens_per_block=tokens_per_block)
    Href, rho_ref = oracle.newton(Pref, inp["params"], 3, cu_seqlens=cu)
    assert np.max(np.abs(as_f64(H) - Href)) <= TOL["f32"]
    assert abs(rho - rho_ref) <= TOL["f32"]


def test_x_input_pageable_empty_and_errors(nr):
    inp, Pref = _x_case("f32", 2, 150, 16, 24, seed=67)
    Wd = torch.from_numpy(inp["W_x"]).cuda()
    H, rho = nr.newton_forward_x_host(host_tensor(inp["x"], torch.float32, pinned=False), Wd,
                                      inp["params"], K=2, out=torch.empty((2, 150, 24)),
                                      tokens_per_block=150)
    Href, _ = oracle.newton(Pref, inp["params"], 2)
    assert np.max(np.abs(as_f64(H) - Href)) <= TOL["f32"]
    He, re = nr.newton_forward_x_host(torch.empty((3, 0, 16)), Wd, inp["params"], K=3)
    assert He.shape == (3, 0, 24) and re == 0.0
    # a NaN in x reaches the residual gate of its block
    x2 = inp["x"].copy()
    x2[1, 70, 5] = np.nan
    with pytest.raises(nr.NewtonDivergenceError) as ei:
        nr.newton_forward_x_host(host_tensor(x2, torch.float32), Wd, inp["params"], K=3,
                                 tokens_per_block=150)
    assert math.isinf(ei.value.residual)
    # W_x misaligned on the device: rejected before any work
    lib = nr.load()
    need = nr.x_host_staging_bytes(2, 150, 16, 24, torch.float32, 3)
    stg = torch.empty(need, dtype=torch.uint8, device="cuda")
    Wbuf = torch.empty(Wd.numel() + 1, device="cuda")
    Wbuf[1:].copy_(Wd.reshape(-1))
    prm_d = nr.params_tensor(inp["params"], 24, "cuda")
    xh = host_tensor(inp["x"], torch.float32)
    Hh = torch.empty((2, 150, 24)).pin_memory()
    rho_c = ctypes.c_float(0)
    vp = ctypes.c_void_p

    def call(W_ptr, nbytes):
        return lib.nrnn_newton_forward_x_host(vp(xh.data_ptr()), vp(W_ptr), 0, vp(prm_d.data_ptr()),
                                              2, 150, 16, 24, None, 0, 3, 1.0, vp(Hh.data_ptr()),
                                              ctypes.byref(rho_c), vp(stg.data_ptr()), nbytes, 0, None)
    assert call(Wbuf.data_ptr() + 4, need) == -1          # NRNN_ERR_INVALID_ARG
    assert call(Wd.data_ptr(), need - 256) == -7          # NRNN_ERR_WORKSPACE
    assert call(Wd.data_ptr(), need) == 0
    assert np.max(np.abs(as_f64(Hh) - oracle.newton(Pref, inp["params"], 3)[0])) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_x_input_pack_blocks_on_segment_aligned_chunks(nr, dtype):
    """Blocks of 16 whole segments of a 32-segment pack: each block is a pack
    of its own with at most one segment per 8 chunks, so the forward inside
    runs on segment-aligned chunks."""
    lens = syn.segment_lengths(5, 32, 16384, 256, 768)
    cu = syn.cu_from_lengths(lens)
    N = int(cu[-1])
    inp, Pref = _x_case(dtype, 1, N, 32, 40, seed=68)
    H, rho = nr.newton_forward_x_host(host_tensor(inp["x"], TDT[dtype]),
                                      torch.from_numpy(inp["W_x"]).to(TDT[dtype]).cuda(),
                                      inp["params"], cu_seqlens=cu, K=3, tokens_per_block=N // 2)
    Href, rho_ref = oracle.newton(Pref, inp["params"], 3, cu_seqlens=cu)
    assert np.max(np.abs(as_f64(H) - Href)) <= TOL[dtype]
    assert abs(rho - rho_ref) <= TOL[dtype]
