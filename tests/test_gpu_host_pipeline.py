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
