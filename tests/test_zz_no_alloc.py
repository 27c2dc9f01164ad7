"""The no-allocation Newton entry point, called through the C ABI.

nrnn_newton_forward_noalloc serves callers that cannot allocate device memory
(and so cannot hand nrnn_newton_forward a workspace): it keeps its scratch in
one library-owned device array.  These checks run last so that a stop at the
first failure has already run every other test; they pass alone in a fresh
process as well as after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, P, prm, H, rho, K, cu=None, S=0):
    code = 1 if P.dtype == torch.bfloat16 else 0
    B, T, d_h = H.shape
    return lib.nrnn_newton_forward_noalloc(
        _p(P), code, _p(prm), B, T, d_h, None if cu is None else _p(cu), S, K, 1.0,
        _p(H), _p(rho), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ragged", [False, True])
def test_noalloc_matches_workspace_entry_point_on_two_calls(dtype, ragged):
    import nonlinear_rnn_gb300 as nr
    lib = nr.load()
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    if ragged:
        cu_np = syn.cu_from_lengths([130, 1, 0, 300, 77, 256])
        w = syn.small_workload(B=1, T=int(cu_np[-1]), d_h=72, dtype=dtype, seed=31)
        cu = torch.from_numpy(cu_np).cuda()
        S = len(cu_np) - 1
    else:
        w = syn.small_workload(B=3, T=700, d_h=72, dtype=dtype, seed=32)
        cu_np, cu, S = None, None, 0
    P_host = syn.direct_preact(w)
    P = torch.from_numpy(P_host).cuda().to(tdt)
    prm = nr.params_tensor(syn.make_params(w), w.d_h, "cuda")
    H_ref, rho_ref = nr.newton_forward(P, prm, cu_seqlens=cu_np, K=3, algo="fused", check=False)
    # the float64 oracle on the same stored preactivations
    H_orc, rho_orc = oracle.newton(P_host, syn.make_params(w), 3, cu_seqlens=cu_np)
    tol = 1e-4 if dtype == "f32" else 5e-2
    for _ in range(2):   # the second call finds the first call's scratch contents
        H = torch.full_like(H_ref, float("nan"))
        rho = torch.full((), float("nan"), device="cuda")
        assert _noalloc(lib, P, prm, H, rho, 3, cu, S) == 0
        torch.cuda.synchronize()
        assert not torch.isnan(H).any()
        assert (H.float() - H_ref.float()).abs().max().item() <= tol
        assert abs(rho.item() - rho_ref.item()) <= tol
        assert float(np.max(np.abs(H.double().cpu().numpy() - H_orc))) <= tol
        assert abs(rho.item() - rho_orc) <= tol


def test_noalloc_rejects_requests_beyond_its_scratch():
    import nonlinear_rnn_gb300 as nr
    lib = nr.load()
    B, T, d_h, K = 16, 1 << 22, 1024, 3
    need = lib.nrnn_newton_workspace_bytes(B, T, d_h, 0, K, 2)
    assert need > 64 * 1024 * 1024
    # null data pointers: the size check must fail before anything touches them
    st = lib.nrnn_newton_forward_noalloc(None, 0, None, B, T, d_h, None, 0, K, 1.0, None, None,
                                         None, None)
    assert st == -7
