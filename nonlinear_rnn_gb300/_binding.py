"""ctypes binding of libnrnn.so (C ABI in include/nrnn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  torch supplies device memory (outputs and the workspace) and the
current stream.  There is no fallback: if the library cannot be loaded the
import of this module fails."""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass, field

import numpy as np
import torch

from . import build as _build

# status codes (include/nrnn.h)
OK, ERR_INVALID_ARG, ERR_CU_SEQLENS, ERR_UNSUPPORTED = 0, -1, -2, -3
ERR_CUDA, ERR_DIVERGED, ERR_TIMEOUT, ERR_WORKSPACE = -4, -5, -6, -7
F32, BF16 = 0, 1
ALGOS = {"auto": 0, "per_iter": 1, "fused": 2}
GATE_ORDER = ("a_z", "a_r", "a_c", "b_z", "b_r", "b_c")

_lock = threading.Lock()
_lib = None

_c = ctypes
_vp, _i64, _int, _f, _sz, _u64 = _c.c_void_p, _c.c_int64, _c.c_int, _c.c_float, _c.c_size_t, _c.c_uint64
_SIGNATURES = {
    "nrnn_status_string": ([_int], _c.c_char_p),
    "nrnn_version": ([], _int),
    "nrnn_validate_cu_seqlens": ([_vp, _i64, _i64], _int),
    "nrnn_newton_workspace_bytes": ([_i64, _i64, _i64, _int, _int, _int], _sz),
    "nrnn_newton_workspace_bytes_pack": ([_i64, _i64, _int, _int, _int, _i64], _sz),
    "nrnn_newton_forward": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _int, _f, _int, _vp,
                             _vp, _vp, _vp, _sz, _vp], _int),
    "nrnn_newton_forward_init": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _int, _f,
                                  _int, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "nrnn_newton_forward_x": ([_vp, _vp, _int, _vp, _i64, _i64, _i64, _i64, _vp, _i64, _int, _f,
                               _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "nrnn_newton_backward": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _vp,
                              _vp, _sz, _vp], _int),
    "nrnn_picard": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _int, _vp, _vp, _vp], _int),
    "nrnn_decode_step": ([_vp, _int, _vp, _i64, _i64, _vp, _vp, _vp], _int),
    "nrnn_decode_step_x": ([_vp, _vp, _int, _vp, _i64, _i64, _i64, _vp, _vp, _vp], _int),
    "nrnn_sequential_forward": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp], _int),
    "nrnn_residual": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp], _int),
    "nrnn_input_projection_workspace_bytes": ([_int, _i64, _i64], _sz),
    "nrnn_input_projection": ([_vp, _vp, _int, _i64, _i64, _i64, _vp, _vp, _sz, _vp], _int),
    "nrnn_debug_head_mask": ([_vp, _i64, _i64, _vp, _vp], _int),
    "nrnn_debug_bounded_wait": ([_vp, _u64, _vp, _vp], _int),
    "nrnn_set_wait_limit_ns": ([_u64], _u64),
    "nrnn_debug_withhold_publish": ([_i64], _i64),
    "nrnn_debug_lookback_form": ([_i64, _i64, _i64, _int, _int], _int),
    "nrnn_debug_pack_plan": ([_vp, _i64, _i64, _int, _vp, _vp], _int),
    "nrnn_probe_xu_rates": ([ctypes.POINTER(ctypes.c_float)] * 3 + [_vp], _int),
    "nrnn_newton_host_staging_bytes": ([_i64, _i64, _i64, _int, _int, _vp, _i64, _i64], _sz),
    "nrnn_newton_forward_host": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _int, _f, _vp, _vp,
                                  _vp, _sz, _i64, _vp], _int),
    "nrnn_newton_x_host_staging_bytes": ([_i64, _i64, _i64, _i64, _int, _int, _vp, _i64, _i64], _sz),
    "nrnn_newton_forward_x_host": ([_vp, _vp, _int, _vp, _i64, _i64, _i64, _i64, _vp, _i64, _int, _f,
                                    _vp, _vp, _vp, _sz, _i64, _vp], _int),
    "nrnn_newton_forward_noalloc": ([_vp, _int, _vp, _i64, _i64, _i64, _vp, _i64, _int, _f, _vp,
                                     _vp, _vp, _vp], _int),
}
EXPORTED = tuple(_SIGNATURES)


def lib_path() -> str:
    return _build.LIB


def load():
    """Loads libnrnn.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


class NrnnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {load().nrnn_status_string(status).decode()} ({status})")


class NewtonDivergenceError(NrnnError):
    """max|F(H^(K))| above residual_fail (or not finite); H and rho are attached."""

    def __init__(self, status, what, H=None, residual=None):
        super().__init__(status, what)
        self.H = H
        self.residual = residual


class AgreementError(AssertionError):
    pass


def _raise(status: int, what: str, **kw):
    if status == OK:
        return
    if status == ERR_DIVERGED:
        raise NewtonDivergenceError(status, what, **kw)
    if status == ERR_UNSUPPORTED:
        raise TypeError(f"{what}: {load().nrnn_status_string(status).decode()}")
    if status in (ERR_INVALID_ARG, ERR_CU_SEQLENS):
        raise ValueError(f"{what}: {load().nrnn_status_string(status).decode()}")
    raise NrnnError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _device_tensor(t: torch.Tensor, what: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    return t.contiguous()   # strided views are copied (shapes_layout: one extra copy)


def params_tensor(params, d_h: int, device) -> torch.Tensor:
    """(6, d_h) fp32 device tensor from a dict (a_z, a_r, a_c, b_z, b_r, b_c) or array."""
    if isinstance(params, dict):
        rows = [torch.as_tensor(np.asarray(params[k]) if not isinstance(params[k], torch.Tensor)
                                else params[k]) for k in GATE_ORDER]
        p = torch.stack([r.to(torch.float32).reshape(-1).cpu() for r in rows])
    else:
        p = torch.as_tensor(params).to(torch.float32)
    if tuple(p.shape) != (6, d_h):
        raise ValueError(f"params must have shape (6, {d_h}), got {tuple(p.shape)}")
    return p.to(device).contiguous()


def validate_cu_seqlens(cu_seqlens, N: int) -> np.ndarray:
    """Host check of a cu_seqlens array (S+1 offsets, 0 .. N, non-decreasing)."""
    cu = cu_seqlens.detach().cpu().numpy() if isinstance(cu_seqlens, torch.Tensor) else np.asarray(cu_seqlens)
    if cu.ndim != 1 or cu.size < 2:
        raise ValueError("cu_seqlens must be 1-D with at least 2 entries")
    if cu.min() < np.iinfo(np.int32).min or cu.max() > np.iinfo(np.int32).max:
        raise ValueError("cu_seqlens does not fit in int32")
    cu32 = np.ascontiguousarray(cu, dtype=np.int32)
    st = load().nrnn_validate_cu_seqlens(cu32.ctypes.data_as(ctypes.c_void_p), cu32.size - 1, int(N))
    _raise(st, "validate_cu_seqlens")
    return cu32


class DeviceCuSeqlens:
    """cu_seqlens validated once on the host and kept on the device, so that
    calls (and CUDA-graph captures of them) need no host-to-device copy."""

    def __init__(self, cu_seqlens, N: int, device="cuda"):
        cu32 = validate_cu_seqlens(cu_seqlens, N)
        self.N = int(N)
        self.num_segments = cu32.size - 1
        self.tensor = torch.from_numpy(cu32).to(device)


def _cu_device(cu_seqlens, B, T, device):
    if cu_seqlens is None:
        return None, 0
    if B != 1:
        raise ValueError("cu_seqlens requires batch 1 (x of shape (1, N, d))")
    if isinstance(cu_seqlens, DeviceCuSeqlens):
        if cu_seqlens.N != T or cu_seqlens.tensor.device != torch.device(device):
            raise ValueError("cu_seqlens was validated for another length or device")
        return cu_seqlens.tensor, cu_seqlens.num_segments
    cu32 = validate_cu_seqlens(cu_seqlens, T)
    return torch.from_numpy(cu32).to(device), cu32.size - 1


def workspace_bytes(B, T, d_h, dtype=torch.float32, K=3, algo="auto", num_segments: int = 0) -> int:
    """Workspace of nrnn_newton_forward; num_segments > 0: for a cu_seqlens pack
    of that many segments (B = 1), with room for segment-aligned chunks."""
    code = F32 if dtype == torch.float32 else BF16
    if num_segments > 0:
        if B != 1:
            raise ValueError("a cu_seqlens pack has batch 1")
        return int(load().nrnn_newton_workspace_bytes_pack(T, d_h, code, K, ALGOS[algo],
                                                           int(num_segments)))
    return int(load().nrnn_newton_workspace_bytes(B, T, d_h, code, K, ALGOS[algo]))


def newton_forward(preact: torch.Tensor, params, cu_seqlens=None, K: int = 3,
                   residual_fail: float = 1.0, algo: str = "auto", check: bool = True,
                   out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                   H_init: torch.Tensor | None = None, picard_iters: int = 0):
    """Parallel Newton forward.  preact (B, T, 3 d_h) float32/bfloat16 CUDA tensor.

    Returns (H, residual): H (B, T, d_h) in preact's dtype and residual, a
    0-dim float32 CUDA tensor holding max|F(H^(K))|.  With check=True the call
    synchronises and raises NewtonDivergenceError if the residual exceeds
    residual_fail (the pages' runtime gate); with check=False nothing syncs.
    H_init starts Newton from a given iterate; picard_iters > 0 first runs that
    many Picard sweeps from zero and starts Newton from their result."""
    lib = load()
    if picard_iters > 0:
        if H_init is not None:
            raise ValueError("give either H_init or picard_iters")
        H_init = picard(preact, params, picard_iters, cu_seqlens=cu_seqlens)
    preact = _device_tensor(preact, "preact")
    if preact.dim() != 3 or preact.shape[2] % 3:
        raise ValueError("preact must have shape (B, T, 3 d_h)")
    B, T, d_h = preact.shape[0], preact.shape[1], preact.shape[2] // 3
    code = _dtype_code(preact)
    dev = preact.device
    prm = params_tensor(params, d_h, dev)
    cu, S = _cu_device(cu_seqlens, B, T, dev)
    H = out if out is not None else torch.empty((B, T, d_h), dtype=preact.dtype, device=dev)
    if tuple(H.shape) != (B, T, d_h) or H.dtype != preact.dtype or not H.is_contiguous():
        raise ValueError("out has the wrong shape, dtype or layout")
    rho = torch.empty((), dtype=torch.float32, device=dev)
    nbytes = (lib.nrnn_newton_workspace_bytes_pack(T, d_h, code, int(K), ALGOS[algo], S) if S > 0
              else lib.nrnn_newton_workspace_bytes(B, T, d_h, code, int(K), ALGOS[algo]))
    if nbytes == 0:
        raise ValueError("invalid shape, K or algo")
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    host = ctypes.c_float(0.0) if check else None
    if H_init is not None:
        H_init = _device_tensor(H_init, "H_init")
        if tuple(H_init.shape) != (B, T, d_h) or H_init.dtype != preact.dtype:
            raise ValueError("H_init must match (B, T, d_h) and preact's dtype")
    with torch.cuda.device(dev):
        st = lib.nrnn_newton_forward_init(_ptr(preact), code, _ptr(prm), B, T, d_h, _ptr(cu), S,
                                          _ptr(H_init), int(K), float(residual_fail),
                                          ALGOS[algo], _ptr(H), _ptr(rho),
                                          ctypes.byref(host) if host is not None else None,
                                          _ptr(workspace), workspace.numel(), _stream(dev))
    _raise(st, "newton_forward", H=H, residual=(host.value if host is not None else None))
    return H, rho


def host_staging_bytes(B, T, d_h, dtype=torch.float32, K=3, cu_seqlens=None,
                       tokens_per_block: int = 0) -> int:
    code = F32 if dtype == torch.float32 else BF16
    cu32 = None if cu_seqlens is None else validate_cu_seqlens(cu_seqlens, T)
    return int(load().nrnn_newton_host_staging_bytes(
        B, T, d_h, code, int(K), None if cu32 is None else cu32.ctypes.data_as(ctypes.c_void_p),
        0 if cu32 is None else cu32.size - 1, int(tokens_per_block)))


def newton_forward_host(preact: torch.Tensor, params, cu_seqlens=None, K: int = 3,
                        residual_fail: float = 1.0, out: torch.Tensor | None = None,
                        staging: torch.Tensor | None = None, tokens_per_block: int = 0,
                        device="cuda", check: bool = True):
    """Newton forward on host tensors with the copies overlapped with the
    kernels (nrnn_newton_forward_host).  preact (B, T, 3 d_h) float32/bfloat16
    CPU tensor, ideally pinned; returns (H, residual): H a CPU tensor (`out`
    if given, else a new pinned one) and residual a Python float.  With
    check=True a residual above residual_fail raises NewtonDivergenceError."""
    lib = load()
    if preact.device.type != "cpu":
        raise ValueError("preact must be a host tensor; use newton_forward for device tensors")
    if not preact.is_contiguous():
        preact = preact.contiguous()
    if preact.dim() != 3 or preact.shape[2] % 3:
        raise ValueError("preact must have shape (B, T, 3 d_h)")
    B, T, d_h = preact.shape[0], preact.shape[1], preact.shape[2] // 3
    code = _dtype_code(preact)
    dev = torch.device(device)
    prm = params_tensor(params, d_h, dev)
    cu32 = None
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens requires batch 1 (x of shape (1, N, d))")
        cu32 = validate_cu_seqlens(cu_seqlens, T)
    H = out if out is not None else torch.empty((B, T, d_h), dtype=preact.dtype).pin_memory()
    if tuple(H.shape) != (B, T, d_h) or H.dtype != preact.dtype or not H.is_contiguous() \
            or H.device.type != "cpu":
        raise ValueError("out must be a contiguous host tensor of shape (B, T, d_h) and preact's dtype")
    cu_ptr = None if cu32 is None else cu32.ctypes.data_as(ctypes.c_void_p)
    S = 0 if cu32 is None else cu32.size - 1
    nbytes = lib.nrnn_newton_host_staging_bytes(B, T, d_h, code, int(K), cu_ptr, S,
                                                int(tokens_per_block))
    if nbytes == 0:
        raise ValueError("invalid shape or K")
    if staging is None or staging.numel() < nbytes:
        staging = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    rho = ctypes.c_float(0.0)
    with torch.cuda.device(dev):
        st = lib.nrnn_newton_forward_host(_ptr(preact), code, _ptr(prm), B, T, d_h, cu_ptr, S,
                                          int(K), float(residual_fail), _ptr(H),
                                          ctypes.byref(rho), _ptr(staging), staging.numel(),
                                          int(tokens_per_block), _stream(dev))
    if st == -5 and not check:
        return H, float(rho.value)
    _raise(st, "newton_forward_host", H=H, residual=float(rho.value))
    return H, float(rho.value)


def x_host_staging_bytes(B, T, d_in, d_h, dtype=torch.float32, K=3, cu_seqlens=None,
                         tokens_per_block: int = 0) -> int:
    code = F32 if dtype == torch.float32 else BF16
    cu32 = None if cu_seqlens is None else validate_cu_seqlens(cu_seqlens, T)
    return int(load().nrnn_newton_x_host_staging_bytes(
        B, T, d_in, d_h, code, int(K),
        None if cu32 is None else cu32.ctypes.data_as(ctypes.c_void_p),
        0 if cu32 is None else cu32.size - 1, int(tokens_per_block)))


def newton_forward_x_host(x: torch.Tensor, W_x: torch.Tensor, params, cu_seqlens=None, K: int = 3,
                          residual_fail: float = 1.0, out: torch.Tensor | None = None,
                          staging: torch.Tensor | None = None, tokens_per_block: int = 0,
                          check: bool = True):
    """Newton forward from x on the host (nrnn_newton_forward_x_host): x (B, T,
    d_in) float32/bfloat16 CPU tensor, ideally pinned; W_x (3 d_h, d_in) a
    device tensor of x's dtype, which names the device.  Each block of x is
    copied in, projected on the device and run through the forward, the
    copies overlapped with the kernels.  Returns (H, residual) as
    newton_forward_host does."""
    lib = load()
    if x.device.type != "cpu":
        raise ValueError("x must be a host tensor; use newton_forward_x for device tensors")
    W_x = _device_tensor(W_x, "W_x")
    if x.dtype != W_x.dtype:
        raise TypeError("x and W_x must share a dtype")
    if not x.is_contiguous():
        x = x.contiguous()
    if x.dim() != 3 or W_x.dim() != 2 or W_x.shape[1] != x.shape[2] or W_x.shape[0] % 3:
        raise ValueError("x must have shape (B, T, d_in) and W_x (3 d_h, d_in)")
    B, T, d_in = x.shape
    d_h = W_x.shape[0] // 3
    code = _dtype_code(x)
    dev = W_x.device
    prm = params_tensor(params, d_h, dev)
    cu32 = None
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens requires batch 1 (x of shape (1, N, d))")
        cu32 = validate_cu_seqlens(cu_seqlens, T)
    H = out if out is not None else torch.empty((B, T, d_h), dtype=x.dtype).pin_memory()
    if tuple(H.shape) != (B, T, d_h) or H.dtype != x.dtype or not H.is_contiguous() \
            or H.device.type != "cpu":
        raise ValueError("out must be a contiguous host tensor of shape (B, T, d_h) and x's dtype")
    cu_ptr = None if cu32 is None else cu32.ctypes.data_as(ctypes.c_void_p)
    S = 0 if cu32 is None else cu32.size - 1
    nbytes = lib.nrnn_newton_x_host_staging_bytes(B, T, d_in, d_h, code, int(K), cu_ptr, S,
                                                  int(tokens_per_block))
    if nbytes == 0:
        raise ValueError("invalid shape or K")
    if staging is None or staging.numel() < nbytes:
        staging = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    rho = ctypes.c_float(0.0)
    with torch.cuda.device(dev):
        st = lib.nrnn_newton_forward_x_host(_ptr(x), _ptr(W_x), code, _ptr(prm), B, T, d_in, d_h,
                                            cu_ptr, S, int(K), float(residual_fail), _ptr(H),
                                            ctypes.byref(rho), _ptr(staging), staging.numel(),
                                            int(tokens_per_block), _stream(dev))
    if st == -5 and not check:
        return H, float(rho.value)
    _raise(st, "newton_forward_x_host", H=H, residual=float(rho.value))
    return H, float(rho.value)


def newton_forward_x(x: torch.Tensor, W_x: torch.Tensor, params, cu_seqlens=None, K: int = 3,
                     residual_fail: float = 1.0, check: bool = True,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Newton forward from x (B, T, d_in) and W_x (3 d_h, d_in), bf16, with the
    input projection computed inside the Newton kernel (P never written)."""
    lib = load()
    x = _device_tensor(x, "x")
    W_x = _device_tensor(W_x, "W_x")
    if x.dim() != 3 or W_x.dim() != 2 or W_x.shape[1] != x.shape[2] or W_x.shape[0] % 3:
        raise ValueError("x must be (B, T, d_in) and W_x (3 d_h, d_in)")
    if x.dtype != W_x.dtype:
        raise TypeError("x and W_x must share a dtype")
    B, T, d_in = x.shape
    d_h = W_x.shape[0] // 3
    code = _dtype_code(x)
    dev = x.device
    prm = params_tensor(params, d_h, dev)
    cu, S = _cu_device(cu_seqlens, B, T, dev)
    H = out if out is not None else torch.empty((B, T, d_h), dtype=x.dtype, device=dev)
    rho = torch.empty((), dtype=torch.float32, device=dev)
    nbytes = lib.nrnn_newton_workspace_bytes(B, T, d_h, code, int(K), ALGOS["fused"])
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    host = ctypes.c_float(0.0) if check else None
    with torch.cuda.device(dev):
        st = lib.nrnn_newton_forward_x(_ptr(x), _ptr(W_x), code, _ptr(prm), B, T, d_in, d_h,
                                       _ptr(cu), S, int(K), float(residual_fail), _ptr(H),
                                       _ptr(rho), ctypes.byref(host) if host is not None else None,
                                       _ptr(workspace), workspace.numel(), _stream(dev))
    _raise(st, "newton_forward_x", H=H, residual=(host.value if host is not None else None))
    return H, rho


def newton_backward(preact: torch.Tensor, params, H: torch.Tensor, gH: torch.Tensor,
                    cu_seqlens=None, workspace: torch.Tensor | None = None):
    """Adjoint of the recurrence at trajectory H for upstream gradient gH = dL/dH.
    Returns (gP (B, T, 3 d_h) in preact's dtype, gparams (6, d_h) fp32).  The
    workspace is allocated here unless given (a uint8 CUDA tensor; for a pack
    its size decides between segment-aligned and time-axis chunks)."""
    lib = load()
    preact = _device_tensor(preact, "preact")
    H = _device_tensor(H, "H")
    gH = _device_tensor(gH, "gH")
    B, T, d_h = preact.shape[0], preact.shape[1], preact.shape[2] // 3
    if tuple(H.shape) != (B, T, d_h) or tuple(gH.shape) != (B, T, d_h):
        raise ValueError("H and gH must be (B, T, d_h)")
    if H.dtype != preact.dtype or gH.dtype != preact.dtype:
        raise TypeError("H and gH must share preact's dtype")
    dev = preact.device
    prm = params_tensor(params, d_h, dev)
    cu, S = _cu_device(cu_seqlens, B, T, dev)
    code = _dtype_code(preact)
    gP = torch.empty_like(preact)
    gprm = torch.empty((6, d_h), dtype=torch.float32, device=dev)
    nbytes = (lib.nrnn_newton_workspace_bytes_pack(T, d_h, code, 1, ALGOS["fused"], S) if S > 0
              else lib.nrnn_newton_workspace_bytes(B, T, d_h, code, 1, ALGOS["fused"]))
    ws = workspace if workspace is not None else torch.empty(max(nbytes, 256), dtype=torch.uint8,
                                                             device=dev)
    with torch.cuda.device(dev):
        st = lib.nrnn_newton_backward(_ptr(preact), code, _ptr(prm), B, T, d_h, _ptr(cu), S,
                                      _ptr(H), _ptr(gH), _ptr(gP), _ptr(gprm), _ptr(ws),
                                      ws.numel(), _stream(dev))
    _raise(st, "newton_backward")
    return gP, gprm


def picard(preact: torch.Tensor, params, sweeps: int, cu_seqlens=None,
           out: torch.Tensor | None = None) -> torch.Tensor:
    """Picard sweeps G_t <- f(G_{t-1}, P_t) from G = 0 on the GPU."""
    lib = load()
    preact = _device_tensor(preact, "preact")
    B, T, d_h = preact.shape[0], preact.shape[1], preact.shape[2] // 3
    dev = preact.device
    prm = params_tensor(params, d_h, dev)
    cu, S = _cu_device(cu_seqlens, B, T, dev)
    G = out if out is not None else torch.empty((B, T, d_h), dtype=preact.dtype, device=dev)
    tmp = torch.empty_like(G) if sweeps >= 2 else None
    with torch.cuda.device(dev):
        st = lib.nrnn_picard(_ptr(preact), _dtype_code(preact), _ptr(prm), B, T, d_h, _ptr(cu), S,
                             int(sweeps), _ptr(G), _ptr(tmp), _stream(dev))
    _raise(st, "picard")
    return G


def sequential_forward(preact: torch.Tensor, params, cu_seqlens=None,
                       out: torch.Tensor | None = None) -> torch.Tensor:
    """Sequential unroll on the GPU (one thread per row/segment and unit)."""
    lib = load()
    preact = _device_tensor(preact, "preact")
    if preact.dim() != 3 or preact.shape[2] % 3:
        raise ValueError("preact must have shape (B, T, 3 d_h)")
    B, T, d_h = preact.shape[0], preact.shape[1], preact.shape[2] // 3
    dev = preact.device
    prm = params_tensor(params, d_h, dev)
    cu, S = _cu_device(cu_seqlens, B, T, dev)
    H = out if out is not None else torch.empty((B, T, d_h), dtype=preact.dtype, device=dev)
    with torch.cuda.device(dev):
        st = lib.nrnn_sequential_forward(_ptr(preact), _dtype_code(preact), _ptr(prm), B, T, d_h,
                                         _ptr(cu), S, _ptr(H), _stream(dev))
    _raise(st, "sequential_forward")
    return H


# above this many slots decode_step(x=, W_x=) projects on the tensor cores
# (nrnn_input_projection) and then steps (nrnn_decode_step)
DECODE_X_MAX_SLOTS = 64
DECODE_XG_MIN_D_IN = 512   # bf16 from here on: the C-ABI call's GEMM form at any slot count


def decode_step(params, h: torch.Tensor | None = None, preact: torch.Tensor | None = None,
                x: torch.Tensor | None = None, W_x: torch.Tensor | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """One T = 1 step per slot: h_out = f(h, P) from preact (slots, 3 d_h), or
    from x (slots, d_in) and W_x (3 d_h, d_in) with the projection fused in.
    h (slots, d_h) is the carried state (None = zeros); out may be h."""
    lib = load()
    if (preact is None) == (x is None):
        raise ValueError("give preact, or x and W_x")
    src = preact if preact is not None else x
    src = _device_tensor(src, "preact" if preact is not None else "x")
    dev = src.device
    slots = src.shape[0]
    d_h = (src.shape[1] // 3) if preact is not None else W_x.shape[0] // 3
    prm = params_tensor(params, d_h, dev)
    if h is not None:
        h = _device_tensor(h, "h")
        if tuple(h.shape) != (slots, d_h) or h.dtype != src.dtype:
            raise ValueError("h must be (slots, d_h) in the input dtype")
    H = out if out is not None else torch.empty((slots, d_h), dtype=src.dtype, device=dev)
    with torch.cuda.device(dev):
        if preact is not None:
            st = lib.nrnn_decode_step(_ptr(src), _dtype_code(src), _ptr(prm), slots, d_h, _ptr(h),
                                      _ptr(H), _stream(dev))
        else:
            W_x = _device_tensor(W_x, "W_x")
            if slots > DECODE_X_MAX_SLOTS and not (src.dtype == torch.bfloat16 and
                                                   src.shape[1] >= DECODE_XG_MIN_D_IN):
                # large batches (fp32, or a short bf16 d_in): the projection on
                # the tensor cores, then the step
                P = input_projection(src, W_x)
                st = lib.nrnn_decode_step(_ptr(P), _dtype_code(P), _ptr(prm), slots, d_h, _ptr(h),
                                          _ptr(H), _stream(dev))
            else:
                st = lib.nrnn_decode_step_x(_ptr(src), _ptr(W_x), _dtype_code(src), _ptr(prm),
                                            slots, src.shape[1], d_h, _ptr(h), _ptr(H),
                                            _stream(dev))
    _raise(st, "decode_step")
    return H


def residual(preact: torch.Tensor, params, G: torch.Tensor, cu_seqlens=None) -> torch.Tensor:
    """max|F(G)| of a trajectory G (B, T, d_h) as a 0-dim CUDA tensor."""
    lib = load()
    preact = _device_tensor(preact, "preact")
    G = _device_tensor(G, "G")
    B, T, d_h = preact.shape[0], preact.shape[1], preact.shape[2] // 3
    if tuple(G.shape) != (B, T, d_h) or G.dtype != preact.dtype:
        raise ValueError("G must match preact's (B, T, d_h) and dtype")
    dev = preact.device
    prm = params_tensor(params, d_h, dev)
    cu, S = _cu_device(cu_seqlens, B, T, dev)
    rho = torch.empty((), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib.nrnn_residual(_ptr(preact), _dtype_code(preact), _ptr(prm), B, T, d_h, _ptr(cu),
                               S, _ptr(G), _ptr(rho), _stream(dev))
    _raise(st, "residual")
    return rho


def projection_workspace_bytes(dtype, d_in: int, d_h: int) -> int:
    """Workspace bytes nrnn_input_projection needs (fp32: the low part of W_x)."""
    code = F32 if dtype == torch.float32 else BF16 if dtype == torch.bfloat16 else -1
    return int(load().nrnn_input_projection_workspace_bytes(code, int(d_in), int(d_h)))


def input_projection(x: torch.Tensor, W_x: torch.Tensor, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None):
    """P = x W_x^T: x (..., d_in), W_x (3 d_h, d_in) -> (..., 3 d_h), same dtype.
    fp32 needs a workspace (the low part of W_x; allocated here if not given)."""
    lib = load()
    x = _device_tensor(x, "x")
    W_x = _device_tensor(W_x, "W_x")
    if x.dtype != W_x.dtype:
        raise TypeError("x and W_x must share a dtype")
    d_in = x.shape[-1]
    n_out = W_x.shape[0]
    if W_x.shape[1] != d_in or n_out % 3:
        raise ValueError("W_x must have shape (3 d_h, d_in)")
    rows = x.numel() // d_in
    P = out if out is not None else torch.empty((*x.shape[:-1], n_out), dtype=x.dtype, device=x.device)
    code = _dtype_code(x)
    nbytes = lib.nrnn_input_projection_workspace_bytes(code, d_in, n_out // 3)
    if nbytes > 0 and (workspace is None or workspace.numel() < nbytes):
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        st = lib.nrnn_input_projection(_ptr(x), _ptr(W_x), code, rows, d_in, n_out // 3, _ptr(P),
                                       _ptr(workspace) if nbytes > 0 else None, int(nbytes),
                                       _stream(x.device))
    _raise(st, "input_projection")
    return P


def head_mask(cu_seqlens, N: int, device="cuda") -> torch.Tensor:
    """Segment-head mask as computed on the device by the Newton kernels' routine."""
    lib = load()
    cu32 = validate_cu_seqlens(cu_seqlens, N)
    cu = torch.from_numpy(cu32).to(device)
    mask = torch.empty(N, dtype=torch.uint8, device=device)
    st = lib.nrnn_debug_head_mask(_ptr(cu), cu32.size - 1, N, _ptr(mask), _stream(torch.device(device)))
    _raise(st, "head_mask")
    return mask


def bounded_wait(flag: torch.Tensor, wait_ns: int) -> int:
    """Runs the device bounded wait on flag (uint32/int32 CUDA tensor); 1 = seen, 2 = gave up."""
    lib = load()
    res = torch.zeros(1, dtype=torch.int32, device=flag.device)
    st = lib.nrnn_debug_bounded_wait(_ptr(flag), int(wait_ns), _ptr(res), _stream(flag.device))
    _raise(st, "bounded_wait")
    return int(res.item())


def set_wait_limit_ns(ns: int) -> int:
    return int(load().nrnn_set_wait_limit_ns(int(ns)))


def debug_withhold_publish(tile: int) -> int:
    """Debug: the given Newton tile stops publishing its look-back slot (-1: off)."""
    return int(load().nrnn_debug_withhold_publish(int(tile)))


def pack_plan(cu_seqlens, N: int, device="cuda", reverse: bool = False) -> torch.Tensor:
    """The segment-aligned chunk plan of a pack as the Newton kernels (or, with
    reverse, the backward kernel) take it (nrnn_debug_pack_plan): an (n, 4)
    int32 tensor of {first row, segment end, chunk index within the segment,
    chunk index in segment order}."""
    lib = load()
    cu32 = validate_cu_seqlens(cu_seqlens, N)
    cu = torch.from_numpy(cu32).to(device)
    S = cu32.size - 1
    plan = torch.zeros((2 + (N + 63) // 64 + S, 4), dtype=torch.int32, device=device)
    st = lib.nrnn_debug_pack_plan(_ptr(cu), S, N, int(bool(reverse)), _ptr(plan),
                                  _stream(torch.device(device)))
    _raise(st, "pack_plan")
    n = int(plan[0, 0].item())
    return plan[1:1 + n].cpu()


LOOKBACK_FORMS = {0: "plain", 1: "early"}


def lookback_form(B: int, T: int, d_h: int, dtype=torch.float32, algo: str = "fused") -> str:
    """The look-back form the Newton kernels take for this shape on the current
    device: "plain" or "early" (nrnn_debug_lookback_form)."""
    code = F32 if dtype == torch.float32 else BF16
    st = load().nrnn_debug_lookback_form(int(B), int(T), int(d_h), code, ALGOS[algo])
    _raise(st if st < 0 else 0, "lookback_form")
    return LOOKBACK_FORMS[st]


@dataclass
class AgreementReport:
    ok: bool
    max_abs: float
    atol: float
    K: int
    residual: float
    dtype: str
    extra: dict = field(default_factory=dict)

    def to_dict(self):
        return {"ok": self.ok, "max_abs": self.max_abs, "atol": self.atol, "K": self.K,
                "residual": self.residual, "dtype": self.dtype, **self.extra}


def default_agreement_atol(dtype) -> float:
    return 1e-4 if dtype == torch.float32 else 5e-2


def verify_agreement(preact, params, K: int = 3, cu_seqlens=None, atol: float | None = None,
                     raise_on_fail: bool = False, algo: str = "auto") -> AgreementReport:
    """Runs Newton and the sequential unroll on the same batch and compares them
    by max-abs (numerics contract, "Four echelons / 3. Opt-in oracle")."""
    Hn, rho = newton_forward(preact, params, cu_seqlens=cu_seqlens, K=K, algo=algo, check=False)
    Hs = sequential_forward(preact, params, cu_seqlens=cu_seqlens)
    tol = default_agreement_atol(preact.dtype) if atol is None else float(atol)
    err = float((Hn.float() - Hs.float()).abs().max().item()) if Hn.numel() else 0.0
    rep = AgreementReport(err <= tol, err, tol, int(K), float(rho.item()), str(preact.dtype))
    if raise_on_fail and not rep.ok:
        raise AgreementError(f"Newton vs sequential max_abs {err:.3e} > atol {tol:.1e}")
    return rep


def probe_xu_rates(device="cuda") -> tuple[float, float, float]:
    """(ex2, rcp, tanh) results per SM clock cycle on `device`, measured by the
    library's special-function throughput probe."""
    lib = load()
    dev = torch.device(device)
    e2, rc, th = ctypes.c_float(0.0), ctypes.c_float(0.0), ctypes.c_float(0.0)
    with torch.cuda.device(dev):
        st = lib.nrnn_probe_xu_rates(ctypes.byref(e2), ctypes.byref(rc), ctypes.byref(th),
                                     _stream(dev))
    _raise(st, "probe_xu_rates")
    return float(e2.value), float(rc.value), float(th.value)
