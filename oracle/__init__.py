"""TEST INFRASTRUCTURE -- float64 CPU oracle for the diagonal-GRU Newton forward.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (``nonlinear_rnn_gb300``)
never does, and nothing here imports the product.

What it computes (pararnn-torch pages: FAQs "Does parallel Newton match
sequential unroll?", numerics contract "Invariant" / "Two thresholds",
shapes_layout "cu_seqlens"):

* ``sequential``     -- the definition: h_t = f(h_{t-1}, P_t) from h = 0 per row
                        or per segment (``sequential_apply``);
* ``newton``         -- the parallel-Newton algorithm run step by step in float64:
                        K iterations from H = 0 of F/J evaluation at the shifted
                        trajectory, the affine recurrence delta_t = J_t delta_{t-1} - F_t
                        solved by a sequential loop, H <- H + delta; returns H and
                        rho = max|F(H^(K))| (J = 0 and shifted state 0 at segment heads);
* ``residual``       -- max|F(G)| for a given trajectory G;
* ``picard``         -- Picard sweeps G_t <- f(G_{t-1}, P_t) from G = 0 (warm start);
* ``newton_init``    -- the Newton algorithm started from a given iterate;
* ``cell``           -- one step f(h, P) and df/dh;
* ``decode_step``    -- one T = 1 step per slot with a carried state;
* ``backward``       -- adjoint of the unroll: dL/dP and dL/d(params) from dL/dH;
* ``input_projection`` -- P = x W_x^T in float64 (a library matmul).

The arithmetic lives in ``nrnn_oracle.c`` (plain C, float64, no fused
multiply-add contraction) and is reached through ctypes.  Calls split the
unit range across threads; ctypes releases the GIL during each call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nrnn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

GATE_ORDER = ("a_z", "a_r", "a_c", "b_z", "b_r", "b_c")


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (float64, IEEE, no contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            lib.oracle_cell.argtypes = [ctypes.c_double] * 4 + [dp, dp, dp]
            lib.oracle_cell.restype = None
            lib.oracle_sequential.argtypes = [dp, dp, i64, i64, i64, lp, i64, i64, i64, dp]
            lib.oracle_sequential.restype = None
            lib.oracle_newton.argtypes = [dp, dp, i64, i64, i64, lp, i64, i64, i64, i64, dp]
            lib.oracle_newton.restype = ctypes.c_double
            lib.oracle_residual.argtypes = [dp, dp, i64, i64, i64, lp, i64, i64, i64, dp]
            lib.oracle_residual.restype = ctypes.c_double
            lib.oracle_picard.argtypes = [dp, dp, i64, i64, i64, lp, i64, i64, i64, i64, dp]
            lib.oracle_picard.restype = None
            lib.oracle_newton_init.argtypes = [dp, dp, i64, i64, i64, lp, i64, i64, dp, i64, i64,
                                               dp]
            lib.oracle_newton_init.restype = ctypes.c_double
            lib.oracle_backward.argtypes = [dp, dp, i64, i64, i64, lp, i64, dp, dp, i64, i64,
                                            dp, dp]
            lib.oracle_backward.restype = None
            _lib = lib
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def pack_params(params) -> np.ndarray:
    """(6, d_h) float64 in the order a_z, a_r, a_c, b_z, b_r, b_c."""
    if isinstance(params, dict):
        rows = [np.asarray(params[k], dtype=np.float64) for k in GATE_ORDER]
        return np.ascontiguousarray(np.stack(rows))
    return np.ascontiguousarray(np.asarray(params, dtype=np.float64))


def _prep(P, params, cu_seqlens):
    P = np.ascontiguousarray(np.asarray(P, dtype=np.float64))
    assert P.ndim == 3 and P.shape[2] % 3 == 0, "P must be (B, T, 3 d_h)"
    B, T, three_dh = P.shape
    d_h = three_dh // 3
    prm = pack_params(params)
    assert prm.shape == (6, d_h)
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        assert B == 1 and cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
        S = len(cu) - 1
    else:
        cu, S = None, 0
    return P, prm, B, T, d_h, cu, S


def _ranges(d_h: int, threads: int):
    threads = max(1, min(threads, d_h))
    step = (d_h + threads - 1) // threads
    return [(j, min(d_h, j + step)) for j in range(0, d_h, step)]


def _run(fn, d_h, threads):
    rs = _ranges(d_h, threads)
    if len(rs) == 1:
        return [fn(*rs[0])]
    with ThreadPoolExecutor(len(rs)) as ex:
        return list(ex.map(lambda r: fn(*r), rs))


def cell(h, pz, pr, pc, prm6):
    """f(h, P) and df/dh for one unit; prm6 = (a_z, a_r, a_c, b_z, b_r, b_c)."""
    lib = _load()
    prm = np.ascontiguousarray(np.asarray(prm6, dtype=np.float64))
    f = ctypes.c_double()
    J = ctypes.c_double()
    lib.oracle_cell(float(h), float(pz), float(pr), float(pc), _dptr(prm),
                    ctypes.byref(f), ctypes.byref(J))
    return f.value, J.value


def sequential(P, params, cu_seqlens=None, threads: int = 1) -> np.ndarray:
    """Sequential unroll; returns H (B, T, d_h) float64."""
    lib = _load()
    P, prm, B, T, d_h, cu, S = _prep(P, params, cu_seqlens)
    H = np.zeros((B, T, d_h), dtype=np.float64)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if cu is not None else None
    _run(lambda j0, j1: lib.oracle_sequential(_dptr(P), _dptr(prm), B, T, d_h, cup, S,
                                              j0, j1, _dptr(H)), d_h, threads)
    return H


def newton(P, params, K: int, cu_seqlens=None, threads: int = 1):
    """K Newton iterations from H = 0; returns (H float64 (B, T, d_h), rho)."""
    lib = _load()
    P, prm, B, T, d_h, cu, S = _prep(P, params, cu_seqlens)
    H = np.zeros((B, T, d_h), dtype=np.float64)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if cu is not None else None
    rhos = _run(lambda j0, j1: lib.oracle_newton(_dptr(P), _dptr(prm), B, T, d_h, cup, S,
                                                 int(K), j0, j1, _dptr(H)), d_h, threads)
    return H, _max_rho(rhos)


def residual(P, params, G, cu_seqlens=None, threads: int = 1) -> float:
    """max |F(G)| of a trajectory G (B, T, d_h)."""
    lib = _load()
    P, prm, B, T, d_h, cu, S = _prep(P, params, cu_seqlens)
    G = np.ascontiguousarray(np.asarray(G, dtype=np.float64))
    assert G.shape == (B, T, d_h)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if cu is not None else None
    rhos = _run(lambda j0, j1: lib.oracle_residual(_dptr(P), _dptr(prm), B, T, d_h, cup, S,
                                                   j0, j1, _dptr(G)), d_h, threads)
    return _max_rho(rhos)


def picard(P, params, sweeps: int, cu_seqlens=None, threads: int = 1) -> np.ndarray:
    """Picard sweeps G_t <- f(G_{t-1}, P_t) from G = 0; returns G (B, T, d_h) float64."""
    lib = _load()
    P, prm, B, T, d_h, cu, S = _prep(P, params, cu_seqlens)
    G = np.zeros((B, T, d_h), dtype=np.float64)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if cu is not None else None
    _run(lambda j0, j1: lib.oracle_picard(_dptr(P), _dptr(prm), B, T, d_h, cup, S, int(sweeps),
                                          j0, j1, _dptr(G)), d_h, threads)
    return G


def newton_init(P, params, K: int, H0, cu_seqlens=None, threads: int = 1):
    """K Newton iterations from the iterate H0; returns (H, rho)."""
    lib = _load()
    P, prm, B, T, d_h, cu, S = _prep(P, params, cu_seqlens)
    H0 = np.ascontiguousarray(np.asarray(H0, dtype=np.float64))
    assert H0.shape == (B, T, d_h)
    H = np.zeros((B, T, d_h), dtype=np.float64)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if cu is not None else None
    rhos = _run(lambda j0, j1: lib.oracle_newton_init(_dptr(P), _dptr(prm), B, T, d_h, cup, S,
                                                      int(K), _dptr(H0), j0, j1, _dptr(H)),
                d_h, threads)
    return H, _max_rho(rhos)


def _max_rho(rhos):
    out = 0.0
    for r in rhos:
        if not (r <= out):
            out = float(r)
    return out


def backward(P, params, H, gH, cu_seqlens=None, threads: int = 1):
    """Adjoint pass through h_t = f(h_{t-1}, P_t) at trajectory H for upstream
    gradient gH (both (B, T, d_h)); returns (gP (B, T, 3 d_h), gparams (6, d_h))."""
    lib = _load()
    P, prm, B, T, d_h, cu, S = _prep(P, params, cu_seqlens)
    H = np.ascontiguousarray(np.asarray(H, dtype=np.float64))
    gH = np.ascontiguousarray(np.asarray(gH, dtype=np.float64))
    assert H.shape == gH.shape == (B, T, d_h)
    gP = np.zeros((B, T, 3 * d_h))
    gprm = np.zeros((6, d_h))
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if cu is not None else None
    _run(lambda j0, j1: lib.oracle_backward(_dptr(P), _dptr(prm), B, T, d_h, cup, S, _dptr(H),
                                            _dptr(gH), j0, j1, _dptr(gP), _dptr(gprm)),
         d_h, threads)
    return gP, gprm


def decode_step(P, params, h=None) -> np.ndarray:
    """One T = 1 step per slot: h_out[s, j] = f(h[s, j], P[s]) (h None = zeros);
    P (slots, 3 d_h).  The sequential unroll taken one step at a time."""
    P = np.asarray(P, dtype=np.float64)
    slots, d_h = P.shape[0], P.shape[1] // 3
    h = np.zeros((slots, d_h)) if h is None else np.asarray(h, dtype=np.float64)
    prm = pack_params(params)
    out = np.empty((slots, d_h))
    for s in range(slots):
        for j in range(d_h):
            out[s, j] = cell(h[s, j], P[s, j], P[s, d_h + j], P[s, 2 * d_h + j], prm[:, j])[0]
    return out


def input_projection(x, W_x) -> np.ndarray:
    """P = x W_x^T in float64; x (..., d_in), W_x (3 d_h, d_in)."""
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W_x, dtype=np.float64)
    return x @ W.T


def columns(P, params, units):
    """Restricts a problem to the given hidden units (all three gates of each).

    Units are independent under a diagonal Jacobian, so the oracle can check a
    sample of units of a full-size run exactly."""
    P = np.asarray(P)
    d_h = P.shape[-1] // 3
    units = np.asarray(units, dtype=np.int64)
    idx = np.concatenate([units, d_h + units, 2 * d_h + units])
    prm = pack_params(params)[:, units]
    return P[..., idx], prm
