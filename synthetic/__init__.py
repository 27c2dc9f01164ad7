"""Seeded synthetic inputs for the diagonal-mix GRU Newton forward.

This module is shared by the oracle side (``oracle/``, the tests) and the CUDA
side (the package, ``bench.py``).  It holds the workload shapes and the random
draws only: no cell, no projection, no scan.  Every number the method computes
lives elsewhere.

Generator.  SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based generator: the i-th
draw of stream ``s`` under seed ``k`` mixes ``key(k, s) + (i + 1) * GAMMA``
with the SplitMix64 finaliser.  A uniform in [0, 1) takes the top 53 bits.
Normals use the Box-Muller transform (Box & Muller 1958) on consecutive
uniform pairs.  The whole sequence is defined by integer arithmetic modulo
2**64 and by IEEE double ``log``/``sqrt``/``cos``/``sin``, so it does not
depend on the torch or numpy version.

Workloads.  The five diagonal-GRU workloads (cell and init as stated for the
ParaGRU(mix='diag') benches of pararnn-torch): x ~ N(0, 1); W_x ~ U(+-1/sqrt(d_in));
diagonal recurrent weights a_z, a_r, a_c ~ U(+-1); biases 0; h0 = 0.  The
ragged pack draws S integer segment lengths uniform in [lo, hi], rescales them
to sum to N (floor, then the remainder one token each to segments 0, 1, ...)
and returns ``cu_seqlens`` as the exclusive prefix sum (int32, length S + 1).
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream identifiers (one independent stream per drawn quantity)
STREAM_X = 1
STREAM_WX = 2
STREAM_AZ = 3
STREAM_AR = 4
STREAM_AC = 5
STREAM_SEGLEN = 6
STREAM_PREACT = 7   # direct preactivation draws for kernel-only tests

_BLOCK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wraps modulo 2**64)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    base = np.array([(seed * 0x10001 + stream * 0x9E37) & 0xFFFFFFFFFFFFFFFF],
                    dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base)[0]


def uniform64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Draws ``start .. start+n-1`` of a stream as float64 in [0, 1)."""
    key = _key(seed, stream)
    out = np.empty(n, dtype=np.float64)
    with np.errstate(over="ignore"):
        for o in range(0, n, _BLOCK):
            m = min(_BLOCK, n - o)
            ctr = np.arange(start + o + 1, start + o + m + 1, dtype=np.uint64)
            z = _mix(key + ctr * GAMMA)
            out[o:o + m] = (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return out


def _blocks(fn, n_blocks: int) -> None:
    """Runs fn(i) for every block index; blocks write disjoint slices, and numpy
    releases the GIL inside its array operations, so large draws use threads."""
    if n_blocks <= 1:
        for i in range(n_blocks):
            fn(i)
        return
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(min(n_blocks, os.cpu_count() or 1)) as ex:
        list(ex.map(fn, range(n_blocks)))


def normal64(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller on uniform pairs), float64."""
    out = np.empty(n, dtype=np.float64)
    pairs = (n + 1) // 2
    blk = _BLOCK // 2

    def one(i):
        o = i * blk
        m = min(blk, pairs - o)
        u = uniform64(seed, stream, 2 * m, start=2 * o)
        u1 = 1.0 - u[0::2]            # (0, 1]: log is finite
        u2 = u[1::2]
        rad = np.sqrt(-2.0 * np.log(u1))
        ang = 2.0 * math.pi * u2
        seg = np.empty(2 * m, dtype=np.float64)
        seg[0::2] = rad * np.cos(ang)
        seg[1::2] = rad * np.sin(ang)
        lo = 2 * o
        hi = min(n, lo + 2 * m)
        out[lo:hi] = seg[: hi - lo]

    _blocks(one, -(-pairs // blk))
    return out


def uniform_pm(seed: int, stream: int, n: int, half_width: float) -> np.ndarray:
    """n draws of U(-half_width, +half_width), float64."""
    return (2.0 * uniform64(seed, stream, n) - 1.0) * half_width


def segment_lengths(seed: int, S: int, N: int, lo: int, hi: int) -> np.ndarray:
    """S integer lengths, uniform in [lo, hi], rescaled to sum to N."""
    u = uniform64(seed, STREAM_SEGLEN, S)
    raw = lo + np.floor(u * (hi - lo + 1)).astype(np.int64)
    raw = np.minimum(raw, hi)
    scaled = (raw * N) // int(raw.sum())
    rem = N - int(scaled.sum())
    for i in range(rem):
        scaled[i % S] += 1
    return scaled


def cu_from_lengths(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    d_in: int
    d_h: int
    K: int
    dtype: str                      # storage type of x, W_x, preact and H: "f32" | "bf16"
    segments: int = 0               # > 0: ragged pack of that many segments in one row
    seg_lo: int = 0
    seg_hi: int = 0
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = [
    Workload("diag-gru f32 B1 T1024 d_in8 d_h16 K3", 1, 1024, 8, 16, 3, "f32", seed=0),
    Workload("diag-gru f32 B8 T4096 d_in256 d_h256 K3", 8, 4096, 256, 256, 3, "f32", seed=1),
    Workload("diag-gru f32 B4 T131072 d_in64 d_h64 K2", 4, 131072, 64, 64, 2, "f32", seed=2),
    Workload("diag-gru bf16 B16 T16384 d_in1024 d_h1024 K3", 16, 16384, 1024, 1024, 3, "bf16", seed=3),
    Workload("diag-gru f32 ragged N262144 S64 d512 K3", 1, 262144, 512, 512, 3, "f32",
             segments=64, seg_lo=256, seg_hi=8192, seed=4),
]


def small_workload(B=2, T=300, d_in=8, d_h=40, K=3, dtype="f32", seed=11,
                   segments=0, seg_lo=1, seg_hi=64) -> Workload:
    """A test-sized workload with the same distributions."""
    return Workload(f"small B{B} T{T} d{d_h}", B, T, d_in, d_h, K, dtype,
                    segments=segments, seg_lo=seg_lo, seg_hi=seg_hi, seed=seed)


def _round_bf16_flat(a: np.ndarray, r: np.ndarray) -> None:
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r[:] = (((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)).astype(np.uint32)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = np.uint32(0x7FC00000)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even), returned as float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    flat = a.reshape(-1)
    r = np.empty(flat.shape, dtype=np.uint32)
    _blocks(lambda i: _round_bf16_flat(flat[i * _BLOCK:(i + 1) * _BLOCK],
                                       r[i * _BLOCK:(i + 1) * _BLOCK]),
            -(-flat.size // _BLOCK))
    return r.view(np.float32).reshape(a.shape)


def make_params(w: Workload) -> dict:
    """Diagonal recurrent weights U(+-1) and zero biases, float32 (d_h each)."""
    s, d = w.seed, w.d_h
    return {
        "a_z": uniform_pm(s, STREAM_AZ, d, 1.0).astype(np.float32),
        "a_r": uniform_pm(s, STREAM_AR, d, 1.0).astype(np.float32),
        "a_c": uniform_pm(s, STREAM_AC, d, 1.0).astype(np.float32),
        "b_z": np.zeros(d, np.float32),
        "b_r": np.zeros(d, np.float32),
        "b_c": np.zeros(d, np.float32),
    }


def make_inputs(w: Workload, with_x: bool = True) -> dict:
    """x (B, T, d_in), W_x (3 d_h, d_in), params and cu_seqlens for a workload.

    Arrays are float32; for ``dtype == "bf16"`` x and W_x are already rounded to
    bfloat16 values (still held as float32)."""
    s = w.seed
    out = {"params": make_params(w)}
    W = uniform_pm(s, STREAM_WX, 3 * w.d_h * w.d_in, 1.0 / math.sqrt(w.d_in))
    W = W.astype(np.float32).reshape(3 * w.d_h, w.d_in)
    if with_x:
        n = w.B * w.T * w.d_in
        x64 = normal64(s, STREAM_X, n)
        x = np.empty(n, dtype=np.float32)
        _blocks(lambda i: np.copyto(x[i * _BLOCK:(i + 1) * _BLOCK], x64[i * _BLOCK:(i + 1) * _BLOCK],
                                    casting="same_kind"), -(-n // _BLOCK))
        del x64
        x = x.reshape(w.B, w.T, w.d_in)
    else:
        x = None
    if w.dtype == "bf16":
        W = round_bf16(W)
        if x is not None:
            x = round_bf16(x)
    out["W_x"] = W
    out["x"] = x
    if w.segments > 0:
        assert w.B == 1
        lens = segment_lengths(s, w.segments, w.T, w.seg_lo, w.seg_hi)
        out["cu_seqlens"] = cu_from_lengths(lens)
    else:
        out["cu_seqlens"] = None
    return out


def direct_preact(w: Workload, scale: float = 1.0 / math.sqrt(3.0)) -> np.ndarray:
    """Preactivations drawn directly as N(0, scale**2), shape (B, T, 3 d_h), float32.

    x ~ N(0,1) against W_x ~ U(+-1/sqrt(d_in)) gives preactivations of variance
    1/3; this draws values of that distribution without the projection, for
    kernel-level tests whose input is the preactivation buffer itself."""
    n = w.B * w.T * 3 * w.d_h
    p = (normal64(w.seed, STREAM_PREACT, n) * scale).astype(np.float32)
    p = p.reshape(w.B, w.T, 3 * w.d_h)
    if w.dtype == "bf16":
        p = round_bf16(p)
    return p


# ------------------------------------------------------------------------
# Preactivations drawn directly, reproducible bit for bit on any device.
#
# For kernel-level runs at full size the preactivation buffer itself is the
# input.  P ~ U(-1, 1) has the variance (1/3) of x W_x^T with x ~ N(0, 1) and
# W_x ~ U(+-1/sqrt(d_in)).  The value at flat index i of the (B, T, 3 d_h)
# buffer is 2 u_i - 1 with u_i the i-th uniform of stream STREAM_PREACT; the
# computation is integer mixing, an exact scaling and one rounding to float32,
# so torch on the GPU and numpy on the host produce identical values.  The
# host side can therefore regenerate any sampled columns without the rest.
# ------------------------------------------------------------------------
def _as_i64(v: int) -> int:
    v &= 0xFFFFFFFFFFFFFFFF
    return v - (1 << 64) if v >= (1 << 63) else v


def _torch_mix(z):
    import torch
    m30 = (1 << 34) - 1
    m27 = (1 << 37) - 1
    m31 = (1 << 33) - 1
    z = (z ^ ((z >> 30) & m30)) * _as_i64(0xBF58476D1CE4E5B9)
    z = (z ^ ((z >> 27) & m27)) * _as_i64(0x94D049BB133111EB)
    return z ^ ((z >> 31) & m31)


def preact_uniform_torch(w: Workload, device="cuda", dtype=None):
    """Full (B, T, 3 d_h) preactivation buffer of U(-1, 1) draws as a torch tensor."""
    import torch
    n = w.B * w.T * 3 * w.d_h
    key = _as_i64(int(_key(w.seed, STREAM_PREACT)))
    out = torch.empty(n, dtype=torch.float32, device=device)
    blk = 1 << 26
    for o in range(0, n, blk):
        m = min(blk, n - o)
        ctr = torch.arange(o + 1, o + m + 1, dtype=torch.int64, device=device)
        z = _torch_mix(ctr * _as_i64(int(GAMMA)) + key)
        u = ((z >> 11) & ((1 << 53) - 1)).to(torch.float64) * (1.0 / 9007199254740992.0)
        out[o:o + m] = (2.0 * u - 1.0).to(torch.float32)
    out = out.reshape(w.B, w.T, 3 * w.d_h)
    if dtype is None:
        dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return out.to(dtype)


def preact_uniform_at(w: Workload, flat_index: np.ndarray) -> np.ndarray:
    """Values of the same buffer at the given flat indices (numpy float32; for a
    bf16 workload, rounded to bfloat16 values)."""
    idx = np.asarray(flat_index, dtype=np.uint64)
    key = _key(w.seed, STREAM_PREACT)
    with np.errstate(over="ignore"):
        z = _mix(key + (idx + np.uint64(1)) * GAMMA)
    u = (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    p = (2.0 * u - 1.0).astype(np.float32)
    return round_bf16(p) if w.dtype == "bf16" else p


def preact_uniform_columns(w: Workload, units, rows=None) -> np.ndarray:
    """(len(rows), T, 3 len(units)) slice of the buffer: all three gates of the
    given hidden units, gate-major like the full buffer."""
    units = np.asarray(units, dtype=np.int64)
    rows = np.arange(w.B) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.concatenate([units, w.d_h + units, 2 * w.d_h + units])
    t = np.arange(w.T, dtype=np.int64)
    flat = ((rows[:, None, None] * w.T + t[None, :, None]) * (3 * w.d_h) + cols[None, None, :])
    return preact_uniform_at(w, flat.reshape(-1)).reshape(len(rows), w.T, len(cols))
