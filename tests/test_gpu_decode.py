"""Decode steps on the GPU against the oracle: one step, carried state over
many steps (equals the unroll), and the projection-fused variant."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dtype)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_matches_oracle_and_carries_state(dtype):
    import nonlinear_rnn_gb300 as nr
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w = syn.small_workload(B=37, T=50, d_h=20, dtype=dtype, seed=61)   # 37 slots
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    Pd = dev(P, tdt)
    h = nr.decode_step(prm, preact=Pd[:, 0])
    np.testing.assert_allclose(host(h), oracle.decode_step(P[:, 0], prm), atol=1e-6 if dtype == "f32" else 4e-3)
    Hs = oracle.sequential(P, prm)
    for t in range(1, w.T):
        h = nr.decode_step(prm, h=h, preact=Pd[:, t], out=h)          # in place
    tol = 1e-5 if dtype == "f32" else 3e-2                            # bf16 carry rounds every step
    assert np.max(np.abs(host(h) - Hs[:, -1])) <= tol


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_h, offset, slots", [(6, 0, 333), (16, 0, 333), (40, 0, 333), (16, 1, 333),
                                                (256, 0, 5001)])
def test_decode_step_vector_and_scalar_paths(dtype, d_h, offset, slots):
    # d_h a multiple of 4 with aligned buffers takes the vector kernel (each
    # thread walks the slots two per pass: 5001 slots of 256 units take
    # several passes and end on a single slot); d_h = 6 or an output one
    # element off alignment takes the scalar one; both against the oracle,
    # h_in given
    import nonlinear_rnn_gb300 as nr
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w = syn.small_workload(B=slots, T=1, d_h=d_h, dtype=dtype, seed=64 + d_h)
    P = syn.direct_preact(w)[:, 0]
    prm = syn.make_params(w)
    rng = np.random.default_rng(65 + d_h)
    h0 = rng.uniform(-0.9, 0.9, size=(slots, d_h)).astype(np.float32)
    if dtype == "bf16":
        P, h0 = syn.round_bf16(P), syn.round_bf16(h0)
    buf = torch.full((slots * d_h + offset,), float("nan"), dtype=tdt, device="cuda")
    out = buf[offset:].view(slots, d_h)
    h = nr.decode_step(prm, h=dev(h0, tdt), preact=dev(P, tdt), out=out)
    assert h.data_ptr() == out.data_ptr()
    ref = oracle.decode_step(P, prm, h0)
    assert np.max(np.abs(host(h) - ref)) <= (1e-6 if dtype == "f32" else 4e-3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_with_fused_projection(dtype):
    import nonlinear_rnn_gb300 as nr
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    slots, d_in, d_h = 13, 72, 24
    rng = np.random.default_rng(62)
    x = rng.normal(size=(slots, d_in)).astype(np.float32)
    W = (rng.uniform(-1, 1, size=(3 * d_h, d_in)) / math.sqrt(d_in)).astype(np.float32)
    h0 = rng.uniform(-0.5, 0.5, size=(slots, d_h)).astype(np.float32)
    if dtype == "bf16":
        x, W, h0 = syn.round_bf16(x), syn.round_bf16(W), syn.round_bf16(h0)
    prm = syn.make_params(syn.small_workload(d_h=d_h, seed=63))
    P = oracle.input_projection(x, W)
    if dtype == "bf16":
        P = syn.round_bf16(P.astype(np.float32))
    ref = oracle.decode_step(P, prm, h0)
    h = nr.decode_step(prm, h=dev(h0, tdt), x=dev(x, tdt), W_x=dev(W, tdt))
    assert np.max(np.abs(host(h) - ref)) <= (2e-6 if dtype == "f32" else 1.6e-2)


@pytest.mark.parametrize("slots,d_in,d_h", [(40, 72, 24), (300, 512, 48)])
def test_decode_step_with_projection_in_place(slots, d_in, d_h):
    # bf16, out = h: the carried state is overwritten by the step (one tile of
    # 8-unit CTAs; the GEMM form, whose epilogue reads and writes each 8-unit
    # group of a slot in the same thread)
    import nonlinear_rnn_gb300 as nr
    rng = np.random.default_rng(slots + 3 * d_h)
    x = syn.round_bf16(rng.normal(size=(slots, d_in)).astype(np.float32))
    W = syn.round_bf16((rng.uniform(-1, 1, size=(3 * d_h, d_in)) / math.sqrt(d_in)).astype(np.float32))
    h0 = syn.round_bf16(rng.uniform(-0.5, 0.5, size=(slots, d_h)).astype(np.float32))
    prm = syn.make_params(syn.small_workload(d_h=d_h, seed=66))
    P = syn.round_bf16(oracle.input_projection(x, W).astype(np.float32))
    ref = oracle.decode_step(P, prm, h0)
    hd = dev(h0, torch.bfloat16)
    h = nr.decode_step(prm, h=hd, x=dev(x, torch.bfloat16), W_x=dev(W, torch.bfloat16), out=hd)
    assert h.data_ptr() == hd.data_ptr()
    assert np.max(np.abs(host(h) - ref)) <= 1.6e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("slots,d_in,d_h", [(64, 2048, 16), (300, 136, 40), (8, 8, 8), (300, 512, 48)])
def test_decode_step_with_projection_at_other_sizes(dtype, slots, d_in, d_h):
    # 64 slots x d_in 2048: the fused kernel reading x from global memory (it
    # does not fit the staging buffer); 300 slots: the binding's
    # projection-then-step path (fp32, or bf16 with d_in 136), or for bf16
    # with d_in 512 the C-ABI call's GEMM form; 8 x 8: the smallest shape
    import nonlinear_rnn_gb300 as nr
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    rng = np.random.default_rng(slots + d_in)
    x = rng.normal(size=(slots, d_in)).astype(np.float32)
    W = (rng.uniform(-1, 1, size=(3 * d_h, d_in)) / math.sqrt(d_in)).astype(np.float32)
    h0 = rng.uniform(-0.5, 0.5, size=(slots, d_h)).astype(np.float32)
    if dtype == "bf16":
        x, W, h0 = syn.round_bf16(x), syn.round_bf16(W), syn.round_bf16(h0)
    prm = syn.make_params(syn.small_workload(d_h=d_h, seed=64))
    P = oracle.input_projection(x, W)
    if dtype == "bf16":
        P = syn.round_bf16(P.astype(np.float32))
    ref = oracle.decode_step(P, prm, h0)
    h = nr.decode_step(prm, h=dev(h0, tdt), x=dev(x, tdt), W_x=dev(W, tdt))
    assert np.max(np.abs(host(h) - ref)) <= (1e-5 if dtype == "f32" else 1.6e-2)


@pytest.mark.parametrize("slots,d_in,d_h,zero_h", [(200, 200, 96, False), (512, 136, 512, False),
                                                   (70, 64, 40, True), (64, 1024, 1024, False),
                                                   (33, 296, 72, False), (64, 256, 40, True),
                                                   (64, 72, 96, False), (200, 520, 96, False),
                                                   (129, 512, 200, False), (1000, 1024, 1024, False),
                                                   (300, 512, 8, False), (70, 640, 40, True)])
def test_decode_step_x_bf16_tensor_core_path_through_the_c_abi(slots, d_in, d_h, zero_h):
    """nrnn_decode_step_x for bf16 runs the projection on the tensor cores for
    any slot count.  Above one 64-slot tile with d_in >= 512 it is a GEMM of
    128-slot by 64-unit tiles (z, r and c rows of W_x) on persistent CTAs with
    the step in the epilogue: 200 x 520 -> 96 (a K tail of 8), 129 x 512 -> 200
    (ragged slot and unit tiles), 1000 x 1024 -> 1024 (several tiles per CTA,
    both TMEM accumulators in turn), 300 x 512 -> 8 (one 8-unit group of a
    64-unit tile), 70 x 640 -> 40 from the zero state.  Otherwise 64 slots by 8
    or 32 units per CTA: 200 x 200 -> 96 and 70 x 64 -> 40 (8-unit tiles),
    512 x 136 -> 512 (32-unit tiles), 64 x 72 -> 96; ragged tiles and a K tail
    are zero-filled by TMA.  One tile of at most 64 slots with at least four
    64-wide slices of d_in takes the split-K cluster form (64 x 1024 -> 1024;
    33 slots with a 296-wide d_in split 1 / 1 / 1 / 2 slices and a ragged unit
    tile; 64 x 256 -> 40 from the zero state)."""
    import ctypes
    import nonlinear_rnn_gb300 as nr
    lib = nr.load()
    rng = np.random.default_rng(slots * 7 + d_h)
    x = syn.round_bf16(rng.normal(size=(slots, d_in)).astype(np.float32))
    W = syn.round_bf16((rng.uniform(-1, 1, size=(3 * d_h, d_in)) / math.sqrt(d_in)).astype(np.float32))
    h0 = np.zeros((slots, d_h), np.float32) if zero_h else \
        syn.round_bf16(rng.uniform(-0.5, 0.5, size=(slots, d_h)).astype(np.float32))
    prm = syn.make_params(syn.small_workload(d_h=d_h, seed=65))
    P = syn.round_bf16(oracle.input_projection(x, W).astype(np.float32))
    ref = oracle.decode_step(P, prm, None if zero_h else h0)
    xd, Wd = dev(x, torch.bfloat16), dev(W, torch.bfloat16)
    hd = dev(h0, torch.bfloat16)
    out = torch.full((slots, d_h), float("nan"), dtype=torch.bfloat16, device="cuda")
    pd = nr.params_tensor(prm, d_h, "cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())   # noqa: E731
    st = lib.nrnn_decode_step_x(p(xd), p(Wd), 1, p(pd), slots, d_in, d_h,
                                None if zero_h else p(hd), p(out),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    assert np.max(np.abs(host(out) - ref)) <= 1.6e-2


@pytest.mark.parametrize("i", range(8))
def test_decode_step_x_bf16_random_shapes(i):
    """Seeded random slot counts, d_in and d_h through nrnn_decode_step_x
    (bf16): both tensor-core forms, ragged slot and unit tiles, K tails, the
    zero state and in-place updates, against the oracle on the float64
    projection rounded to bf16."""
    import ctypes
    import nonlinear_rnn_gb300 as nr
    rng = np.random.default_rng(9100 + i)
    slots = int(rng.integers(1, 1500))
    d_in = int(8 * rng.integers(1, 160))      # 8 .. 1272
    d_h = int(8 * rng.integers(1, 40))        # 8 .. 312
    zero_h, in_place = bool(i % 3 == 0), bool(i % 2 == 1)
    lib = nr.load()
    x = syn.round_bf16(rng.normal(size=(slots, d_in)).astype(np.float32))
    W = syn.round_bf16((rng.uniform(-1, 1, size=(3 * d_h, d_in)) / math.sqrt(d_in)).astype(np.float32))
    h0 = np.zeros((slots, d_h), np.float32) if zero_h else \
        syn.round_bf16(rng.uniform(-0.5, 0.5, size=(slots, d_h)).astype(np.float32))
    prm = syn.make_params(syn.small_workload(d_h=d_h, seed=9200 + i))
    P = syn.round_bf16(oracle.input_projection(x, W).astype(np.float32))
    ref = oracle.decode_step(P, prm, None if zero_h else h0)
    xd, Wd, hd = dev(x, torch.bfloat16), dev(W, torch.bfloat16), dev(h0, torch.bfloat16)
    out = hd if in_place else torch.full((slots, d_h), float("nan"), dtype=torch.bfloat16, device="cuda")
    pd = nr.params_tensor(prm, d_h, "cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())   # noqa: E731
    st = lib.nrnn_decode_step_x(p(xd), p(Wd), 1, p(pd), slots, d_in, d_h,
                                None if zero_h else p(hd), p(out),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, (slots, d_in, d_h)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any(), (slots, d_in, d_h)
    assert np.max(np.abs(host(out) - ref)) <= 1.6e-2, (slots, d_in, d_h)
