"""Host-side checks of the C ABI: the library loads, exports every entry point
the header declares, and its host logic (cu_seqlens rules, workspace sizes,
status strings, argument checks) behaves as documented.  No GPU needed."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import nonlinear_rnn_gb300 as nr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "nrnn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nrnn_\w+)\s*\(", src)))


def test_header_symbols_are_exported_and_bound():
    lib = nr.load()
    names = _declared()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(nr.EXPORTED) == names


def test_status_strings_and_version():
    lib = nr.load()
    assert lib.nrnn_version() >= 100
    for code in range(0, -8, -1):
        s = lib.nrnn_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.nrnn_status_string(-99).decode() == "unknown status"


def _validate(cu, N):
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    return nr.load().nrnn_validate_cu_seqlens(cu.ctypes.data_as(ctypes.c_void_p), cu.size - 1, N)


def test_validate_cu_seqlens_rules():
    assert _validate([0, 3, 3, 10], 10) == 0          # empty segment allowed
    assert _validate([0, 10], 10) == 0
    assert _validate([1, 3, 10], 10) == -2            # must start at 0
    assert _validate([0, 5, 4, 10], 10) == -2         # decreasing
    assert _validate([0, 3, 9], 10) == -2             # must end at N
    assert _validate([0], 0) == -2                    # at least one segment
    assert nr.load().nrnn_validate_cu_seqlens(None, 1, 1) == -1
    with pytest.raises(ValueError):
        nr.validate_cu_seqlens([0, 4, 2], 2)


def test_workspace_bytes():
    lib = nr.load()
    f = lib.nrnn_newton_workspace_bytes
    fused = f(8, 4096, 256, 0, 3, 2)
    per = f(8, 4096, 256, 0, 3, 1)
    # per-iteration keeps one extra H buffer (B*T*d_h*4 bytes)
    assert per - fused >= 8 * 4096 * 256 * 4
    assert f(8, 4096, 256, 0, 1, 1) < per               # K = 1 needs no H buffer
    assert f(8, 4096, 256, 0, 3, 0) == fused            # auto = fused
    assert f(8, 4096, 256, 0, 65, 2) == 0               # K above the limit
    assert f(8, 4096, 256, 5, 3, 2) == 0                # bad dtype
    assert fused % 256 == 0


def test_forward_rejects_bad_arguments_before_any_launch():
    lib = nr.load()
    fake = ctypes.c_void_p(256)   # never dereferenced: checks fail first
    res = ctypes.c_void_p(512)
    hout = ctypes.c_void_p(1 << 24)   # apart from preact
    args = dict(pre=fake, dtype=0, prm=fake, B=1, T=8, d=16, cu=None, S=0, K=3, fail=1.0, algo=0,
                H=hout, rd=res, rh=None, ws=fake, wsb=1 << 20, st=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.nrnn_newton_forward(a["pre"], a["dtype"], a["prm"], a["B"], a["T"], a["d"],
                                       a["cu"], a["S"], a["K"], a["fail"], a["algo"], a["H"],
                                       a["rd"], a["rh"], a["ws"], a["wsb"], a["st"])
    assert call(dtype=7) == -1
    assert call(d=12) == -3                       # d_h % 8 != 0
    assert call(B=1 << 20, T=1 << 20, d=64) == -3   # more than 2^31 tiles
    assert call(K=-1) == -1
    assert call(K=65) == -1
    assert call(algo=9) == -1
    assert call(B=2, cu=fake, S=2) == -2          # packs need B == 1
    assert call(H=ctypes.c_void_p(256 + 3 * 8 * 16 * 4 - 16)) == -1   # H_out overlaps preact
    assert call(wsb=16) == -7                     # workspace too small
    assert call(ws=ctypes.c_void_p(256 + 16)) == -7   # workspace misaligned
    assert call(pre=ctypes.c_void_p(260)) == -1   # preact misaligned
    assert call(rd=None) == -1


def test_decode_overlap_check_uses_each_buffer_size():
    # h_out (slots x d_h) ending right before preact (slots x 3 d_h) does not
    # overlap it; h_out inside preact does.  Fake pointers: the overlap check
    # runs before anything touches them (the GPU-less call then fails on CUDA).
    lib = nr.load()
    slots, d_h = 300, 40
    pre = 1 << 24
    h_before = pre - slots * d_h * 4
    if not torch.cuda.is_available():   # with a GPU this call would launch on fake pointers
        st = lib.nrnn_decode_step(ctypes.c_void_p(pre), 0, ctypes.c_void_p(256), slots, d_h, None,
                                  ctypes.c_void_p(h_before), None)
        assert st != -1
    st = lib.nrnn_decode_step(ctypes.c_void_p(pre), 0, ctypes.c_void_p(256), slots, d_h, None,
                              ctypes.c_void_p(pre + 64), None)
    assert st == -1


def test_projection_workspace_size_and_checks():
    """fp32 takes the low part of W_x (3 d_h x d_in fp32) in the caller's
    workspace; bf16 needs none.  Checks run before any launch."""
    lib = nr.load()
    assert lib.nrnn_input_projection_workspace_bytes(0, 512, 512) == 3 * 512 * 512 * 4
    assert lib.nrnn_input_projection_workspace_bytes(1, 512, 512) == 0
    assert lib.nrnn_input_projection_workspace_bytes(5, 512, 512) == 0
    fake = ctypes.c_void_p(256)
    need = 3 * 16 * 64 * 4

    def call(ws, wsb, dtype=0, rows=100):
        return lib.nrnn_input_projection(fake, fake, dtype, rows, 64, 16, ctypes.c_void_p(1 << 24),
                                         ws, wsb, None)
    assert call(None, 0) == -7                            # fp32 without a workspace
    assert call(ctypes.c_void_p(4096), need - 4) == -7    # too small
    assert call(ctypes.c_void_p(4096 + 16), need) == -7   # not 256-byte aligned
    assert call(None, 0, rows=0) == 0                     # nothing to do
    assert lib.nrnn_input_projection(fake, fake, 0, 100, 60, 16, fake, None, 0, None) == -3


def test_host_staging_sizes():
    """The x-input host forward stages each slot's x rows besides what the
    preactivation form stages, plus the projection's workspace (fp32)."""
    f32, bf16 = torch.float32, torch.bfloat16
    base = nr.host_staging_bytes(4, 1000, 64, f32, 3, tokens_per_block=1000)
    xs = nr.x_host_staging_bytes(4, 1000, 32, 64, f32, 3, tokens_per_block=1000)
    # three slots of 1000 x 32 fp32 rows, the low part of W_x (192 x 32 fp32)
    assert xs - base >= 3 * 1000 * 32 * 4 + 192 * 32 * 4
    xb = nr.x_host_staging_bytes(4, 1000, 32, 64, bf16, 3, tokens_per_block=1000)
    assert xb - nr.host_staging_bytes(4, 1000, 64, bf16, 3, tokens_per_block=1000) >= 3 * 1000 * 32 * 2
    assert nr.x_host_staging_bytes(4, 1000, 30, 64, f32, 3) == 0      # d_in % 8
    assert nr.x_host_staging_bytes(4, 1000, 0, 64, f32, 3) == 0
    assert nr.x_host_staging_bytes(4, 1000, 32, 60, f32, 3) == 0      # d_h % 8
    assert nr.x_host_staging_bytes(1, 10, 32, 64, f32, 3, cu_seqlens=[0, 4, 10]) > 0
    lib = nr.load()
    fake = ctypes.c_void_p(256)
    # d_in not positive / not a multiple of 8, before anything touches a pointer
    assert lib.nrnn_newton_forward_x_host(fake, fake, 0, fake, 1, 8, 0, 16, None, 0, 3, 1.0,
                                          fake, fake, fake, 1 << 20, 0, None) == -1
    assert lib.nrnn_newton_forward_x_host(fake, fake, 0, fake, 1, 8, 12, 16, None, 0, 3, 1.0,
                                          fake, fake, fake, 1 << 20, 0, None) == -3


def test_lookback_form_query_checks_its_arguments():
    lib = nr.load()
    assert lib.nrnn_debug_lookback_form(0, 10, 16, 0, 0) == -1      # B < 1
    assert lib.nrnn_debug_lookback_form(1, 10, 16, 5, 0) == -1      # dtype
    assert lib.nrnn_debug_lookback_form(1, 10, 16, 0, 7) == -1      # algo
    assert lib.nrnn_debug_lookback_form(1, 10, 16, 0, 2) in (0, 1)


def test_pack_workspace_and_plan_checks():
    """A pack of 2..4096 segments with num_segments <= chunks / 8 gets room for
    segment-aligned chunks (more look-back slots and the chunk plan); other
    packs need what the time-axis chunks need."""
    lib = nr.load()
    plain = lib.nrnn_newton_workspace_bytes(1, 4096, 64, 0, 3, 2)
    pack = lib.nrnn_newton_workspace_bytes_pack(4096, 64, 0, 3, 2, 8)      # 64 chunks, 8 segments
    # 8 more chunks per unit tile in the slots (3 iterations x 2 unit tiles x
    # 8 x 32 words) and the plan (1 + 64 + 8 entries of 16 bytes)
    assert pack >= plain + 3 * 2 * 8 * 32 * 8 + 73 * 16
    assert lib.nrnn_newton_workspace_bytes_pack(4096, 64, 0, 3, 2, 1) == plain   # one segment
    assert lib.nrnn_newton_workspace_bytes_pack(4096, 64, 0, 3, 2, 9) == plain   # 9 > 64 / 8
    assert lib.nrnn_newton_workspace_bytes_pack(4096, 64, 0, 3, 2, 0) == 0
    assert lib.nrnn_newton_workspace_bytes_pack(4096, 64, 0, 99, 2, 8) == 0      # K
    assert nr.workspace_bytes(1, 4096, 64, torch.float32, 3, "fused", num_segments=8) == pack
    fake = ctypes.c_void_p(256)
    assert lib.nrnn_debug_pack_plan(fake, 1, 4096, 0, fake, None) == -1
    assert lib.nrnn_debug_pack_plan(fake, 9, 4096, 1, fake, None) == -1
    assert lib.nrnn_debug_pack_plan(None, 8, 4096, 0, fake, None) == -1


def test_host_pipeline_default_blocks():
    """By default the host-buffer forward cuts the problem into about 16
    blocks: the three staging slots then hold one block each, so the staging
    area is about 3/16 of what one block of all rows takes (plus workspaces)."""
    f32 = torch.float32
    B, T, d_h = 16, 4096, 256
    one = nr.host_staging_bytes(B, T, d_h, f32, 3, tokens_per_block=B * T)
    default = nr.host_staging_bytes(B, T, d_h, f32, 3)
    row = nr.host_staging_bytes(B, T, d_h, f32, 3, tokens_per_block=T)
    assert default == row                     # 16 blocks of one row each
    assert default < one / 4
    # the x-input form adds the x rows of each slot and the projection's workspace
    xs = nr.x_host_staging_bytes(B, T, 128, d_h, f32, 3)
    assert xs >= default + 3 * T * 128 * 4 + 3 * d_h * 128 * 4
