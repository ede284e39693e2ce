"""The C-ABI library builds, loads and exports every entry point of include/kda.h.

No compute call is made here (no GPU needed): only symbol lookups and the pure
host arithmetic entry points.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from kda_gated_delta_02_gb300 import build
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_three_calls():
    fns = header_functions()
    for name in ("kda_chunk_fwd", "kda_segment_compose", "kda_decode_verify_replay"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in include/kda.h but not exported"


def test_status_strings_and_version(lib):
    lib.kda_status_string.restype = ctypes.c_char_p
    assert lib.kda_status_string(0) == b"ok"
    for code in (-1, -2, -3, -4, -5):
        assert lib.kda_status_string(code) not in (b"ok", b"unknown status")
    assert lib.kda_status_string(12345) == b"unknown status"
    assert lib.kda_version() >= 100


def test_cp_plan_and_workspace_arithmetic(lib):
    lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_size_t
    # CP off: no workspace
    assert lib.kda_chunk_fwd_workspace_size(1, 32768, 96, 128, 128, 0, 0) == 0
    assert lib.kda_chunk_fwd_plan(1, 32768, 96, 128, 128, 0, 0) == 0
    # many heads: auto keeps one pass per (sequence, head)
    assert lib.kda_chunk_fwd_plan(1, 32768, 96, 128, 128, -1, 0) == 0
    # few heads, long sequence: auto turns CP on with a 64-multiple segment
    seg = lib.kda_chunk_fwd_plan(1, 1 << 20, 12, 128, 128, -1, 0)
    assert seg > 0 and seg % 64 == 0
    # explicit segment length: M, N and S_in for T/seg + N segments at least
    ws = lib.kda_chunk_fwd_workspace_size(1, 1 << 20, 12, 128, 128, 1, 32768)
    P = (1 << 20) // 32768 + 1
    assert ws >= 3 * P * 12 * 128 * 128 * 4


def test_invalid_arguments_rejected_before_launch(lib):
    P = ctypes.c_void_p
    f = lib.kda_chunk_fwd
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, P, P] + [ctypes.c_int] * 5 + [P, P, P, ctypes.c_float, ctypes.c_float] + \
        [ctypes.c_int] * 3 + [P, ctypes.c_size_t, P, P]
    buf = ctypes.create_string_buffer(64)
    aligned = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    misaligned = ctypes.c_void_p(aligned.value + 4)
    # unsupported head size
    assert f(aligned, aligned, aligned, aligned, aligned, aligned, 1, 64, 2, 96, 128, None, None, aligned,
             1.0, -5.0, 0, 0, 0, None, 0, None, None) == -2
    # no cu_seqlens
    assert f(aligned, aligned, aligned, aligned, aligned, None, 1, 64, 2, 128, 128, None, None, aligned,
             1.0, -5.0, 0, 0, 0, None, 0, None, None) == -1
    # misaligned q
    assert f(misaligned, aligned, aligned, aligned, aligned, aligned, 1, 64, 2, 128, 128, None, None, aligned,
             1.0, -5.0, 0, 0, 0, None, 0, None, None) == -3
    # CP on without workspace
    assert f(aligned, aligned, aligned, aligned, aligned, aligned, 1, 1 << 16, 2, 128, 128, None, None, aligned,
             1.0, -5.0, 0, 1, 4096, None, 0, None, None) == -4
    # segment length not a multiple of 64
    assert f(aligned, aligned, aligned, aligned, aligned, aligned, 1, 1 << 16, 2, 128, 128, None, None, aligned,
             1.0, -5.0, 0, 1, 100, None, 0, None, None) == -1
    v = lib.kda_decode_verify_replay
    v.restype = ctypes.c_int
    v.argtypes = [P] * 12 + [ctypes.c_int] * 6 + [ctypes.c_float] * 4 + [ctypes.c_int, P, P]
    args = [aligned] * 12
    # draft window above 7 does not fit the 16-token tile
    assert v(*args, 4, 2, 128, 128, 4, 8, 1.0, -5.0, 1e-6, 1e-6, 1, None, None) == -1
    # dk != dv is not supported by the verify kernel
    assert v(*args, 4, 2, 128, 64, 4, 7, 1.0, -5.0, 1e-6, 1e-6, 1, None, None) == -2
    # conv width above 4
    assert v(*args, 4, 2, 128, 128, 5, 7, 1.0, -5.0, 1e-6, 1e-6, 1, None, None) == -1


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    import kda_gated_delta_02_gb300 as kda
    x = torch.zeros(64, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(kda.KDAError):
        kda.chunk_fwd(x, x, x, x.float(), torch.zeros(64, 2), torch.tensor([0, 64], dtype=torch.int32))


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("N,T,H,cp,seg", [(1, 32768, 96, 0, 0), (16, 68775, 96, 0, 0), (1, 1 << 20, 12, 1, 32768),
                                          (3, 1771, 4, 0, 0), (1, 1 << 21, 96, 0, 0)])
def test_prep_workspace_arithmetic(lib, N, T, H, cp, seg):
    """The two-kernel area after the CP scratch: slot list (8 B per slot,
    floor(T/64) + units slots), one item counter per slot, two carry states
    2 x H x 128 x 128 f32, and the operand blobs (66,048 B per slot and head):
    all slots in one piece for a context-parallel call or few slots, else two
    buffers of a quarter of the slots (pipelined pieces), the blobs capped at
    16 GiB."""
    from parity import split_layout, split_wanted_room
    lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_size_t
    lib.kda_chunk_fwd_prep_workspace_size.restype = ctypes.c_size_t
    base = lib.kda_chunk_fwd_workspace_size(N, T, H, 128, 128, cp, seg)
    got = lib.kda_chunk_fwd_prep_workspace_size(N, T, H, 128, 128, cp, seg)
    plan = lib.kda_chunk_fwd_plan(N, T, H, 128, 128, cp, seg)
    units = (T // plan + N) if plan else N
    room = split_wanted_room(T, H, units, plan != 0)
    piece, nbuf, pieces, area = split_layout(T, H, units, room, plan != 0)
    assert got == _align256(base) + area
    nslots = T // 64 + units
    if plan == 0 and nslots >= 64 and units * H < 152:
        assert nbuf == 2 and pieces >= 4
    else:
        assert nbuf * piece * H * 66048 <= (16384 << 20)
    # other shapes keep the one-kernel workspace
    assert lib.kda_chunk_fwd_prep_workspace_size(N, T, H, 64, 64, cp, seg) == \
        lib.kda_chunk_fwd_workspace_size(N, T, H, 64, 64, cp, seg)


def test_kernel_timing_without_launches(lib):
    """Start / stop with nothing launched: no CUDA call, zero counts."""
    n = 8
    launches = (ctypes.c_int * n)(*([7] * n))
    total = (ctypes.c_float * n)(*([7.0] * n))
    assert lib.kda_kernel_timing_start() == 0
    assert lib.kda_kernel_timing_stop(launches, total, n) == 0
    assert list(launches) == [0] * n and list(total) == [0.0] * n
    assert lib.kda_kernel_timing_stop(None, None, 2) != 0  # outputs required


def _bwd_tc_bytes(N, T, H):
    """The tensor-core backward's workspace (d = 128, bf16): the slot list, the
    item counters and two carry states per head, then per (slot, head) the operand blob (66,048 B), T and M^T
    (f32, 32 KB), the walk's S^T and U^T tiles (32 + 16 KB) and the reverse
    walk's dS'^T and dU'^T tiles (32 + 16 KB), each part 256-byte aligned."""
    slots = T // 64 + N
    sh = slots * H
    carry = _align256(2 * H * 128 * 128 * 4)  # two states per head for a sequence cut between pieces
    return (_align256(slots * 8) + 256 + carry + _align256(sh * 66048) + _align256(sh * 32768) +
            _align256(sh * 32768) + _align256(sh * 16384) + _align256(sh * 32768) + _align256(sh * 16384))


def test_backward_workspace_arithmetic(lib):
    """CUDA-core form: chunk checkpoints (floor(T/64) + N slots) and 64 states
    per (sequence, head) in flight, d x d fp32 each, two buffers of 64 x (3d +
    1) fp32 column partials per CTA (d/32 CTAs per unit), then w = v - p of
    every token (T x H x d fp32).  At d = 128 the size is the larger of that
    and the tensor-core form's (bf16 inputs take that form); 0 for
    unsupported shapes."""
    lib.kda_chunk_bwd_workspace_size.restype = ctypes.c_size_t
    N, T, H = 3, 1000, 4
    for d in (128, 64):
        dd = d * d * 4
        parts = lambda units: units * (d // 32) * 2 * 64 * (3 * d + 1) * 4
        wb = lambda h: _align256(T * h * d * 4)  # w = v - p of every token
        want = _align256((T // 64 + N) * H * dd) + _align256(N * H * 64 * dd) + _align256(parts(N * H)) + wb(H)
        if d == 128:
            want = max(want, _bwd_tc_bytes(N, T, H))
        assert lib.kda_chunk_bwd_workspace_size(N, T, H, d, d) == want
        # many units: scratch and partials stop growing at 160 units in flight
        N2, H2 = 100, 96
        want2 = (_align256((T // 64 + N2) * H2 * dd) + _align256(160 * 64 * dd) + _align256(parts(160)) +
                 wb(H2))
        if d == 128:
            want2 = max(want2, _bwd_tc_bytes(N2, T, H2))
        assert lib.kda_chunk_bwd_workspace_size(N2, T, H2, d, d) == want2
    d = 128
    assert lib.kda_chunk_bwd_workspace_size(N, T, H, 128, 64) == 0
    assert lib.kda_chunk_bwd_workspace_size(0, T, H, d, d) == 0


@pytest.mark.parametrize("N,T,H,cp,seg", [(1, 1 << 20, 12, -1, 0), (1, 1 << 20, 12, 1, 32768), (3, 5000, 2, 1, 1024),
                                          (1, 32768, 96, -1, 0), (2, 3000, 4, 0, 0), (1, 70000, 2, 1, 0)])
def test_cp_backward_workspace_arithmetic(lib, N, T, H, cp, seg):
    """The context-parallel backward's workspace: the CP prefill's scratch,
    the tensor-core backward's layout over the P_max = floor(T / segment) + N
    segment slots, then r and the segment-end gradients (P_max x H x 128 x 128
    f32 each), every part 256-byte aligned; the sequence form's size when the
    call is not cut (cp off, or automatic and declined), and never less."""
    lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_size_t
    lib.kda_chunk_bwd_workspace_size.restype = ctypes.c_size_t
    lib.kda_chunk_bwd_cp_workspace_size.restype = ctypes.c_size_t
    base = lib.kda_chunk_bwd_workspace_size(N, T, H, 128, 128)
    got = lib.kda_chunk_bwd_cp_workspace_size(N, T, H, 128, 128, cp, seg)
    plan = lib.kda_chunk_fwd_plan(N, T, H, 128, 128, cp, seg)
    if cp == 0 or plan == 0:
        assert got == base
        return
    assert plan % 64 == 0 and (seg == 0 or plan == seg)
    pm = T // plan + N
    cp_total = lib.kda_chunk_fwd_workspace_size(N, T, H, 128, 128, cp, seg)
    per_seg = _align256(pm * H * 128 * 128 * 4)
    want = _align256(cp_total) + _align256(_bwd_tc_bytes(pm, T, H)) + 2 * per_seg
    assert got == max(base, want)
    assert lib.kda_chunk_bwd_cp_workspace_size(N, T, H, 128, 128, 5, seg) == 0
