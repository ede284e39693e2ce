"""The allocation-free context-parallel prefill (kda_chunk_fwd_cp_noalloc).

It serves callers that may not call cudaMalloc or hand over a workspace (a
host that forbids device allocation after start-up, a plugin whose host owns
every buffer): its scratch is a fixed device array inside the library.  This
test calls it through the C ABI, twice in a row on different inputs, and
checks each result against kda_chunk_fwd with a caller workspace bit for bit
(the forms the fixed scratch selects run the same operations in the same
order as the workspace call's), and one result against the oracle within the
parity bars the other tests use.  The sizes cover the three forms the fixed
scratch leads to: everything in one piece, the two-kernel form in several
pieces, and the one-kernel form when the carried states do not fit beside
the context-parallel scratch.  It sits in a file of its own, collected last,
and works alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

from parity import OUT_TOL, STATE_TOL, normwise_err, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kda_gated_delta_02_gb300 import build
    build.build()
    import kda_gated_delta_02_gb300 as kda
    L = kda.load_library()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.kda_chunk_fwd_cp_noalloc.restype = I
    L.kda_chunk_fwd_cp_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, F, F, I, I, P, P]
    return L


def _inputs(lens, H, seed):
    gen = torch.Generator().manual_seed(seed)
    T = sum(lens)
    q = torch.nn.functional.normalize(torch.randn(T, H, 128, generator=gen), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(T, H, 128, generator=gen), dim=-1)
    v = torch.randn(T, H, 128, generator=gen)
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, 128, generator=gen)), -5.0)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen))
    S0 = 0.02 * torch.randn(len(lens), H, 128, 128, generator=gen)
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32)
    c = lambda x: x.cuda()
    return dict(q=c(q.bfloat16()), k=c(k.bfloat16()), v=c(v.bfloat16()), g=c(g), beta=c(beta), S0=c(S0),
                cu=c(cu))


def _noalloc(lib, x, seg):
    T, H, dk = x["k"].shape
    N = x["cu"].shape[0] - 1
    o = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    Sf = torch.empty(N, H, dk, 128, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.kda_chunk_fwd_cp_noalloc(p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]), p(x["cu"]),
                                      N, T, H, dk, 128, p(x["S0"]), p(Sf), p(o), 1.0, -5.0, 0, seg, None,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.kda_status_string(rc)
    return o, Sf


def _with_workspace(x, seg):
    import kda_gated_delta_02_gb300 as kda
    return kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"],
                         cp_mode=kda.CP_ON, segment_len=seg)


def _layout(lib, x, seg):
    """(pieces, two-kernel form?) that 64 MiB of scratch leads to, from the
    library's workspace arithmetic."""
    import kda_gated_delta_02_gb300 as kda
    from parity import split_layout
    T, H, _ = x["k"].shape
    N = x["cu"].shape[0] - 1
    cp = kda.chunk_fwd_workspace_size(N, T, H, 128, 128, kda.CP_ON, seg)
    units = T // kda.chunk_fwd_plan(N, T, H, 128, 128, kda.CP_ON, seg) + N
    fixed = split_layout(T, H, units, 0, True)[3]
    room = ((64 << 20) - (cp + 255) // 256 * 256 - fixed) // (H * 66048)
    pieces = split_layout(T, H, units, max(room, 0), True)[2]
    return pieces, pieces > 0


def test_noalloc_matches_workspace_entry_point_twice(lib, oracle):
    cases = [(_inputs([3000, 1500], 3, seed=1), 1024, (1, True)),   # one piece
             (_inputs([8192], 8, seed=2), 1024, (3, True)),          # pipelined pieces
             (_inputs([2048], 96, seed=4), 1024, (0, False))]        # one-kernel form
    for x, seg, form in cases:  # calls in a row share the fixed scratch
        assert _layout(lib, x, seg) == form
        o, Sf = _noalloc(lib, x, seg)
        o_ref, Sf_ref = _with_workspace(x, seg)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), f"outputs differ: max {float((o.float() - o_ref.float()).abs().max()):.3e}"
        assert torch.equal(Sf, Sf_ref), f"states differ: max {float((Sf - Sf_ref).abs().max()):.3e}"
    x, seg, _ = cases[0]
    o, Sf = _noalloc(lib, x, seg)
    torch.cuda.synchronize()
    o_or, S_or = oracle.prefill(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["g"]), to64(x["beta"]),
                                x["cu"].cpu().numpy(), S0=to64(x["S0"]))
    assert normwise_err(to64(o), o_or, 1) <= OUT_TOL
    assert normwise_err(to64(Sf), S_or, 1) <= STATE_TOL


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    x = _inputs([64], 1, seed=3)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    # a million tokens x 96 heads in 1024-token segments needs far more than 64 MiB
    rc = lib.kda_chunk_fwd_cp_noalloc(p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]), p(x["cu"]),
                                      1, 1 << 20, 96, 128, 128, None, None, p(x["q"]), 1.0, -5.0, 0, 1024,
                                      None, None)
    assert rc == -6
    assert b"scratch" in lib.kda_status_string(rc)
