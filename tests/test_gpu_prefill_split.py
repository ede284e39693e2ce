"""The two-kernel form of the tcgen05 prefill (chunk-local products of every
chunk first, then the state walk) against the one-kernel form and the oracle.

Both forms run the same operations in the same order, so their outputs,
final states and checkpoints must agree bit for bit; the oracle bars of the
other prefill tests apply to the two-kernel form as well.  A workspace with
room for a few slots' operand blobs forces many pieces, so units cross piece
boundaries (carried states) and empty units fall inside pieces.
"""
import numpy as np
import pytest
import torch

from parity import OUT_TOL, STATE_TOL, normwise_err, split_layout, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kda_gated_delta_02_gb300 import build
    build.build()
    import kda_gated_delta_02_gb300 as k
    k.load_library()
    return k


def _inputs(lens, H, seed, s0=True, d=128):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1)
    v = torch.randn(T, H, d, generator=gen)
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, d, generator=gen)), -5.0)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen))
    S0 = 0.02 * torch.randn(len(lens), H, d, d, generator=gen) if s0 else None
    c = lambda x: None if x is None else x.cuda()
    return dict(q=c(q.bfloat16()), k=c(k.bfloat16()), v=c(v.bfloat16()), g=c(g), beta=c(beta), cu=c(cu), S0=c(S0))


def _align256(n):
    return (n + 255) // 256 * 256


def piece_workspace(kda, x, room, cp=0, seg=0):
    """A workspace with room for the blobs of `room` chunk slots (all heads)
    after the context-parallel scratch, the slot list, the item counters and
    two carry states, laid out as the library lays them out; returns it with
    the pieces it leads to."""
    N, (T, H) = x["cu"].shape[0] - 1, x["q"].shape[:2]
    plan = kda.chunk_fwd_plan(N, T, H, 128, 128, cp, seg)
    units = (T // plan + N) if plan else N
    _, _, pieces, _ = split_layout(T, H, units, room, plan != 0)
    _, _, _, fixed = split_layout(T, H, units, 0, plan != 0)
    nbytes = _align256(kda.chunk_fwd_workspace_size(N, T, H, 128, 128, cp, seg)) + fixed + room * H * 66048
    return torch.empty(nbytes, dtype=torch.uint8, device="cuda"), pieces


def _run(kda, x, prep, cp=0, seg=0, scale=1.0, every=0, K=0, slots=None):
    ck = None
    if every:
        N, H = x["cu"].shape[0] - 1, x["q"].shape[1]
        ck = torch.full((N, K, H, 128, 128), 7.0, device="cuda")
    ws = piece_workspace(kda, x, slots, cp, seg)[0] if (prep and slots) else None
    o, Sf = kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"], scale=scale,
                          cp_mode=cp, segment_len=seg, prep=prep, ckpt_every=every, ckpt=ck, workspace=ws)
    torch.cuda.synchronize()
    return o, Sf, ck


CASES = {
    # name: (lengths, H, cp_mode, segment_len, blob room in slots or None (all), checkpoint every, count)
    # (two buffers of room // 2 slots: pipelined pieces)
    "varlen_ragged": ([3 * 64 + 17, 0, 1, 64, 700], 3, 0, 0, None, 0, 0),
    "pieces_varlen": ([1000, 130, 0, 640, 1], 4, 0, 0, 6, 0, 0),
    "pieces_ckpt": ([640, 1000, 1536], 4, 0, 0, 14, 256, 6),
    "pieces_serial": ([1000, 130, 0, 640, 1], 4, 0, 0, 1, 0, 0),
    "pipeline_default": ([5000, 3000], 2, 0, 0, None, 0, 0),
    "cp_one_piece": ([5000], 2, 1, 1024, None, 0, 0),
    "cp_pieces": ([3000, 0, 1500, 64], 2, 1, 1024, 14, 0, 0),
    "cp_ckpt": ([4096], 2, 1, 1024, None, 768, 5),
}


@pytest.mark.parametrize("name", list(CASES))
def test_two_kernel_form_equals_one_kernel_form(kda, name):
    lens, H, cp, seg, slots, every, K = CASES[name]
    x = _inputs(lens, H, seed=len(name))
    T = int(sum(lens))
    ws_split = kda.chunk_fwd_prep_workspace_size(len(lens), T, H, 128, 128, cp, seg)
    ws_one = kda.chunk_fwd_workspace_size(len(lens), T, H, 128, 128, cp, seg)
    assert ws_split > ws_one
    o1, S1, c1 = _run(kda, x, prep=False, cp=cp, seg=seg, scale=0.5, every=every, K=K)
    o2, S2, c2 = _run(kda, x, prep=True, cp=cp, seg=seg, scale=0.5, every=every, K=K, slots=slots)
    assert torch.equal(o1, o2), f"outputs differ: max {float((o1.float() - o2.float()).abs().max()):.3e}"
    assert torch.equal(S1, S2), f"final states differ: max {float((S1 - S2).abs().max()):.3e}"
    if every:
        assert torch.equal(c1, c2), "checkpoints differ"


def test_pieces_match_oracle(kda, oracle):
    """Many pipelined pieces (3 slots each at H = 4): every unit of the three
    crosses piece boundaries; outputs and final states within the oracle bars."""
    lens = [700, 64, 0, 1300]
    x = _inputs(lens, 4, seed=5)
    o, Sf, _ = _run(kda, x, prep=True, scale=0.75, slots=6)
    o_ref, S_ref = oracle.prefill(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["g"]), to64(x["beta"]),
                                  x["cu"].cpu().numpy(), S0=to64(x["S0"]), scale=0.75)
    assert normwise_err(to64(o), o_ref, head_axis=1) <= OUT_TOL
    assert normwise_err(to64(Sf), S_ref, head_axis=1) <= STATE_TOL
    assert torch.equal(Sf[2], x["S0"][2])  # the empty sequence keeps its state


def test_two_kernel_form_reports_bad_seqlens(kda):
    x = _inputs([64, 64], 1, seed=13, s0=False)
    cu = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")  # not monotone
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((128, 1, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, out=o, cp_mode=0, status=status, prep=True)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.STATUS_BAD_SEQLENS
    assert torch.all(o[100:] == 7.0)


def test_kernel_timing_counts_the_launches(kda):
    """Launch timing around one two-kernel call: one slot list, and one
    chunk-local launch and one walk per piece (5 pieces here)."""
    x = _inputs([500, 300], 4, seed=3)  # 14 slots in two buffers of 3 (5 pieces)
    assert piece_workspace(kda, x, 6)[1] == 5
    kda.kernel_timing_start()
    _run(kda, x, prep=True, slots=6)
    kern = kda.kernel_timing_stop()
    n_pieces = 5
    assert kern["kda_chunk_list_kernel"]["launches"] == 1
    assert kern["kda_chunk_prep_kernel"]["launches"] == n_pieces
    assert kern["kda_chunk_walk_kernel"]["launches"] == n_pieces
    assert all(v["ms"] > 0 for v in kern.values())
    assert kda.kernel_timing_stop() == {}  # nothing recorded after stop


def test_pipelined_pieces_on_a_side_stream_graph(kda):
    """The pipelined form forks onto the library's two streams and joins back:
    the caller's stream sees the whole call (a graph captured on it replays
    the same bits as an eager call)."""
    x = _inputs([5000, 3000], 2, seed=17)
    ref = _run(kda, x, prep=True)
    o = torch.empty_like(x["v"])
    Sf = torch.empty(2, 2, 128, 128, dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.chunk_fwd_prep_workspace_size(2, 8000, 2, 128, 128, 0), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"], out=o,
                      final_state=Sf, cp_mode=0, workspace=ws)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"], out=o,
                          final_state=Sf, cp_mode=0, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref[0]) and torch.equal(Sf, ref[1])
