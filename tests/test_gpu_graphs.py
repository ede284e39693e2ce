"""The device calls are capturable in CUDA graphs (serving loops and training
steps replay a captured step instead of launching it): a captured verify,
single-token decode, two-kernel prefill and backward (sequence form and over
context-parallel segments) replay to the eager results bit for bit."""
import numpy as np
import pytest
import torch

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


def _decode_inputs(Wd, seed):
    from kda_gated_delta_02_gb300 import synth
    w = synth.DecodeWorkload("graph", 8, 4, 128, 128, W=4, Wd=Wd, seed=seed)
    acc = [0] * 8 if Wd == 0 else None
    return synth.make_decode(w, device="cuda", accepted=acc)


@pytest.mark.parametrize("Wd", [7, 0])
def test_verify_and_decode_replay_in_a_graph(kda, Wd):
    d = _decode_inputs(Wd, seed=20 + Wd)
    R, H, D = 8, 4, 128
    args = lambda st, tl, o: kda.decode_verify_replay(st, tl, d["conv_w"], d["cached_qkv"], d["cached_g"],
                                                       d["cached_b"], d["accepted"], d["new_qkv"], d["new_g"],
                                                       d["new_b"], d["out_w"], out=o)
    # eager: three steps in place (state and tail advance each step)
    st_e, tl_e = d["state"].clone(), d["tail"].clone()
    o_e = torch.empty((R, Wd + 1, H, D), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        args(st_e, tl_e, o_e)
    # graph: one captured step replayed three times
    st_g, tl_g = d["state"].clone(), d["tail"].clone()
    o_g = torch.empty_like(o_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        args(st_g.clone(), tl_g.clone(), o_g.clone())  # warm-up outside the capture (attributes, maps)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        args(st_g, tl_g, o_g)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st_g, st_e) and torch.equal(tl_g, tl_e) and torch.equal(o_g, o_e)


def test_two_kernel_prefill_in_a_graph(kda):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(5)
    lens = [300, 0, 129]
    T, H, D = sum(lens), 4, 128
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    q = torch.nn.functional.normalize(torch.randn(T, H, D, generator=gen), dim=-1).bfloat16().cuda()
    k = torch.nn.functional.normalize(torch.randn(T, H, D, generator=gen), dim=-1).bfloat16().cuda()
    v = torch.randn(T, H, D, generator=gen).bfloat16().cuda()
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, D, generator=gen)), -5.0).cuda()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).cuda()
    S0 = (0.02 * torch.randn(len(lens), H, D, D, generator=gen)).cuda()
    ws = torch.empty(kda.chunk_fwd_prep_workspace_size(len(lens), T, H, D, D, 0, 0), dtype=torch.uint8,
                     device="cuda")
    o_e, S_e = kda.chunk_fwd(q, k, v, g, beta, cu, initial_state=S0, cp_mode=0, workspace=ws)
    o_g = torch.empty_like(o_e)
    S_g = torch.empty_like(S_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kda.chunk_fwd(q, k, v, g, beta, cu, initial_state=S0, cp_mode=0, workspace=ws, out=o_g, final_state=S_g)
    torch.cuda.current_stream().wait_stream(s)
    o_g.zero_()
    S_g.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kda.chunk_fwd(q, k, v, g, beta, cu, initial_state=S0, cp_mode=0, workspace=ws, out=o_g, final_state=S_g)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(S_g, S_e)


def test_ragged_verify_in_a_graph(kda):
    d = _decode_inputs(7, seed=30)
    dl = torch.tensor([3, 7, 0, 5, 4, 6, 1, 2], dtype=torch.int32, device="cuda")
    R, H, D = 8, 4, 128
    run = lambda st, tl, o: kda.decode_verify_replay(st, tl, d["conv_w"], d["cached_qkv"], d["cached_g"],
                                                      d["cached_b"], d["accepted"], d["new_qkv"], d["new_g"],
                                                      d["new_b"], d["out_w"], out=o, draft_len=dl)
    st_e, tl_e = d["state"].clone(), d["tail"].clone()
    o_e = torch.zeros((R, 8, H, D), dtype=torch.bfloat16, device="cuda")
    run(st_e, tl_e, o_e)
    st_g, tl_g = d["state"].clone(), d["tail"].clone()
    o_g = torch.zeros_like(o_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(st_g.clone(), tl_g.clone(), o_g.clone())
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(st_g, tl_g, o_g)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(st_g, st_e) and torch.equal(tl_g, tl_e) and torch.equal(o_g, o_e)


@pytest.mark.parametrize("cp", [0, 1])
def test_backward_in_a_graph(kda, cp):
    """The tensor-core backward (its pipelined pieces: programmatic dependent
    launches) and the context-parallel backward replay from a CUDA graph to
    the eager gradients bit for bit; the outputs are allocated inside the
    capture, from the graph's pool."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(7 + cp)
    lens = [3000, 1500, 0, 2000] if not cp else [2500, 700]
    T, H, D = sum(lens), 2, 128
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    q = torch.nn.functional.normalize(torch.randn(T, H, D, generator=gen), dim=-1).bfloat16().cuda()
    k = torch.nn.functional.normalize(torch.randn(T, H, D, generator=gen), dim=-1).bfloat16().cuda()
    v = torch.randn(T, H, D, generator=gen).bfloat16().cuda()
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, D, generator=gen)), -5.0).cuda()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).cuda()
    S0 = (0.02 * torch.randn(len(lens), H, D, D, generator=gen)).cuda()
    do = torch.randn(T, H, D, generator=gen).bfloat16().cuda()
    lib = kda.load_library()
    need = (lib.kda_chunk_bwd_workspace_size(len(lens), T, H, D, D) if not cp else
            lib.kda_chunk_bwd_cp_workspace_size(len(lens), T, H, D, D, kda.CP_ON, 1024))
    ws = torch.empty(int(need), dtype=torch.uint8, device="cuda")

    def call():
        if cp:
            return kda.chunk_bwd_cp(q, k, v, g, beta, cu, do, initial_state=S0, scale=0.8, cp_mode=kda.CP_ON,
                                    segment_len=1024, workspace=ws)
        return kda.chunk_bwd(q, k, v, g, beta, cu, do, initial_state=S0, scale=0.8, workspace=ws)

    eager = [x.clone() for x in call()]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside the capture (attributes, maps)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = call()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(out, eager):
        assert torch.equal(a, b)


def test_training_pair_in_a_graph(kda):
    """A captured training step (the forward keeping its operands, then the
    reverse pass from them) replays to the eager outputs and gradients bit
    for bit."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(11)
    lens = [1500, 700]
    T, H, D = sum(lens), 2, 128
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    q = torch.nn.functional.normalize(torch.randn(T, H, D, generator=gen), dim=-1).bfloat16().cuda()
    k = torch.nn.functional.normalize(torch.randn(T, H, D, generator=gen), dim=-1).bfloat16().cuda()
    v = torch.randn(T, H, D, generator=gen).bfloat16().cuda()
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, D, generator=gen)), -5.0).cuda()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).cuda()
    do = torch.randn(T, H, D, generator=gen).bfloat16().cuda()
    saved = torch.empty(int(kda.load_library().kda_chunk_bwd_workspace_size(2, T, H, D, D)), dtype=torch.uint8,
                        device="cuda")

    def step():
        o, Sf, _ = kda.chunk_fwd_train(q, k, v, g, beta, cu, scale=0.6, saved=saved)
        return (o, Sf) + tuple(kda.chunk_bwd_saved(q, k, v, g, beta, cu, do, saved, scale=0.6))

    eager = [None if x is None else x.clone() for x in step()]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = step()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(out, eager):
        assert (a is None and b is None) or torch.equal(a, b)
