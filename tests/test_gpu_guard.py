"""Guard bands around every output buffer: each entry point writes into views
in the middle of larger buffers whose two bands (16 KiB or more each side)
hold a sentinel byte pattern.  After the call the bands must still hold it
bit for bit (no write past either end of an output), and the results must
equal those of the same call on ordinary buffers (nothing depends on the
neighbouring memory).  Covered: the two-kernel prefill in pipelined pieces and
with context-parallel segments, the tensor-core and CUDA-core backward, the
context-parallel backward, the training pair, verify-replay (uniform and
ragged) and single-token decode, whose state and conv tail are updated in
place."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
G = 4096  # guard elements on each side
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kda_gated_delta_02_gb300 import build
    build.build()
    import kda_gated_delta_02_gb300 as k
    k.load_library()
    return k


def guarded(shape, dtype, init=None):
    """(whole buffer, view of `shape` in its middle); the bands hold the
    sentinel, the view `init` (copied) or the sentinel too."""
    n = int(np.prod(shape))
    full = torch.empty(n + 2 * G, dtype=dtype, device="cuda")
    full.view(torch.uint8).fill_(SENTINEL)
    view = full[G:G + n].view(shape)
    if init is not None:
        view.copy_(init)
    return full, view


def intact(full):
    b = full.view(torch.uint8)
    eb = G * full.element_size()
    return bool(torch.all(b[:eb] == SENTINEL)) and bool(torch.all(b[-eb:] == SENTINEL))


def _prefill_case(lens, H, d, dtype, seed):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    v = torch.randn(T, H, d, generator=gen).to(dtype)
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, d, generator=gen)), -4.9)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen))
    S0 = 0.05 * torch.randn(len(lens), H, d, d, generator=gen)
    do = torch.randn(T, H, d, generator=gen).to(dtype)
    dSf = 0.1 * torch.randn(len(lens), H, d, d, generator=gen)
    c = lambda x: x.cuda()
    return dict(q=c(q), k=c(k), v=c(v), g=c(g), beta=c(beta), cu=c(cu), S0=c(S0), do=c(do), dSf=c(dSf),
                N=len(lens), T=T, H=H, d=d)


@pytest.mark.parametrize("cp,seg", [(0, 0), (1, 1024)])
def test_prefill_writes_stay_in_bounds(kda, cp, seg):
    """Two-kernel prefill: four pipelined pieces (cp off) or segments of
    1,024 tokens; an empty sequence passes its state through."""
    x = _prefill_case([3000, 0, 1500, 2000], 2, 128, torch.bfloat16, seed=81)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"])
    fo, o = guarded((x["T"], 2, 128), torch.bfloat16)
    fs, S = guarded((x["N"], 2, 128, 128), torch.float32)
    kda.chunk_fwd(*args, initial_state=x["S0"], scale=0.5, cp_mode=cp, segment_len=seg, out=o, final_state=S)
    o_ref, S_ref = kda.chunk_fwd(*args, initial_state=x["S0"], scale=0.5, cp_mode=cp, segment_len=seg)
    torch.cuda.synchronize()
    assert intact(fo) and intact(fs)
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)


def _bwd_abi(kda, x, outs, ws, cp=None):
    lib = kda.load_library()
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    dt = 0 if x["q"].dtype == torch.bfloat16 else 1
    head = (P(x["q"]), P(x["k"]), P(x["v"]), P(x["g"]), P(x["beta"]), P(x["cu"]), x["N"], x["T"], x["H"], x["d"],
            x["d"], P(x["S0"]), P(x["do"]), P(x["dSf"])) + tuple(P(t) for t in outs) + (0.7, -5.0, dt)
    tail = (P(ws), ctypes.c_size_t(ws.numel()), None, None)
    if cp is None:
        rc = lib.kda_chunk_bwd(*head, *tail)
    else:
        rc = lib.kda_chunk_bwd_cp(*head, kda.CP_ON, cp, *tail)
    kda._check(rc, "backward")


@pytest.mark.parametrize("d,dtype,lens,cp", [(128, torch.bfloat16, [3000, 0, 1500, 2000], None),
                                             (128, torch.bfloat16, [2500, 700], 1024),
                                             (64, torch.float32, [150, 0, 64], None)])
def test_backward_writes_stay_in_bounds(kda, d, dtype, lens, cp):
    """Tensor-core backward (four pieces), its context-parallel form and the
    CUDA-core form: dq, dk, dv, dg, dbeta and dS0 in guarded buffers."""
    x = _prefill_case(lens, 2, d, dtype, seed=83 + d)
    T, H, N = x["T"], x["H"], x["N"]
    shapes = [(T, H, d)] * 4 + [(T, H), (N, H, d, d)]
    fulls, views = zip(*[guarded(s, torch.float32) for s in shapes])
    lib = kda.load_library()
    need = (lib.kda_chunk_bwd_workspace_size(N, T, H, d, d) if cp is None else
            lib.kda_chunk_bwd_cp_workspace_size(N, T, H, d, d, kda.CP_ON, cp))
    fw, ws = guarded((int(need),), torch.uint8)
    _bwd_abi(kda, x, views, ws, cp)
    refs = [torch.empty(s, dtype=torch.float32, device="cuda") for s in shapes]
    _bwd_abi(kda, x, refs, torch.empty(int(need), dtype=torch.uint8, device="cuda"), cp)
    torch.cuda.synchronize()
    for name, f in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0", "workspace"), list(fulls) + [fw]):
        assert intact(f), name
    for a, b in zip(views, refs):
        assert torch.equal(a, b)


def test_training_pair_writes_stay_in_bounds(kda):
    """kda_chunk_fwd_train's outputs and saved operands, then
    kda_chunk_bwd_saved's gradients, all in guarded buffers."""
    x = _prefill_case([1500, 700], 2, 128, torch.bfloat16, seed=89)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"])
    lib = kda.load_library()
    need = int(lib.kda_chunk_bwd_workspace_size(x["N"], x["T"], 2, 128, 128))
    fsv, saved = guarded((need,), torch.uint8)
    o, Sf, _ = kda.chunk_fwd_train(*args, initial_state=x["S0"], scale=0.7, saved=saved)
    got = kda.chunk_bwd_saved(*args, x["do"], saved, dS_final=x["dSf"], scale=0.7)
    ref = kda.chunk_bwd(*args, x["do"], initial_state=x["S0"], dS_final=x["dSf"], scale=0.7)
    torch.cuda.synchronize()
    assert intact(fsv)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("ragged,Wd", [(False, 7), (True, 7), (False, 0)])
def test_verify_and_decode_write_stay_in_bounds(kda, ragged, Wd):
    """Verify-replay (uniform and ragged) and single-token decode (no draft
    window): the state and conv tail updated in place inside guarded buffers,
    the outputs in one; ragged rows past a request's drafts stay unwritten."""
    from kda_gated_delta_02_gb300 import synth
    w = synth.DecodeWorkload("guard", 8, 4, 128, 128, Wd=Wd, seed=91)
    d = synth.make_decode(w, device="cuda", accepted=None if Wd else [0] * 8)
    dl = None
    if ragged:
        dl = torch.tensor([0, 7, 3, 5, 7, 1, 4, 6], dtype=torch.int32, device="cuda")
    fst, st = guarded(tuple(d["state"].shape), torch.bfloat16, d["state"])
    ftl, tl = guarded(tuple(d["tail"].shape), torch.bfloat16, d["tail"])
    fo, o = guarded((8, Wd + 1, 4, 128), torch.bfloat16)
    ins = (d["conv_w"], d["cached_qkv"], d["cached_g"], d["cached_b"], d["accepted"], d["new_qkv"], d["new_g"],
           d["new_b"], d["out_w"])
    kda.decode_verify_replay(st, tl, *ins, out=o, draft_len=dl)
    st2, tl2 = d["state"].clone(), d["tail"].clone()
    o2 = kda.decode_verify_replay(st2, tl2, *ins, draft_len=dl)
    torch.cuda.synchronize()
    assert intact(fst) and intact(ftl) and intact(fo)
    assert torch.equal(st, st2) and torch.equal(tl, tl2)
    if dl is None:
        assert torch.equal(o, o2)
    else:
        for r in range(8):
            n = int(dl[r]) + 1
            assert torch.equal(o[r, :n], o2[r, :n])
            assert bool(torch.all(o[r, n:].view(torch.uint8) == SENTINEL))
