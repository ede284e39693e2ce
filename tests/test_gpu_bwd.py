"""kda_chunk_bwd (backward of the prefill) against the fp64 reverse-mode
oracle, on the same seeded inputs (the GPU's bf16 inputs rounded once, given
to both).

Two forms, chosen by shape and input type:
- bf16 inputs at d = 128: the chunk (WY) form on the tensor cores (forward
  pass keeping its operands, reverse state walk, chunk gradients).  Its
  products take bf16 operands with fp32 accumulation, so the bar is 1e-2
  normwise per head: the error budget of exactly that rounding is pinned on
  the CPU (tests/test_oracle_chunk_reverse.py::test_bf16_operand_error_budget).
- d = 64, or fp32 inputs: the token-level reverse mode in fp32 on the CUDA
  cores; bar 1e-3 (fp32 accumulation over the sequence).
Every gradient (dq, dk, dv, dg, dbeta, dS0) is compared as max |gpu - oracle|
/ max |oracle| per head; dg is exactly zero where g is under the floor.
"""
import numpy as np
import pytest
import torch

from parity import normwise_err, to64

pytestmark = pytest.mark.gpu
BWD_TOL = 1e-3
TC_TOL = 1e-2


def _tol(d, dtype):
    return TC_TOL if (d == 128 and dtype == torch.bfloat16) else BWD_TOL


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kda_gated_delta_02_gb300 import build
    build.build()
    import kda_gated_delta_02_gb300 as k
    k.load_library()
    return k


def _case(lens, H, d, dtype, seed, floor_frac=0.1):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    v = torch.randn(T, H, d, generator=gen).to(dtype)
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, d, generator=gen)), -4.9)
    below = torch.rand(T, H, d, generator=gen) < floor_frac
    g[below] = -5.5 - torch.rand(int(below.sum()), generator=gen)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen))
    S0 = 0.05 * torch.randn(len(lens), H, d, d, generator=gen)
    do = torch.randn(T, H, d, generator=gen).to(dtype)
    dSf = 0.1 * torch.randn(len(lens), H, d, d, generator=gen)
    c = lambda x: x.cuda()
    return dict(q=c(q), k=c(k), v=c(v), g=c(g), beta=c(beta), cu=c(cu), S0=c(S0), do=c(do), dSf=c(dSf))


def _compare(kda, oracle, x, scale, tol, heads=None, segment_len=None):
    if segment_len is None:
        got = kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], initial_state=x["S0"],
                            dS_final=x["dSf"], scale=scale)
    else:
        got = kda.chunk_bwd_cp(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], initial_state=x["S0"],
                               dS_final=x["dSf"], scale=scale, cp_mode=kda.CP_ON, segment_len=segment_len)
    torch.cuda.synchronize()
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    ref = oracle.backward(to64(sel(x["q"])), to64(sel(x["k"])), to64(sel(x["v"])), to64(sel(x["g"])),
                          to64(sel(x["beta"])), x["cu"].cpu().numpy(), to64(sel(x["do"])), S0=to64(sel(x["S0"])),
                          dS_final=to64(sel(x["dSf"])), scale=scale)
    names = ("dq", "dk", "dv", "dg", "dbeta", "dS0")
    for name, a, b in zip(names, got, ref):
        a64 = to64(sel(a))
        assert np.all(np.isfinite(a64)), f"{name}: non-finite"
        if name == "dbeta":
            e = np.max(np.abs(a64 - b)) / max(np.max(np.abs(b)), 1e-30)
        else:
            e = normwise_err(a64, b, head_axis=1)
        assert e <= tol, f"{name}: error {e:.3e}"
    g = x["g"].cpu()
    assert torch.all(got[3].cpu()[g < -5.0] == 0.0), "gradient through the floor"
    return got


@pytest.mark.parametrize("d,dtype,lens", [(128, torch.bfloat16, [200, 0, 65, 1]),
                                          (64, torch.float32, [150, 64]),
                                          (128, torch.float32, [64, 129]),
                                          (64, torch.bfloat16, [100, 37])])
def test_backward_matches_oracle(kda, oracle, d, dtype, lens):
    x = _case(lens, 2, d, dtype, seed=d + len(lens))
    got = _compare(kda, oracle, x, scale=0.7, tol=_tol(d, dtype))
    # the empty sequence passes its final-state gradient straight to dS0
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.equal(got[5][n], x["dSf"][n])


def test_backward_many_chunks(kda, oracle):
    """2,048 tokens (32 chunks) x 4 heads, bf16 (tensor-core form)."""
    x = _case([2048], 4, 128, torch.bfloat16, seed=7)
    _compare(kda, oracle, x, scale=1.0, tol=TC_TOL)


def test_backward_bad_seqlens_and_workspace(kda):
    x = _case([64, 64], 1, 128, torch.bfloat16, seed=9)
    cu = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, x["do"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.STATUS_BAD_SEQLENS
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    lib = kda.load_library()
    need = lib.kda_chunk_bwd_workspace_size(2, 128, 1, 128, 128)
    assert need > 1024
    with pytest.raises(kda.KDAError):
        # a caller-provided workspace below the size is reallocated by the
        # binding, so call the ABI directly
        import ctypes
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        outs = [torch.empty(128, 1, 128, device="cuda") for _ in range(4)] + [torch.empty(128, 1, device="cuda")]
        rc = lib.kda_chunk_bwd(P(x["q"]), P(x["k"]), P(x["v"]), P(x["g"]), P(x["beta"]), P(x["cu"]), 2, 128, 1,
                               128, 128, None, P(x["do"]), None, *[P(o) for o in outs], None, 1.0, -5.0, 0,
                               P(small), ctypes.c_size_t(1024), None, None)
        kda._check(rc, "kda_chunk_bwd")


def test_backward_more_units_than_ctas(kda, oracle):
    """30 sequences x 8 heads = 240 (sequence, head) units over at most 160
    persistent CTAs (CUDA-core form, d = 64): units share a CTA's scratch in turn."""
    rng = np.random.default_rng(13)
    lens = rng.integers(0, 140, size=30).tolist()
    x = _case(lens, 8, 64, torch.bfloat16, seed=13)
    _compare(kda, oracle, x, scale=1.0, tol=BWD_TOL)


def test_tensor_core_backward_many_short_sequences(kda, oracle):
    """40 ragged sequences (0 to 150 tokens) x 6 heads in the tensor-core form:
    many more (chunk, head) items than persistent CTAs, partial chunks,
    empty sequences."""
    rng = np.random.default_rng(17)
    lens = rng.integers(0, 150, size=40).tolist()
    lens[3] = 0
    x = _case(lens, 6, 128, torch.bfloat16, seed=17)
    got = _compare(kda, oracle, x, scale=0.5, tol=TC_TOL)
    assert torch.equal(got[5][3], x["dSf"][3])


def test_tensor_core_backward_in_pieces(kda, oracle):
    """105 chunk slots over 2 heads run as four pipelined pieces (the forward
    pass, then the reverse walk newest piece first with each piece's chunk
    gradients overlapping the next piece's walk): sequences cross piece
    boundaries in both passes (carried states and state gradients), one is
    empty."""
    lens = [3000, 1500, 0, 2000]
    x = _case(lens, 2, 128, torch.bfloat16, seed=37)
    kda.kernel_timing_start()
    got = _compare(kda, oracle, x, scale=0.9, tol=TC_TOL)
    kern = kda.kernel_timing_stop()
    assert kern["kda_bwd_walk_kernel"]["launches"] == 4 and kern["kda_bwd_chunk_kernel"]["launches"] == 4
    assert kern["kda_chunk_walk_kernel"]["launches"] == 4
    assert torch.equal(got[5][2], x["dSf"][2])


def test_tensor_core_backward_scale_zero(kda, oracle):
    """scale = 0: the outputs are zero, so do enters no gradient; the state
    gradient still flows from dS_final."""
    x = _case([300, 70], 2, 128, torch.bfloat16, seed=19)
    _compare(kda, oracle, x, scale=0.0, tol=TC_TOL)


def test_tensor_core_backward_full_length_sampled_heads(kda, oracle):
    """The bench's workload, 32,768 tokens x 96 heads in one launch; heads 0
    and 95 against the oracle at every token (the heads are independent)."""
    x = _case([32768], 96, 128, torch.bfloat16, seed=23, floor_frac=0.02)
    _compare(kda, oracle, x, scale=128 ** -0.5, tol=TC_TOL, heads=[0, 95])


def test_tensor_core_backward_launches(kda):
    """One slot list, one chunk-local launch (keeping T and M), one forward
    walk (keeping its tiles), one reverse walk and one chunk-gradient launch."""
    x = _case([500, 300], 2, 128, torch.bfloat16, seed=29)
    kda.kernel_timing_start()
    kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], initial_state=x["S0"])
    kern = kda.kernel_timing_stop()
    assert {k: v["launches"] for k, v in kern.items()} == {
        "kda_chunk_list_kernel": 1, "kda_chunk_prep_kernel": 1, "kda_chunk_walk_kernel": 1,
        "kda_bwd_walk_kernel": 1, "kda_bwd_chunk_kernel": 1}


def _grads(kda, x, scale):
    got = kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], initial_state=x["S0"],
                        dS_final=x["dSf"], scale=scale)
    torch.cuda.synchronize()
    return got


def test_tensor_core_backward_is_deterministic(kda):
    """Items are claimed dynamically, but every result is written by one
    thread in a fixed order: two calls give the same bits."""
    x = _case([1000, 333], 3, 128, torch.bfloat16, seed=31)
    a = _grads(kda, x, 0.8)
    b = _grads(kda, x, 0.8)
    for u, w in zip(a, b):
        assert torch.equal(u, w)


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_absent_states_and_no_dS0(kda, oracle, d, dtype):
    """initial_state and dS_final absent (zero), dS0 not asked for."""
    x = _case([130, 64], 2, d, dtype, seed=41)
    got = kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], scale=0.8, want_dS0=False)
    torch.cuda.synchronize()
    assert got[5] is None
    ref = oracle.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["g"]), to64(x["beta"]),
                          x["cu"].cpu().numpy(), to64(x["do"]), scale=0.8)
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got[:5], ref[:5]):
        e = normwise_err(to64(a), b, head_axis=1)
        assert e <= _tol(d, dtype), f"{name}: error {e:.3e}"


def test_floor_held_on_whole_chunks(kda, oracle):
    """g at the floor exactly (-5) on whole chunks passes its gradient; g below
    it on other chunks passes none (tensor-core form: e^{-5 x 64} inside a
    chunk is carried by the 16-token block anchoring)."""
    x = _case([256], 2, 128, torch.bfloat16, seed=43, floor_frac=0.0)
    g = x["g"].clone()
    g[0:64] = -5.0
    g[128:192] = -6.0
    x["g"] = g
    got = _compare(kda, oracle, x, scale=1.0, tol=TC_TOL)
    assert torch.all(got[3][128:192] == 0.0)
    assert torch.count_nonzero(got[3][0:64]) > 0


def test_training_pair_equals_forward_and_backward(kda, oracle):
    """chunk_fwd_train returns chunk_fwd's outputs bit for bit and keeps what
    chunk_bwd_saved needs; chunk_bwd_saved returns chunk_bwd's gradients bit
    for bit (same kernels on the same operands), in four pieces with a cut
    sequence, an empty one, and dS_final."""
    lens = [3000, 0, 1500, 2000]
    x = _case(lens, 2, 128, torch.bfloat16, seed=47)
    o_ref, S_ref = kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"],
                                 scale=0.6)
    o, Sf, saved = kda.chunk_fwd_train(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"],
                                       scale=0.6)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(Sf, S_ref)
    ref = kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], initial_state=x["S0"],
                        dS_final=x["dSf"], scale=0.6)
    got = kda.chunk_bwd_saved(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], saved,
                              dS_final=x["dSf"], scale=0.6)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    # and the pair's backward against the oracle
    r = oracle.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["g"]), to64(x["beta"]),
                        x["cu"].cpu().numpy(), to64(x["do"]), S0=to64(x["S0"]), dS_final=to64(x["dSf"]), scale=0.6)
    assert normwise_err(to64(got[0]), r[0], head_axis=1) <= TC_TOL
    assert normwise_err(to64(got[3]), r[3], head_axis=1) <= TC_TOL


def test_training_pair_rejects_other_shapes(kda):
    x = _case([100], 1, 64, torch.bfloat16, seed=53)
    with pytest.raises(kda.KDAError):
        kda.chunk_fwd_train(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"])


@pytest.mark.parametrize("lens,seg", [([5000], 1024), ([3000, 0, 1500, 2000], 1024), ([1100, 64, 1], 512),
                                      ([700], 64)])
def test_context_parallel_backward_matches_oracle(kda, oracle, lens, seg):
    """The backward over context-parallel segments: the forward pass as the CP
    prefill runs it (transitions, their ordered composition, the replay
    keeping its tiles), every segment walked back from zero, the state
    gradient scanned over the segments last to first, every segment walked
    back again from its exact end gradient, then the chunk gradients.
    Sequences span several segments, end mid-segment and mid-chunk, are
    shorter than one segment or empty; segments of one chunk each."""
    x = _case(lens, 2, 128, torch.bfloat16, seed=59 + seg)
    kda.kernel_timing_start()
    got = _compare(kda, oracle, x, scale=0.7, tol=TC_TOL, segment_len=seg)
    kern = kda.kernel_timing_stop()
    assert kern["kda_bwd_walk_kernel"]["launches"] == 2 and kern["kda_bwd_chunk_kernel"]["launches"] == 1
    assert kern["kda_bwd_compose_kernel"]["launches"] == 1 and kern["kda_compose_kernel"]["launches"] == 1
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.equal(got[5][n], x["dSf"][n])


def test_context_parallel_backward_long_sampled_heads(kda, oracle):
    """Two long sequences (24,576 and 8,000 tokens) over 16 heads cut into
    2,048-token segments; heads 0 and 15 against the oracle."""
    x = _case([24576, 8000], 16, 128, torch.bfloat16, seed=61, floor_frac=0.02)
    _compare(kda, oracle, x, scale=128 ** -0.5, tol=TC_TOL, heads=[0, 15], segment_len=2048)


def test_context_parallel_backward_arguments(kda):
    """A segment length that is not a multiple of the chunk, an unknown mode
    and a workspace below the size are refused; cp off (or no segment for the
    call) is the sequence form bit for bit."""
    x = _case([300, 200], 1, 128, torch.bfloat16, seed=67)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"])
    with pytest.raises(kda.KDAError):
        kda.chunk_bwd_cp(*args, cp_mode=kda.CP_ON, segment_len=100)
    with pytest.raises(kda.KDAError):
        kda.chunk_bwd_cp(*args, cp_mode=7, segment_len=128)
    lib = kda.load_library()
    need = lib.kda_chunk_bwd_cp_workspace_size(2, 500, 1, 128, 128, kda.CP_ON, 128)
    assert need >= lib.kda_chunk_bwd_workspace_size(2, 500, 1, 128, 128)
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    outs = [torch.empty(500, 1, 128, device="cuda") for _ in range(4)] + [torch.empty(500, 1, device="cuda")]
    small = torch.empty(4096, dtype=torch.uint8, device="cuda")
    rc = lib.kda_chunk_bwd_cp(P(x["q"]), P(x["k"]), P(x["v"]), P(x["g"]), P(x["beta"]), P(x["cu"]), 2, 500, 1,
                              128, 128, None, P(x["do"]), None, *[P(o) for o in outs], None, 1.0, -5.0, 0,
                              kda.CP_ON, 128, P(small), ctypes.c_size_t(4096), None, None)
    with pytest.raises(kda.KDAError):
        kda._check(rc, "kda_chunk_bwd_cp")
    ref = _grads(kda, x, 0.9)
    for mode, seg in ((kda.CP_OFF, 0), (kda.CP_AUTO, 0)):
        got = kda.chunk_bwd_cp(*args, initial_state=x["S0"], dS_final=x["dSf"], scale=0.9, cp_mode=mode,
                               segment_len=seg)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_context_parallel_training_pair(kda, oracle):
    """The training pair on the context-parallel schedule: chunk_fwd_train
    returns chunk_fwd's CP outputs bit for bit and keeps the segments'
    operands; chunk_bwd_saved returns chunk_bwd_cp's gradients bit for bit;
    sequences over several segments, an empty one, dS_final."""
    lens = [3000, 0, 1500, 2000]
    x = _case(lens, 2, 128, torch.bfloat16, seed=71)
    cp = dict(cp_mode=kda.CP_ON, segment_len=1024)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"])
    o_ref, S_ref = kda.chunk_fwd(*args, initial_state=x["S0"], scale=0.6, **cp)
    kda.kernel_timing_start()
    o, Sf, saved = kda.chunk_fwd_train(*args, initial_state=x["S0"], scale=0.6, **cp)
    kern = kda.kernel_timing_stop()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(Sf, S_ref)
    assert torch.equal(Sf[1], x["S0"][1])
    assert kern["kda_chunk_walk_kernel"]["launches"] == 2 and "kda_bwd_walk_kernel" not in kern
    ref = kda.chunk_bwd_cp(*args, x["do"], initial_state=x["S0"], dS_final=x["dSf"], scale=0.6, **cp)
    kda.kernel_timing_start()
    got = kda.chunk_bwd_saved(*args, x["do"], saved, dS_final=x["dSf"], scale=0.6, **cp)
    kern = kda.kernel_timing_stop()
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    assert "kda_chunk_walk_kernel" not in kern and kern["kda_bwd_walk_kernel"]["launches"] == 2
    r = oracle.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["g"]), to64(x["beta"]),
                        x["cu"].cpu().numpy(), to64(x["do"]), S0=to64(x["S0"]), dS_final=to64(x["dSf"]), scale=0.6)
    for i in (0, 1, 2, 3, 5):
        assert normwise_err(to64(got[i]), r[i], head_axis=1) <= TC_TOL


@pytest.mark.parametrize("scale,floor", [(0.0, False), (0.8, True)])
def test_context_parallel_backward_edges(kda, oracle, scale, floor):
    """Context-parallel segments with absent initial state and end gradient
    (zero), dS0 not asked for; scale 0 (the state gradient is zero, dO enters
    no product), or chunks held at and below the floor."""
    x = _case([2500, 700], 2, 128, torch.bfloat16, seed=73 + int(floor), floor_frac=0.0)
    if floor:
        g = x["g"].clone()
        g[0:64] = -5.0
        g[1024:1100] = -6.0
        g[2600:2700] = -5.5
        x["g"] = g
    got = kda.chunk_bwd_cp(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["do"], scale=scale,
                           cp_mode=kda.CP_ON, segment_len=1024, want_dS0=False)
    torch.cuda.synchronize()
    assert got[5] is None
    ref = oracle.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["g"]), to64(x["beta"]),
                          x["cu"].cpu().numpy(), to64(x["do"]), scale=scale)
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got[:5], ref[:5]):
        a64 = to64(a)
        assert np.all(np.isfinite(a64)), name
        if np.max(np.abs(b)) == 0.0:
            assert np.all(a64 == 0.0), name
            continue
        e = normwise_err(a64, b, head_axis=1) if name != "dbeta" else np.max(np.abs(a64 - b)) / np.max(np.abs(b))
        assert e <= TC_TOL, f"{name}: error {e:.3e}"
    g = x["g"].cpu()
    assert torch.all(got[3].cpu()[g < -5.0] == 0.0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_context_parallel_backward_random_cuts(kda, oracle, seed):
    """Random sequence counts and lengths (empty and sub-chunk ones
    included) and random segment lengths (multiples of 64 from one chunk to
    sixteen) against the oracle; the training pair on the same cut gives the
    same bits."""
    rng = np.random.default_rng(200 + seed)
    n = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.integers(0, 1500, size=n)]
    lens[int(rng.integers(0, n))] = int(rng.integers(1, 64)) if n > 1 else lens[0]
    seg = 64 * int(rng.integers(1, 17))
    x = _case(lens, 2, 128, torch.bfloat16, seed=300 + seed)
    if sum(lens) == 0:
        pytest.skip("no tokens drawn")
    got = _compare(kda, oracle, x, scale=0.75, tol=TC_TOL, segment_len=seg)
    cp = dict(cp_mode=kda.CP_ON, segment_len=seg)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"])
    _, _, saved = kda.chunk_fwd_train(*args, initial_state=x["S0"], scale=0.75, **cp)
    pair = kda.chunk_bwd_saved(*args, x["do"], saved, dS_final=x["dSf"], scale=0.75, **cp)
    torch.cuda.synchronize()
    for a, b in zip(pair, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_backward_beta_zero(kda, oracle, d, dtype):
    """beta = 0 (the state only decays): dv is exactly zero, the rest against
    the oracle, dbeta included (its gradient does not vanish)."""
    x = _case([400, 130], 2, d, dtype, seed=131 + d)
    x["beta"] = torch.zeros_like(x["beta"])
    got = _compare(kda, oracle, x, scale=0.8, tol=_tol(d, dtype))
    assert torch.count_nonzero(got[2]) == 0
    assert torch.count_nonzero(got[4]) > 0
