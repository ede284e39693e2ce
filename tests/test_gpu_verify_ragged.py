"""kda_decode_verify_replay_ragged: a draft count per request against the
fp64 oracle (the same ragged rule), on inputs whose padded draft rows hold
NaN, and against the uniform call.

Bars as for the uniform verify: valid output rows 2e-2 and the written-back
bf16 state 1e-2 normwise relative error per head; conv tail, skipped requests
and unwritten rows bit-exact; with every count equal to the window the ragged
call equals the uniform one bit for bit.
"""
import numpy as np
import pytest
import torch

from parity import OUT_TOL, STATE_TOL, normwise_err, to64

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


def _inputs(R, H, D, accepted, Wd, seed, W=4):
    from kda_gated_delta_02_gb300 import synth
    w = synth.DecodeWorkload("ragged", R, H, D, D, W=W, Wd=Wd, seed=seed)
    return synth.make_decode(w, device="cuda", accepted=accepted)


def _poison(inp, d):
    """NaN in every new row past each request's draft count."""
    for r, dr in enumerate(d):
        for key in ("new_qkv", "new_g", "new_b"):
            inp[key][r, dr + 1:] = float("nan")
    return inp


def _run(kda, inp, d=None, scale=1.0):
    st, tl = inp["state"].clone(), inp["tail"].clone()
    R, H, D, _ = st.shape
    Wd = inp["new_qkv"].shape[1] - 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((R, Wd + 1, H, D), -3.0, dtype=torch.bfloat16, device="cuda")
    dl = None if d is None else torch.as_tensor(d, dtype=torch.int32, device="cuda")
    kda.decode_verify_replay(st, tl, inp["conv_w"], inp["cached_qkv"], inp["cached_g"], inp["cached_b"],
                             inp["accepted"], inp["new_qkv"], inp["new_g"], inp["new_b"], inp["out_w"],
                             scale=scale, out=o, status=status, draft_len=dl)
    torch.cuda.synchronize()
    return st, tl, o, int(status.item())


def _oracle(oracle, inp, d, scale=1.0):
    return oracle.decode_verify(to64(inp["state"]), to64(inp["tail"]), to64(inp["conv_w"]),
                                to64(inp["cached_qkv"]), to64(inp["cached_g"]), to64(inp["cached_b"]),
                                inp["accepted"].cpu().numpy(), to64(inp["new_qkv"]), to64(inp["new_g"]),
                                to64(inp["new_b"]), to64(inp["out_w"]), scale=scale,
                                draft_len=np.asarray(d, dtype=np.int32))


def _check(inp, got, ref, d):
    st, tl, o, status = got
    st_r, tl_r, o_r, bad = ref
    assert status == 0 and bad == 0
    o64 = to64(o)
    rows = [(r, t) for r in range(len(d)) for t in range(d[r] + 1)]
    ro = np.stack([o64[r, t] for r, t in rows])      # [rows, H, D]
    rr = np.stack([o_r[r, t] for r, t in rows])
    e_o = normwise_err(ro, rr, head_axis=1)
    e_s = normwise_err(to64(st), st_r, head_axis=1)
    assert e_o <= OUT_TOL, f"output error {e_o:.3e}"
    assert e_s <= STATE_TOL, f"state error {e_s:.3e}"
    assert torch.equal(tl.cpu(), torch.from_numpy(tl_r).to(torch.bfloat16)), "conv tail not bit-exact"
    for r, dr in enumerate(d):
        assert torch.all(o[r, dr + 1:] == -3.0), f"request {r}: rows past its drafts were written"
    return e_o, e_s


@pytest.mark.parametrize("D,Wd", [(128, 7), (128, 3), (64, 7)])
def test_ragged_matches_oracle_with_nan_padding(kda, oracle, D, Wd):
    rng = np.random.default_rng(D + Wd)
    R, H = 12, 3
    acc = rng.integers(0, Wd + 1, size=R).tolist()
    d = rng.integers(0, Wd + 1, size=R)
    d[0], d[1] = 0, Wd
    d = d.tolist()
    inp = _poison(_inputs(R, H, D, acc, Wd, seed=D + 3 * Wd), d)
    got = _run(kda, inp, d, scale=0.5)
    ref = _oracle(oracle, inp, d, scale=0.5)
    _check(inp, got, ref, d)


@pytest.mark.parametrize("D", [128, 64])
def test_full_counts_equal_the_uniform_call(kda, D):
    """The uniform call is the ragged one with every count = Wd, bit for bit."""
    inp = _inputs(8, 2, D, list(range(8)), 7, seed=40 + D)
    a = _run(kda, inp, None)
    b = _run(kda, inp, [7] * 8)
    assert a[3] == 0 and b[3] == 0
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


def test_bad_draft_len_skips_request(kda):
    inp = _inputs(4, 2, 128, [2, 3, 1, 0], 7, seed=50)
    st, tl, o, status = _run(kda, inp, [2, 8, -1, 0])
    assert status & kda.STATUS_BAD_DRAFT_LEN
    for r in (1, 2):
        assert torch.equal(st[r], inp["state"][r])
        assert torch.equal(tl[r], inp["tail"][r])
        assert torch.all(o[r] == -3.0)
    assert not torch.equal(st[0], inp["state"][0])  # valid requests still ran


def test_window_zero_counts(kda):
    """Single-token decode (window 0): counts of 0 are the plain call; any
    other count is rejected per request."""
    inp = _inputs(4, 2, 128, [0] * 4, 0, seed=60)
    a = _run(kda, inp, None)
    b = _run(kda, inp, [0] * 4)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)
    st, tl, o, status = _run(kda, inp, [0, 1, 0, 0])
    assert status & kda.STATUS_BAD_DRAFT_LEN
    assert torch.equal(st[1], inp["state"][1]) and torch.all(o[1] == -3.0)
    assert torch.equal(st[0], a[0][0])


def test_full_ragged_r256_h96(kda, oracle):
    """256 requests x 96 heads, window 7, drafts per request U{3..7} (the
    pages' range) and accepted lengths U{0..7}; padding rows NaN."""
    rng = np.random.default_rng(70)
    R, H, D, Wd = 256, 96, 128, 7
    acc = rng.integers(0, Wd + 1, size=R).tolist()
    d = rng.integers(3, Wd + 1, size=R).tolist()
    inp = _poison(_inputs(R, H, D, acc, Wd, seed=70), d)
    got = _run(kda, inp, d)
    ref = _oracle(oracle, inp, d)
    _check(inp, got, ref, d)
