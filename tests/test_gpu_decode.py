"""GPU parity of kda_decode_verify_replay against the fp64 oracle.

Bars: output rows (bonus + drafts) 2e-2 and written-back bf16 state 1e-2
normwise relative error per head; conv-tail write-back, skipped requests and
untouched buffers bit-exact; the device status word exact.
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


def gpu_inputs(R, H, D, accepted, seed=0, Wd=7, W=4):
    from kda_gated_delta_02_gb300 import synth
    w = synth.DecodeWorkload("test", R, H, D, D, W=W, Wd=Wd, seed=seed)
    return synth.make_decode(w, device="cuda", accepted=accepted)


def run_both(kda, oracle, inp, conv_act=1, scale=1.0):
    st = inp["state"].clone()
    tl = inp["tail"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    R, H, D, _ = st.shape
    Wd = inp["new_qkv"].shape[1] - 1
    o = torch.full((R, Wd + 1, H, D), -3.0, dtype=torch.bfloat16, device="cuda")
    kda.decode_verify_replay(st, tl, inp["conv_w"], inp["cached_qkv"], inp["cached_g"], inp["cached_b"],
                             inp["accepted"], inp["new_qkv"], inp["new_g"], inp["new_b"], inp["out_w"],
                             scale=scale, conv_act=conv_act, out=o, status=status)
    torch.cuda.synchronize()
    ref = oracle.decode_verify(to64(inp["state"]), to64(inp["tail"]), to64(inp["conv_w"]),
                               to64(inp["cached_qkv"]), to64(inp["cached_g"]), to64(inp["cached_b"]),
                               inp["accepted"].cpu().numpy(), to64(inp["new_qkv"]), to64(inp["new_g"]),
                               to64(inp["new_b"]), to64(inp["out_w"]), conv_act=conv_act, scale=scale)
    return (st, tl, o, int(status.item())), ref


def compare(inp, got, ref, check_rows=None):
    st, tl, o, status = got
    st_r, tl_r, o_r, bad = ref
    acc = inp["accepted"].cpu().numpy()
    good = np.nonzero((acc >= 0) & (acc <= inp["new_qkv"].shape[1] - 1))[0]
    e_o = normwise_err(to64(o)[good], o_r[good], head_axis=2)
    e_s = normwise_err(to64(st)[good], st_r[good], head_axis=1)
    assert e_o <= OUT_TOL, f"output error {e_o:.3e}"
    assert e_s <= STATE_TOL, f"state error {e_s:.3e}"
    # conv tail: bitwise copies of bf16 rows
    tl_ref = torch.from_numpy(tl_r).to(torch.bfloat16)
    assert torch.equal(tl.cpu(), tl_ref), "conv tail write-back is not bit-exact"
    return e_o, e_s


@pytest.mark.parametrize("conv_act", [0, 1])
@pytest.mark.parametrize("D", [128, 64])
def test_every_accepted_length(kda, oracle, D, conv_act):
    inp = gpu_inputs(8, 3, D, accepted=list(range(8)), seed=D + conv_act)
    got, ref = run_both(kda, oracle, inp, conv_act=conv_act)
    assert got[3] == 0 and ref[3] == 0
    compare(inp, got, ref)


def test_scale_and_random_lengths(kda, oracle):
    inp = gpu_inputs(16, 4, 128, accepted=None, seed=5)
    got, ref = run_both(kda, oracle, inp, scale=0.125)
    compare(inp, got, ref)


def test_shorter_window_and_conv(kda, oracle):
    """Draft window 3 and conv width 2 (non-default sizes)."""
    inp = gpu_inputs(6, 2, 128, accepted=[0, 1, 2, 3, 3, 0], seed=6, Wd=3, W=2)
    got, ref = run_both(kda, oracle, inp)
    compare(inp, got, ref)


def test_invalid_accepted_length_skips_request(kda, oracle):
    inp = gpu_inputs(4, 2, 128, accepted=[2, 9, -1, 7], seed=7)
    got, ref = run_both(kda, oracle, inp)
    st, tl, o, status = got
    assert status & kda.STATUS_BAD_ACCEPTED_LEN
    assert ref[3] == 2
    for r in (1, 2):
        assert torch.equal(st[r], inp["state"][r])
        assert torch.equal(tl[r], inp["tail"][r])
        assert torch.all(o[r] == -3.0)
    compare(inp, got, ref)


def test_two_steps_with_buffer_swap(kda, oracle):
    """Step 2 replays step 1's draft rows: cached <- new[:, 1:]."""
    inp = gpu_inputs(8, 2, 128, accepted=[7, 0, 3, 5, 1, 6, 2, 4], seed=8)
    got1, ref1 = run_both(kda, oracle, inp)
    compare(inp, got1, ref1)
    nxt = gpu_inputs(8, 2, 128, accepted=[3, 7, 0, 1, 6, 2, 5, 4], seed=9)
    nxt["state"] = got1[0]
    nxt["tail"] = got1[1]
    nxt["conv_w"], nxt["out_w"] = inp["conv_w"], inp["out_w"]
    nxt["cached_qkv"] = inp["new_qkv"][:, 1:].contiguous()
    nxt["cached_g"] = inp["new_g"][:, 1:].contiguous()
    nxt["cached_b"] = inp["new_b"][:, 1:].contiguous()
    got2, ref2 = run_both(kda, oracle, nxt)
    compare(nxt, got2, ref2)


def test_full_verify_r256_h96(kda, oracle):
    """256 requests, 1 layer, H=96, dk=dv=128, W=4, window 7, accepted ~ U{0..7}."""
    from kda_gated_delta_02_gb300 import synth
    inp = synth.make_decode(synth.VERIFY, device="cuda")
    got, ref = run_both(kda, oracle, inp)
    assert got[3] == 0
    compare(inp, got, ref)


@pytest.mark.parametrize("D", [128, 64])
def test_single_token_decode_chain(kda, oracle, D):
    """Non-speculative decode: window 0, accepted 0, one token per request per
    step; three steps chained through the written-back state and conv tail."""
    R, H = 8, 3
    inp = gpu_inputs(R, H, D, accepted=[0] * R, seed=20 + D, Wd=0)
    assert inp["new_qkv"].shape[1] == 1 and inp["cached_qkv"].shape[1] == 0
    for step in range(3):
        got, ref = run_both(kda, oracle, inp)
        assert got[3] == 0 and ref[3] == 0
        compare(inp, got, ref)
        nxt = gpu_inputs(R, H, D, accepted=[0] * R, seed=30 + 10 * step + D, Wd=0)
        nxt["state"], nxt["tail"] = got[0], got[1]
        nxt["conv_w"], nxt["out_w"] = inp["conv_w"], inp["out_w"]
        inp = nxt
