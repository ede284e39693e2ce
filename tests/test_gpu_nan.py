"""A NaN log-decay takes the floor on the GPU as in the oracle (the floor is
an IEEE maximum, which returns the non-NaN operand): every entry point gives
the same bits with NaN as with g = g_min at those positions (verify: with a
raw gate of +inf), and the prefill with NaN inputs still matches the oracle."""
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


def _case(lens, H, d, dtype, seed):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    v = torch.randn(T, H, d, generator=gen).to(dtype)
    g = -torch.nn.functional.softplus(torch.randn(T, H, d, generator=gen))
    nan = torch.rand(T, H, d, generator=gen) < 0.1
    g_nan, g_flr = g.clone(), g.clone()
    g_nan[nan] = float("nan")
    g_flr[nan] = -5.0
    beta = torch.sigmoid(torch.randn(T, H, generator=gen))
    S0 = 0.05 * torch.randn(len(lens), H, d, d, generator=gen)
    do = torch.randn(T, H, d, generator=gen).to(dtype)
    c = lambda x: x.cuda()
    return dict(q=c(q), k=c(k), v=c(v), g_nan=c(g_nan), g_flr=c(g_flr), beta=c(beta), cu=c(cu), S0=c(S0),
                do=c(do))


@pytest.mark.parametrize("d,dtype,cp", [(128, torch.bfloat16, 0), (128, torch.bfloat16, 1), (64, torch.float32, 0)])
def test_prefill_nan_log_decay_takes_the_floor(kda, oracle, d, dtype, cp):
    x = _case([700, 0, 330], 2, d, dtype, seed=101 + d + cp)
    run = lambda g: kda.chunk_fwd(x["q"], x["k"], x["v"], g, x["beta"], x["cu"], initial_state=x["S0"],
                                  scale=0.6, cp_mode=cp, segment_len=256 if cp else 0)
    o_n, S_n = run(x["g_nan"])
    o_f, S_f = run(x["g_flr"])
    torch.cuda.synchronize()
    assert torch.equal(o_n, o_f) and torch.equal(S_n, S_f)
    ref_o, ref_S = oracle.prefill(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["g_nan"]), to64(x["beta"]),
                                  x["cu"].cpu().numpy(), S0=to64(x["S0"]), scale=0.6)
    assert normwise_err(to64(o_n), ref_o, head_axis=1) <= OUT_TOL
    assert normwise_err(to64(S_n), ref_S, head_axis=1) <= STATE_TOL


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_backward_nan_log_decay_takes_the_floor(kda, d, dtype):
    """dg at a NaN position is that of g = g_min (the floor passes its
    gradient); every other gradient is unchanged, bit for bit."""
    x = _case([300, 200], 2, d, dtype, seed=107 + d)
    run = lambda g: kda.chunk_bwd(x["q"], x["k"], x["v"], g, x["beta"], x["cu"], x["do"], initial_state=x["S0"],
                                  scale=0.8)
    a, b = run(x["g_nan"]), run(x["g_flr"])
    torch.cuda.synchronize()
    for u, w in zip(a, b):
        assert torch.equal(u, w)
        assert bool(torch.all(torch.isfinite(u)))


@pytest.mark.parametrize("Wd", [7, 0])
def test_verify_nan_gate_takes_the_floor(kda, Wd):
    from kda_gated_delta_02_gb300 import synth
    w = synth.DecodeWorkload("nan gate", 8, 4, 128, 128, Wd=Wd, seed=109)
    d = synth.make_decode(w, device="cuda", accepted=None if Wd else [0] * 8)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(113)
    outs = []
    for fill in (float("nan"), float("inf")):
        e = dict(d)
        for key in ("cached_g", "new_g"):
            m = (torch.rand(d[key].shape, generator=gen) < 0.3).cuda()
            e[key] = torch.where(m, torch.tensor(fill, dtype=torch.bfloat16, device="cuda"), d[key])
        gen.manual_seed(113)
        st, tl = d["state"].clone(), d["tail"].clone()
        o = kda.decode_verify_replay(st, tl, e["conv_w"], e["cached_qkv"], e["cached_g"], e["cached_b"],
                                     e["accepted"], e["new_qkv"], e["new_g"], e["new_b"], e["out_w"])
        outs.append((o, st, tl))
    torch.cuda.synchronize()
    for u, w in zip(*outs):
        assert torch.equal(u, w)
