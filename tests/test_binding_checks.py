"""The Python binding checks dtypes and shapes before anything reaches the C
ABI (which takes bare pointers and cannot).  CPU only: every case is rejected
before a pointer is taken or the library is loaded."""
import pytest
import torch

import kda_gated_delta_02_gb300 as kda


def _prefill(T=70, H=2, d=64, dtype=torch.bfloat16, N=2):
    q = torch.zeros(T, H, d, dtype=dtype)
    return dict(q=q, k=q.clone(), v=q.clone(), g=torch.zeros(T, H, d), beta=torch.zeros(T, H),
                cu=torch.tensor([0, 30, T][:N + 1], dtype=torch.int32), S0=torch.zeros(N, H, d, d))


def _fwd(x, **kw):
    return kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"], **kw)


@pytest.mark.parametrize("key,bad,msg", [
    ("g", lambda x: x["g"].bfloat16(), "g must be"),
    ("v", lambda x: x["v"].float(), "v must be"),
    ("k", lambda x: x["k"][:, :1].contiguous(), "k must have shape"),
    ("beta", lambda x: x["beta"][:-1].contiguous(), "beta must have shape"),
    ("cu", lambda x: x["cu"].long(), "cu_seqlens must be int32"),
    ("S0", lambda x: x["S0"][:1].contiguous(), "initial_state must have shape"),
])
def test_prefill_rejects(key, bad, msg):
    x = _prefill()
    x[key] = bad(x)
    with pytest.raises(kda.KDAError, match=msg):
        _fwd(x)


def test_prefill_rejects_outputs_and_checkpoints():
    x = _prefill()
    with pytest.raises(kda.KDAError, match="out must be"):
        _fwd(x, out=torch.zeros(70, 2, 64))
    with pytest.raises(kda.KDAError, match="final_state must have shape"):
        _fwd(x, final_state=torch.zeros(2, 2, 64, 32))
    with pytest.raises(kda.KDAError, match="ckpt must have shape"):
        _fwd(x, ckpt_every=64, ckpt=torch.zeros(2, 1, 3, 64, 64))
    with pytest.raises(kda.KDAError, match="unsupported input dtype"):
        y = _prefill(dtype=torch.float16)
        _fwd(y)


def test_backward_rejects():
    x = _prefill()
    with pytest.raises(kda.KDAError, match="do must be"):
        kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], torch.zeros(70, 2, 64))
    with pytest.raises(kda.KDAError, match="dS_final must have shape"):
        kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["v"],
                      dS_final=torch.zeros(1, 2, 64, 64))


def test_host_prefill_rejects():
    x = _prefill()
    with pytest.raises(kda.KDAError, match="g must be"):
        kda.chunk_fwd_host(x["q"], x["k"], x["v"], x["g"].double(), x["beta"], x["cu"])
    with pytest.raises(kda.KDAError, match="cu_seqlens must be int32"):
        kda.chunk_fwd_host(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"].float())


def _verify(R=3, H=2, d=64, W=4, Wd=3):
    bf = torch.bfloat16
    Cq = H * 3 * d
    return dict(state=torch.zeros(R, H, d, d, dtype=bf), tail=torch.zeros(R, W - 1, Cq, dtype=bf),
                conv_w=torch.zeros(Cq, W), cq=torch.zeros(R, Wd, Cq, dtype=bf), cg=torch.zeros(R, Wd, H * d, dtype=bf),
                cb=torch.zeros(R, Wd, H, dtype=bf), acc=torch.zeros(R, dtype=torch.int32),
                nq=torch.zeros(R, Wd + 1, Cq, dtype=bf), ng=torch.zeros(R, Wd + 1, H * d, dtype=bf),
                nb=torch.zeros(R, Wd + 1, H, dtype=bf), w=torch.ones(d))


def _call_verify(x, **kw):
    return kda.decode_verify_replay(x["state"], x["tail"], x["conv_w"], x["cq"], x["cg"], x["cb"], x["acc"],
                                    x["nq"], x["ng"], x["nb"], x["w"], **kw)


@pytest.mark.parametrize("key,bad,msg", [
    ("cg", lambda x: x["cg"].float(), "cached_g must be"),
    ("acc", lambda x: x["acc"].long(), "accepted_len must be"),
    ("tail", lambda x: x["tail"][:, :1].contiguous(), "conv_tail must have shape"),
    ("state", lambda x: x["state"].float(), "state must be"),
    ("nb", lambda x: x["nb"][:, :2].contiguous(), "new_beta must have shape"),
    ("w", lambda x: x["w"][:5].contiguous(), "out_norm_w must have shape"),
])
def test_verify_rejects(key, bad, msg):
    x = _verify()
    x[key] = bad(x)
    with pytest.raises(kda.KDAError, match=msg):
        _call_verify(x)


def test_verify_rejects_draft_counts_and_output():
    x = _verify()
    with pytest.raises(kda.KDAError, match="draft_len must have shape"):
        _call_verify(x, draft_len=torch.zeros(2, dtype=torch.int32))
    with pytest.raises(kda.KDAError, match="out must have shape"):
        _call_verify(x, out=torch.zeros(3, 3, 2, 64, dtype=torch.bfloat16))


def test_segment_calls_reject():
    with pytest.raises(kda.KDAError, match="M must have shape"):
        kda.segment_compose(torch.zeros(3, 2, 64, 32), torch.zeros(3, 2, 64, 64))
    with pytest.raises(kda.KDAError, match="S0 must be"):
        kda.segment_compose(torch.zeros(3, 2, 64, 64), torch.zeros(3, 2, 64, 64), S0=torch.zeros(2, 64, 64).double())
    x = _prefill()
    with pytest.raises(kda.KDAError, match="segment_len must be positive"):
        kda.segment_transition(x["k"], x["v"], x["g"], x["beta"], 0)
    with pytest.raises(kda.KDAError, match="beta must be"):
        kda.segment_transition(x["k"], x["v"], x["g"], x["beta"].half(), 64)
