"""kda_chunk_fwd_host: the prefill on host buffers with transfers overlapped
with the kernels gives the device call's results bit for bit (any number of
pieces; the non-pipelined shapes too), and checks cu_seqlens on the host."""
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


def _host_inputs(lens, H, d, dtype, seed):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).to(dtype)
    v = torch.randn(T, H, d, generator=gen).to(dtype)
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, d, generator=gen)), -5.0)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen))
    S0 = 0.02 * torch.randn(len(lens), H, d, d, generator=gen)
    pin = lambda x: x.contiguous().pin_memory()
    return dict(q=pin(q), k=pin(k), v=pin(v), g=pin(g), beta=pin(beta), cu=cu, S0=pin(S0))


def _device_ref(kda, x):
    d = {k_: v_.cuda() for k_, v_ in x.items()}
    o, Sf = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], initial_state=d["S0"], cp_mode=0)
    torch.cuda.synchronize()
    return o.cpu(), Sf.cpu()


@pytest.mark.parametrize("pieces", [1, 3, 7])
def test_host_pipeline_equals_device_call(kda, pieces):
    x = _host_inputs([1000, 130, 0, 640, 1], 4, 128, torch.bfloat16, seed=pieces)
    o, Sf = kda.chunk_fwd_host(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"],
                               pieces=pieces)
    torch.cuda.current_stream().synchronize()
    o_ref, Sf_ref = _device_ref(kda, x)
    assert torch.equal(o, o_ref)
    assert torch.equal(Sf, Sf_ref)


def test_host_fallback_shapes(kda):
    """f32 inputs, d = 64: copied in, one device call, copied out."""
    x = _host_inputs([300, 77], 3, 64, torch.float32, seed=11)
    o, Sf = kda.chunk_fwd_host(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], initial_state=x["S0"])
    torch.cuda.current_stream().synchronize()
    o_ref, Sf_ref = _device_ref(kda, x)
    assert torch.equal(o, o_ref)
    assert torch.equal(Sf, Sf_ref)


def test_host_rejects_bad_seqlens(kda):
    x = _host_inputs([64, 64], 1, 128, torch.bfloat16, seed=12)
    bad = torch.tensor([0, 100, 64], dtype=torch.int32)
    with pytest.raises(kda.KDAError):
        kda.chunk_fwd_host(x["q"], x["k"], x["v"], x["g"], x["beta"], bad)
