"""Bounded waits of the tensor-core kernels, exercised through a test build.

Every wait of the library's tcgen05 kernels on an mbarrier (for a TMA copy or
a tensor-core product) gives up after a bounded number of polls; the kernel
then sets KDA_STATUS_TIMEOUT in the caller's status word, waits (bounded) for
every copy and product it issued, frees its tensor memory and returns, so the
context stays usable.  A test build of the library (libkda_shortwait.so,
compiled with KDA_TEST_SHORT_FIRST_WAIT) gives up on one wait at once: the
state walk's wait for its first chunk's operand copy (a copy in flight), the
verify kernel's wait for its first batch of products (products in flight),
and in the backward the reverse walk's wait for its first chunk's copies and
the chunk-gradient kernel's wait for its first item's copies.  These tests call that build through the C ABI, check the status
word, synchronise (no fault), and then check that the library's ordinary calls
on the same inputs still match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity import OUT_TOL, STATE_TOL, normwise_err, to64

pytestmark = pytest.mark.gpu

STATUS_TIMEOUT = 8


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from kda_gated_delta_02_gb300 import build
    import kda_gated_delta_02_gb300 as kda
    path = build.build_variant("shortwait", ["KDA_TEST_SHORT_FIRST_WAIT"])
    test_lib = ctypes.CDLL(path)
    main = kda.load_library()
    for name in ("kda_chunk_fwd", "kda_decode_verify_replay", "kda_chunk_bwd", "kda_chunk_bwd_workspace_size"):
        getattr(test_lib, name).restype = getattr(main, name).restype
        getattr(test_lib, name).argtypes = getattr(main, name).argtypes
    return kda, test_lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_walk_copy_timeout_drains_and_reports(libs, oracle):
    kda, test_lib = libs
    gen = torch.Generator().manual_seed(11)
    lens, H, d = [300, 200], 2, 128
    T = sum(lens)
    q = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).bfloat16().cuda()
    k = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).bfloat16().cuda()
    v = torch.randn(T, H, d, generator=gen).bfloat16().cuda()
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, d, generator=gen)), -5.0).cuda()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).cuda()
    cu = torch.tensor([0, lens[0], T], dtype=torch.int32).cuda()
    o = torch.zeros(T, H, d, dtype=torch.bfloat16, device="cuda")
    Sf = torch.zeros(2, H, d, d, dtype=torch.float32, device="cuda")
    ws_bytes = kda.chunk_fwd_prep_workspace_size(2, T, H, d, d, kda.CP_OFF)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = test_lib.kda_chunk_fwd(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu), 2, T, H, d, d, None, _p(Sf), _p(o),
                                1.0, -5.0, 0, kda.CP_OFF, 0, _p(ws), ctypes.c_size_t(ws_bytes), _p(status),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()  # the kernels returned: nothing left running
    assert int(status.item()) & STATUS_TIMEOUT
    # the ordinary library on the same inputs
    o2, S2 = kda.chunk_fwd(q, k, v, g, beta, cu)
    torch.cuda.synchronize()
    o_r, S_r = oracle.prefill(to64(q), to64(k), to64(v), to64(g), to64(beta), cu.cpu().numpy())
    assert normwise_err(to64(o2), o_r, head_axis=1) <= OUT_TOL
    assert normwise_err(to64(S2), S_r, head_axis=1) <= STATE_TOL


def test_verify_product_timeout_drains_and_reports(libs, oracle):
    kda, test_lib = libs
    from kda_gated_delta_02_gb300 import synth
    dw = synth.DecodeWorkload("timeout", 4, 2, 128, 128, seed=12)
    dd = synth.make_decode(dw, device="cuda", accepted=[0, 3, 7, 5])
    st, tl = dd["state"].clone(), dd["tail"].clone()
    R, H, D = 4, 2, 128
    o = torch.zeros((R, dw.Wd + 1, H, D), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = test_lib.kda_decode_verify_replay(
        _p(st), _p(tl), _p(dd["conv_w"]), _p(dd["cached_qkv"]), _p(dd["cached_g"]), _p(dd["cached_b"]),
        _p(dd["accepted"]), _p(dd["new_qkv"]), _p(dd["new_g"]), _p(dd["new_b"]), _p(dd["out_w"]), _p(o), R, H, D, D,
        dw.W, dw.Wd, 1.0, -5.0, 1e-6, 1e-6, kda.CONV_SILU, _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) & STATUS_TIMEOUT
    assert torch.equal(st, dd["state"])  # no state was written back
    # the ordinary library on the same inputs
    st2, tl2 = dd["state"].clone(), dd["tail"].clone()
    o2 = kda.decode_verify_replay(st2, tl2, dd["conv_w"], dd["cached_qkv"], dd["cached_g"], dd["cached_b"],
                                  dd["accepted"], dd["new_qkv"], dd["new_g"], dd["new_b"], dd["out_w"])
    torch.cuda.synchronize()
    st_r, tl_r, o_r, _ = oracle.decode_verify(to64(dd["state"]), to64(dd["tail"]), to64(dd["conv_w"]),
                                              to64(dd["cached_qkv"]), to64(dd["cached_g"]), to64(dd["cached_b"]),
                                              dd["accepted"].cpu().numpy(), to64(dd["new_qkv"]), to64(dd["new_g"]),
                                              to64(dd["new_b"]), to64(dd["out_w"]))
    assert normwise_err(to64(o2), o_r, head_axis=2) <= OUT_TOL
    assert normwise_err(to64(st2), st_r, head_axis=1) <= STATE_TOL
    assert torch.equal(tl2.cpu(), torch.from_numpy(tl_r).to(torch.bfloat16))


def test_backward_copy_timeouts_drain_and_report(libs, oracle):
    """The tensor-core backward (d = 128, bf16): the reverse walk and the chunk
    kernel give up on their first copy; the call reports KDA_STATUS_TIMEOUT
    and leaves nothing running; the ordinary library then matches the oracle."""
    kda, test_lib = libs
    gen = torch.Generator().manual_seed(13)
    lens, H, d = [300, 150], 2, 128
    T = sum(lens)
    q = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).bfloat16().cuda()
    k = torch.nn.functional.normalize(torch.randn(T, H, d, generator=gen), dim=-1).bfloat16().cuda()
    v = torch.randn(T, H, d, generator=gen).bfloat16().cuda()
    g = torch.clamp_min(-torch.nn.functional.softplus(torch.randn(T, H, d, generator=gen)), -5.0).cuda()
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).cuda()
    do = torch.randn(T, H, d, generator=gen).bfloat16().cuda()
    cu = torch.tensor([0, lens[0], T], dtype=torch.int32).cuda()
    outs = [torch.zeros(T, H, d, device="cuda") for _ in range(4)] + [torch.zeros(T, H, device="cuda")]
    dS0 = torch.zeros(2, H, d, d, device="cuda")
    ws_bytes = int(test_lib.kda_chunk_bwd_workspace_size(2, T, H, d, d))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = test_lib.kda_chunk_bwd(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu), 2, T, H, d, d, None, _p(do), None,
                                *[_p(o) for o in outs], _p(dS0), 1.0, -5.0, 0, _p(ws), ctypes.c_size_t(ws_bytes),
                                _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()  # the kernels returned: nothing left running
    assert int(status.item()) & STATUS_TIMEOUT
    # the ordinary library on the same inputs
    got = kda.chunk_bwd(q, k, v, g, beta, cu, do)
    torch.cuda.synchronize()
    ref = oracle.backward(to64(q), to64(k), to64(v), to64(g), to64(beta), cu.cpu().numpy(), to64(do))
    for a, b in zip(got[:5], ref[:5]):
        if b.ndim == 2:
            assert np.max(np.abs(to64(a) - b)) <= 1e-2 * max(np.max(np.abs(b)), 1e-30)
        else:
            assert normwise_err(to64(a), b, head_axis=1) <= 1e-2
