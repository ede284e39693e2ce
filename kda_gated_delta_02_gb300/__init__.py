"""KDA (Kimi Delta Attention) recurrence hot path for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/kda.h`` (``libkda.so``, built
in-tree by ``kda_gated_delta_02_gb300.build``).  Every function marshals
torch tensors into pointers and sizes, passes the current CUDA stream and
checks the returned status; all arithmetic runs in the library's kernels.
There is no CPU fallback: without the compiled library or a CUDA device the
calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

__all__ = ["chunk_fwd", "chunk_fwd_workspace_size", "chunk_fwd_prep_workspace_size", "chunk_fwd_plan", "segment_transition",
           "segment_compose", "decode_verify_replay", "KDAError", "load_library", "library_path",
           "CP_OFF", "CP_ON", "CP_AUTO", "CONV_NONE", "CONV_SILU", "STATUS_BAD_SEQLENS",
           "STATUS_BAD_ACCEPTED_LEN", "STATUS_SEGMENT_OVERFLOW", "STATUS_TIMEOUT", "STATUS_BAD_DRAFT_LEN",
           "KERNEL_FAMILIES", "chunk_bwd", "chunk_fwd_host", "kernel_timing_start",
           "kernel_timing_stop"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libkda.so")
_lock = threading.Lock()
_lib = None

CP_OFF, CP_ON, CP_AUTO = 0, 1, -1
CONV_NONE, CONV_SILU = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1
STATUS_BAD_SEQLENS, STATUS_BAD_ACCEPTED_LEN, STATUS_SEGMENT_OVERFLOW = 1, 2, 4
STATUS_TIMEOUT, STATUS_BAD_DRAFT_LEN = 8, 16


class KDAError(RuntimeError):
    pass


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise KDAError(f"{_LIB_PATH} is missing: run `python -m kda_gated_delta_02_gb300.build` "
                           "(the KDA path has no CPU fallback)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [I]
        lib.kda_version.restype = I
        lib.kda_chunk_fwd.restype = I
        lib.kda_chunk_fwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, F, F, I, I, I, P, S, P, P]
        lib.kda_chunk_fwd_ckpt.restype = I
        lib.kda_chunk_fwd_ckpt.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, F, F, I, I, I, P, S,
                                           I, I, P, P, P]
        lib.kda_chunk_fwd_workspace_size.restype = S
        lib.kda_chunk_fwd_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.kda_chunk_fwd_prep_workspace_size.restype = S
        lib.kda_chunk_fwd_prep_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.kda_chunk_fwd_plan.restype = I
        lib.kda_chunk_fwd_plan.argtypes = [I, I, I, I, I, I, I]
        lib.kda_segment_transition.restype = I
        lib.kda_segment_transition.argtypes = [P, P, P, P, I, I, I, I, I, P, P, F, I, P]
        lib.kda_segment_compose.restype = I
        lib.kda_segment_compose.argtypes = [P, P, P, P, P, I, I, I, I, P]
        lib.kda_chunk_fwd_host.restype = I
        lib.kda_chunk_fwd_host.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, F, F, I, I, P, S, P, P]
        lib.kda_chunk_fwd_host_workspace_size.restype = S
        lib.kda_chunk_fwd_host_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.kda_chunk_bwd.restype = I
        lib.kda_chunk_bwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, F, F, I, P, S, P, P]
        lib.kda_chunk_bwd_cp.restype = I
        lib.kda_chunk_bwd_cp.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, F, F, I, I, I, P, S,
                                         P, P]
        lib.kda_chunk_bwd_cp_workspace_size.restype = S
        lib.kda_chunk_bwd_cp_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.kda_chunk_fwd_train.restype = I
        lib.kda_chunk_fwd_train.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, F, F, I, P, S, P, P]
        lib.kda_chunk_bwd_saved.restype = I
        lib.kda_chunk_bwd_saved.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, P, P, F, F, I, P, S, P,
                                            P]
        lib.kda_chunk_fwd_train_cp.restype = I
        lib.kda_chunk_fwd_train_cp.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, F, F, I, I, I, P, S, P, P]
        lib.kda_chunk_bwd_saved_cp.restype = I
        lib.kda_chunk_bwd_saved_cp.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, P, P, F, F, I, I, I,
                                               P, S, P, P]
        lib.kda_chunk_bwd_workspace_size.restype = S
        lib.kda_chunk_bwd_workspace_size.argtypes = [I, I, I, I, I]
        lib.kda_kernel_timing_start.restype = I
        lib.kda_kernel_timing_start.argtypes = []
        lib.kda_kernel_timing_stop.restype = I
        lib.kda_kernel_timing_stop.argtypes = [P, P, I]
        lib.kda_decode_verify_replay_ragged.restype = I
        lib.kda_decode_verify_replay_ragged.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I,
                                                        F, F, F, F, I, P, P]
        lib.kda_decode_verify_replay.restype = I
        lib.kda_decode_verify_replay.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I,
                                                 F, F, F, F, I, P, P]
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load_library().kda_status_string(rc).decode()
        raise KDAError(f"{what} failed: {msg} ({rc})")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise KDAError("KDA calls take CUDA tensors")
    if not t.is_contiguous():
        raise KDAError("KDA calls take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _hptr(t):
    """Host pointer of a contiguous CPU tensor (for the host-buffer entry point)."""
    if t is None:
        return None
    if t.is_cuda:
        raise KDAError("kda_chunk_fwd_host takes CPU (host) tensors")
    if not t.is_contiguous():
        raise KDAError("KDA calls take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _on(stream):
    """Allocate the tensors a call owns on the stream it launches on.  The
    caching allocator hands a freed block to the next allocation on the stream
    that allocated it without waiting for other streams, so a workspace
    allocated on the current stream but used by kernels on `stream` could be
    reused by the current stream while those kernels still run."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def _in_dtype(t):
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise KDAError(f"unsupported input dtype {t.dtype}")


def _expect(t, name, dtype, shape):
    """The C ABI takes bare pointers, so dtypes and shapes are checked here."""
    if t is None:
        return
    if t.dtype != dtype:
        raise KDAError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise KDAError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_prefill(q, k, v, g, beta, cu_seqlens, initial_state=None, cu_any_int=False):
    """(T, H, dk, dv, N) of a prefill call whose tensors agree in dtype and shape."""
    if q.dim() != 3 or v.dim() != 3:
        raise KDAError("q, k, g must be [T, H, dk] and v [T, H, dv]")
    T, H, dk = q.shape
    dv = v.shape[2]
    _in_dtype(q)
    _expect(k, "k", q.dtype, (T, H, dk))
    _expect(v, "v", q.dtype, (T, H, dv))
    _expect(g, "g", torch.float32, (T, H, dk))
    _expect(beta, "beta", torch.float32, (T, H))
    if cu_seqlens.dim() != 1 or cu_seqlens.shape[0] < 2 or (
            cu_seqlens.dtype != torch.int32 and not (cu_any_int and not cu_seqlens.dtype.is_floating_point)):
        raise KDAError("cu_seqlens must be int32 [N + 1] with N >= 1")
    N = cu_seqlens.shape[0] - 1
    _expect(initial_state, "initial_state", torch.float32, (N, H, dk, dv))
    return T, H, dk, dv, N


def chunk_fwd_workspace_size(N, T, H, dk, dv, cp_mode=CP_AUTO, segment_len=0) -> int:
    return int(load_library().kda_chunk_fwd_workspace_size(N, T, H, dk, dv, cp_mode, segment_len))


def chunk_fwd_prep_workspace_size(N, T, H, dk, dv, cp_mode=CP_AUTO, segment_len=0) -> int:
    return int(load_library().kda_chunk_fwd_prep_workspace_size(N, T, H, dk, dv, cp_mode, segment_len))


def chunk_fwd_plan(N, T, H, dk, dv, cp_mode=CP_AUTO, segment_len=0) -> int:
    return int(load_library().kda_chunk_fwd_plan(N, T, H, dk, dv, cp_mode, segment_len))


def chunk_fwd(q, k, v, g, beta, cu_seqlens, initial_state=None, output_final_state=True, scale=1.0,
              g_min=-5.0, cp_mode=CP_AUTO, segment_len=0, out=None, final_state=None,
              workspace=None, status=None, stream=None, ckpt_every=0, ckpt=None, prep=True):
    """Chunkwise KDA prefill.  q,k,g [T,H,dk]; v [T,H,dv]; beta [T,H];
    cu_seqlens int32 [N+1]; initial_state f32 [N,H,dk,dv] or None.
    Returns (o [T,H,dv] in q's dtype, final_state f32 [N,H,dk,dv] or None).
    With ckpt_every > 0 (a multiple of 64) also writes the state after every
    ckpt_every tokens of each sequence into ckpt f32 [N,K,H,dk,dv] (K = its
    second dimension) through kda_chunk_fwd_ckpt.  With prep (the default) a
    bf16, dk = dv = 128 call gets the workspace of the two-kernel form; a
    caller-provided workspace is used as given when it holds at least the
    context-parallel scratch (kda_chunk_fwd_workspace_size): the library runs
    the two-kernel form in as many pieces as its size requires, or the
    one-kernel form when it holds no piece."""
    T, H, dk, dv, N = _check_prefill(q, k, v, g, beta, cu_seqlens, initial_state)
    _expect(out, "out", q.dtype, (T, H, dv))
    _expect(final_state, "final_state", torch.float32, (N, H, dk, dv))
    if ckpt_every:
        if ckpt is None or ckpt.dim() != 5:
            raise KDAError("ckpt must be an f32 tensor [N, K, H, dk, dv]")
        _expect(ckpt, "ckpt", torch.float32, (N, ckpt.shape[1], H, dk, dv))
    with _on(stream):
        lib = load_library()
        if out is None:
            out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
        if final_state is None and output_final_state:
            final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
        need = chunk_fwd_workspace_size(N, T, H, dk, dv, cp_mode, segment_len)
        if workspace is not None and workspace.numel() * workspace.element_size() >= max(need, 1):
            ws_bytes = workspace.numel() * workspace.element_size()
        else:
            ws_bytes = chunk_fwd_prep_workspace_size(N, T, H, dk, dv, cp_mode, segment_len) \
                if (prep and q.dtype == torch.bfloat16) else need
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
        common = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, dk, dv,
                  _ptr(initial_state), _ptr(final_state), _ptr(out), float(scale), float(g_min),
                  _in_dtype(q), int(cp_mode), int(segment_len),
                  _ptr(workspace) if ws_bytes else None, ctypes.c_size_t(ws_bytes))
        if ckpt_every:
            rc = lib.kda_chunk_fwd_ckpt(*common, int(ckpt_every), int(ckpt.shape[1]), _ptr(ckpt), _ptr(status),
                                        _stream(stream))
            _check(rc, "kda_chunk_fwd_ckpt")
        else:
            rc = lib.kda_chunk_fwd(*common, _ptr(status), _stream(stream))
            _check(rc, "kda_chunk_fwd")
        return out, final_state


def segment_transition(k, v, g, beta, segment_len, g_min=-5.0, stream=None):
    """Transitions (M [P,H,dk,dk], N [P,H,dk,dv]) of fixed-length segments of one sequence."""
    if k.dim() != 3 or v.dim() != 3:
        raise KDAError("k, g must be [T, H, dk] and v [T, H, dv]")
    T, H, dk = k.shape
    dv = v.shape[2]
    _in_dtype(k)
    _expect(v, "v", k.dtype, (T, H, dv))
    _expect(g, "g", torch.float32, (T, H, dk))
    _expect(beta, "beta", torch.float32, (T, H))
    if int(segment_len) < 1:
        raise KDAError("segment_len must be positive")
    with _on(stream):
        lib = load_library()
        P = (T + segment_len - 1) // segment_len
        M = torch.empty((P, H, dk, dk), dtype=torch.float32, device=k.device)
        Nm = torch.empty((P, H, dk, dv), dtype=torch.float32, device=k.device)
        rc = lib.kda_segment_transition(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), T, H, dk, dv, int(segment_len),
                                        _ptr(M), _ptr(Nm), float(g_min), _in_dtype(k), _stream(stream))
        _check(rc, "kda_segment_transition")
        return M, Nm


def segment_compose(M, Nm, S0=None, want_segment_states=True, stream=None):
    """Ordered composition: returns (S_in [P,H,dk,dv] or None, S_final [H,dk,dv])."""
    if Nm.dim() != 4:
        raise KDAError("Nm must be f32 [P, H, dk, dv]")
    P, H, dk, dv = Nm.shape
    _expect(Nm, "Nm", torch.float32, (P, H, dk, dv))
    _expect(M, "M", torch.float32, (P, H, dk, dk))
    _expect(S0, "S0", torch.float32, (H, dk, dv))
    with _on(stream):
        lib = load_library()
        S_in = torch.empty_like(Nm) if want_segment_states else None
        Sf = torch.empty((H, dk, dv), dtype=torch.float32, device=Nm.device)
        rc = lib.kda_segment_compose(_ptr(M), _ptr(Nm), _ptr(S0), _ptr(S_in), _ptr(Sf), P, H, dk, dv,
                                     _stream(stream))
        _check(rc, "kda_segment_compose")
        return S_in, Sf


# kernel families of kda_kernel_timing_stop, in KDA_KERNEL_* order
KERNEL_FAMILIES = ("kda_chunk_list_kernel", "kda_chunk_prep_kernel", "kda_chunk_walk_kernel",
                   "kda_chunk_tc_kernel", "kda_chunk_kernel", "kda_compose_kernel", "kda_segment_table_kernel",
                   "kda_decode_verify_replay", "kda_chunk_bwd_kernel", "kda_bwd_walk_kernel",
                   "kda_bwd_chunk_kernel", "kda_bwd_compose_kernel")


def chunk_fwd_host(q, k, v, g, beta, cu_seqlens, initial_state=None, output_final_state=True, scale=1.0,
                   g_min=-5.0, pieces=4, out=None, final_state=None, workspace=None, status=None, stream=None):
    """chunk_fwd (cp off) on CPU tensors (pin them for asynchronous copies):
    the library copies the inputs in and the outputs out by pieces, overlapped
    with the kernels.  cu_seqlens is a CPU int32 tensor.  Returns CPU tensors
    (o, final_state); they are complete once `stream` (default: the current
    one) has completed."""
    T, H, dk, dv, N = _check_prefill(q, k, v, g, beta, cu_seqlens, initial_state, cu_any_int=True)
    _expect(out, "out", q.dtype, (T, H, dv))
    _expect(final_state, "final_state", torch.float32, (N, H, dk, dv))
    with _on(stream):
        lib = load_library()
        if out is None:
            out = torch.empty((T, H, dv), dtype=q.dtype).pin_memory()
        if final_state is None and output_final_state:
            final_state = torch.empty((N, H, dk, dv), dtype=torch.float32).pin_memory()
        dt = _in_dtype(q)
        need = int(lib.kda_chunk_fwd_host_workspace_size(N, T, H, dk, dv, dt, int(pieces)))
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        cu = cu_seqlens.to(torch.int32).contiguous()
        rc = lib.kda_chunk_fwd_host(_hptr(q), _hptr(k), _hptr(v), _hptr(g), _hptr(beta), _hptr(cu), N, T, H, dk, dv,
                                    _hptr(initial_state), _hptr(final_state), _hptr(out), float(scale), float(g_min), dt,
                                    int(pieces), _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                    _ptr(status), _stream(stream))
        _check(rc, "kda_chunk_fwd_host")
        return out, final_state


def chunk_bwd(q, k, v, g, beta, cu_seqlens, do, initial_state=None, dS_final=None, scale=1.0, g_min=-5.0,
              workspace=None, status=None, stream=None, want_dS0=True):
    """Backward of chunk_fwd: returns (dq, dk, dv, dg, dbeta, dS0) in fp32
    (dS0 None unless want_dS0).  do [T,H,dv] in q's dtype; dS_final f32
    [N,H,dk,dv] or None."""
    T, H, dk, dv, N = _check_prefill(q, k, v, g, beta, cu_seqlens, initial_state)
    _expect(do, "do", q.dtype, (T, H, dv))
    _expect(dS_final, "dS_final", torch.float32, (N, H, dk, dv))
    with _on(stream):
        lib = load_library()
        dev = q.device
        f32 = torch.float32
        dq = torch.empty((T, H, dk), dtype=f32, device=dev)
        dkk = torch.empty((T, H, dk), dtype=f32, device=dev)
        dvv = torch.empty((T, H, dv), dtype=f32, device=dev)
        dg = torch.empty((T, H, dk), dtype=f32, device=dev)
        db = torch.empty((T, H), dtype=f32, device=dev)
        dS0 = torch.empty((N, H, dk, dv), dtype=f32, device=dev) if want_dS0 else None
        need = int(lib.kda_chunk_bwd_workspace_size(N, T, H, dk, dv))
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        rc = lib.kda_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, dk, dv,
                               _ptr(initial_state), _ptr(do), _ptr(dS_final), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg),
                               _ptr(db), _ptr(dS0), float(scale), float(g_min), _in_dtype(q), _ptr(workspace),
                               ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(status),
                               _stream(stream))
        _check(rc, "kda_chunk_bwd")
        return dq, dkk, dvv, dg, db, dS0


def chunk_bwd_cp(q, k, v, g, beta, cu_seqlens, do, initial_state=None, dS_final=None, scale=1.0, g_min=-5.0,
                 cp_mode=None, segment_len=0, workspace=None, status=None, stream=None, want_dS0=True):
    """chunk_bwd with the prefill's context-parallel schedule for long
    sequences (cp_mode and segment_len as chunk_fwd; default: automatic)."""
    T, H, dk, dv, N = _check_prefill(q, k, v, g, beta, cu_seqlens, initial_state)
    _expect(do, "do", q.dtype, (T, H, dv))
    _expect(dS_final, "dS_final", torch.float32, (N, H, dk, dv))
    cp = CP_AUTO if cp_mode is None else int(cp_mode)
    with _on(stream):
        lib = load_library()
        dev = q.device
        f32 = torch.float32
        dq = torch.empty((T, H, dk), dtype=f32, device=dev)
        dkk = torch.empty((T, H, dk), dtype=f32, device=dev)
        dvv = torch.empty((T, H, dv), dtype=f32, device=dev)
        dg = torch.empty((T, H, dk), dtype=f32, device=dev)
        db = torch.empty((T, H), dtype=f32, device=dev)
        dS0 = torch.empty((N, H, dk, dv), dtype=f32, device=dev) if want_dS0 else None
        need = int(lib.kda_chunk_bwd_cp_workspace_size(N, T, H, dk, dv, cp, int(segment_len)))
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        rc = lib.kda_chunk_bwd_cp(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, dk, dv,
                                  _ptr(initial_state), _ptr(do), _ptr(dS_final), _ptr(dq), _ptr(dkk), _ptr(dvv),
                                  _ptr(dg), _ptr(db), _ptr(dS0), float(scale), float(g_min), _in_dtype(q), cp,
                                  int(segment_len), _ptr(workspace),
                                  ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(status),
                                  _stream(stream))
        _check(rc, "kda_chunk_bwd_cp")
        return dq, dkk, dvv, dg, db, dS0


def chunk_fwd_train(q, k, v, g, beta, cu_seqlens, initial_state=None, scale=1.0, g_min=-5.0, saved=None,
                    status=None, stream=None, cp_mode=None, segment_len=0):
    """The forward of the training pair (d = 128, bf16): returns (o,
    final_state, saved); `saved` (uint8, device) holds what chunk_bwd_saved
    needs.  o and final_state equal chunk_fwd's bit for bit.  With cp_mode
    (and segment_len) given, the pair of chunk_bwd_cp's schedule: pass the
    same values to chunk_bwd_saved."""
    T, H, dk, dv, N = _check_prefill(q, k, v, g, beta, cu_seqlens, initial_state)
    with _on(stream):
        lib = load_library()
        o = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
        Sf = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
        if cp_mode is None:
            need = int(lib.kda_chunk_bwd_workspace_size(N, T, H, dk, dv))
        else:
            need = int(lib.kda_chunk_bwd_cp_workspace_size(N, T, H, dk, dv, int(cp_mode), int(segment_len)))
        if saved is None or saved.numel() * saved.element_size() < need:
            saved = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, dk, dv,
                _ptr(initial_state), _ptr(Sf), _ptr(o), float(scale), float(g_min), _in_dtype(q))
        tail = (_ptr(saved), ctypes.c_size_t(saved.numel() * saved.element_size()), _ptr(status), _stream(stream))
        if cp_mode is None:
            rc = lib.kda_chunk_fwd_train(*head, *tail)
            _check(rc, "kda_chunk_fwd_train")
        else:
            rc = lib.kda_chunk_fwd_train_cp(*head, int(cp_mode), int(segment_len), *tail)
            _check(rc, "kda_chunk_fwd_train_cp")
        return o, Sf, saved


def chunk_bwd_saved(q, k, v, g, beta, cu_seqlens, do, saved, dS_final=None, scale=1.0, g_min=-5.0, status=None,
                    stream=None, want_dS0=True, cp_mode=None, segment_len=0):
    """The backward of the training pair: the reverse pass over `saved` from
    chunk_fwd_train (same inputs, scale, g_min, cp_mode and segment_len).
    Returns (dq, dk, dv, dg, dbeta, dS0) as chunk_bwd (chunk_bwd_cp with
    cp_mode) does, bit for bit."""
    T, H, dk, dv, N = _check_prefill(q, k, v, g, beta, cu_seqlens, None)
    _expect(do, "do", q.dtype, (T, H, dv))
    _expect(dS_final, "dS_final", torch.float32, (N, H, dk, dv))
    with _on(stream):
        lib = load_library()
        dev = q.device
        f32 = torch.float32
        dq = torch.empty((T, H, dk), dtype=f32, device=dev)
        dkk = torch.empty((T, H, dk), dtype=f32, device=dev)
        dvv = torch.empty((T, H, dv), dtype=f32, device=dev)
        dg = torch.empty((T, H, dk), dtype=f32, device=dev)
        db = torch.empty((T, H), dtype=f32, device=dev)
        dS0 = torch.empty((N, H, dk, dv), dtype=f32, device=dev) if want_dS0 else None
        head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, dk, dv, _ptr(do),
                _ptr(dS_final), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg), _ptr(db), _ptr(dS0), float(scale),
                float(g_min), _in_dtype(q))
        tail = (_ptr(saved), ctypes.c_size_t(saved.numel() * saved.element_size()), _ptr(status), _stream(stream))
        if cp_mode is None:
            rc = lib.kda_chunk_bwd_saved(*head, *tail)
            _check(rc, "kda_chunk_bwd_saved")
        else:
            rc = lib.kda_chunk_bwd_saved_cp(*head, int(cp_mode), int(segment_len), *tail)
            _check(rc, "kda_chunk_bwd_saved_cp")
        return dq, dkk, dvv, dg, db, dS0


def kernel_timing_start():
    """Record CUDA events around every library launch from now on."""
    _check(load_library().kda_kernel_timing_start(), "kda_kernel_timing_start")


def kernel_timing_stop():
    """Stop recording; {family: {"launches": n, "ms": summed device time}} for
    the families that launched (waits for the recorded events)."""
    n = len(KERNEL_FAMILIES)
    launches = (ctypes.c_int * n)()
    total = (ctypes.c_float * n)()
    _check(load_library().kda_kernel_timing_stop(launches, total, n), "kda_kernel_timing_stop")
    return {KERNEL_FAMILIES[i]: {"launches": int(launches[i]), "ms": float(total[i])}
            for i in range(n) if launches[i] > 0}


def decode_verify_replay(state, conv_tail, conv_w, cached_qkv, cached_g, cached_beta, accepted_len,
                         new_qkv, new_g, new_beta, out_norm_w, scale=1.0, g_min=-5.0, eps_in=1e-6,
                         eps_out=1e-6, conv_act=CONV_SILU, out=None, status=None, stream=None, draft_len=None):
    """Fused verify with replay.  Updates state and conv_tail in place; returns
    o [R, Wd+1, H, dv] (bf16): rows for the bonus token and the next drafts.
    draft_len (int32 [R] on the device) makes the batch ragged: request r has
    draft_len[r] drafts (kda_decode_verify_replay_ragged); its rows past that
    are not written."""
    if state.dim() != 4 or conv_w.dim() != 2 or new_qkv.dim() != 3:
        raise KDAError("state [R, H, dk, dv], conv_w [Cq, W] and new_qkv [R, Wd + 1, Cq] expected")
    R, H, dk, dv = state.shape
    W = conv_w.shape[1]
    Wd = new_qkv.shape[1] - 1
    Cq = H * (2 * dk + dv)
    bf = torch.bfloat16
    _expect(state, "state", bf, (R, H, dk, dv))
    _expect(conv_tail, "conv_tail", bf, (R, W - 1, Cq))
    _expect(conv_w, "conv_w", torch.float32, (Cq, W))
    _expect(cached_qkv, "cached_qkv", bf, (R, Wd, Cq))
    _expect(cached_g, "cached_g", bf, (R, Wd, H * dk))
    _expect(cached_beta, "cached_beta", bf, (R, Wd, H))
    _expect(accepted_len, "accepted_len", torch.int32, (R,))
    _expect(new_qkv, "new_qkv", bf, (R, Wd + 1, Cq))
    _expect(new_g, "new_g", bf, (R, Wd + 1, H * dk))
    _expect(new_beta, "new_beta", bf, (R, Wd + 1, H))
    _expect(out_norm_w, "out_norm_w", torch.float32, (dv,))
    _expect(out, "out", bf, (R, Wd + 1, H, dv))
    _expect(draft_len, "draft_len", torch.int32, (R,))
    with _on(stream):
        lib = load_library()
        if out is None:
            out = torch.empty((R, Wd + 1, H, dv), dtype=torch.bfloat16, device=state.device)
        if draft_len is not None:
            rc = lib.kda_decode_verify_replay_ragged(
                _ptr(state), _ptr(conv_tail), _ptr(conv_w), _ptr(cached_qkv), _ptr(cached_g), _ptr(cached_beta),
                _ptr(accepted_len), _ptr(draft_len), _ptr(new_qkv), _ptr(new_g), _ptr(new_beta), _ptr(out_norm_w),
                _ptr(out), R, H, dk, dv, W, Wd, float(scale), float(g_min), float(eps_in), float(eps_out),
                int(conv_act), _ptr(status), _stream(stream))
            _check(rc, "kda_decode_verify_replay_ragged")
            return out
        rc = lib.kda_decode_verify_replay(_ptr(state), _ptr(conv_tail), _ptr(conv_w), _ptr(cached_qkv),
                                          _ptr(cached_g), _ptr(cached_beta), _ptr(accepted_len), _ptr(new_qkv),
                                          _ptr(new_g), _ptr(new_beta), _ptr(out_norm_w), _ptr(out), R, H, dk, dv,
                                          W, Wd, float(scale), float(g_min), float(eps_in), float(eps_out),
                                          int(conv_act), _ptr(status), _stream(stream))
        _check(rc, "kda_decode_verify_replay")
        return out
