"""fp64 CPU oracle for the KDA recurrence (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA path never imports it and shares no
code with it.  The arithmetic lives in ``kda_oracle.c`` (plain C, fp64); this
module compiles it with gcc on first use and wraps it with ctypes/numpy.

Functions and what they follow (page title, section):

* ``prefill`` -- gated delta rule, token by token ("Noyaux KDA et FlashKDA",
  "Le conflit fondamental"; decay floor from "Le role de la decroissance
  bornee").
* ``segment_transition`` / ``segment_compose`` -- affine segment transitions
  and their exact composition ("Noyaux KDA et FlashKDA", "Le parallelisme de
  contexte intra-appareil"; "Dentro de los esfuerzos de optimizacion de Kimi
  K3", section 5).
* ``unit_lower_inverse`` / ``chunk_form_head`` -- the intra-chunk dependency
  inverse and the chunk (WY) form ("Dentro de los esfuerzos...", "Nota
  tecnica: Precision del KDA y memoria on-chip").
* ``decode_verify`` / ``decode_stepwise`` -- replay-based verify and the plain
  one-token-at-a-time decoder it must agree with ("Noyaux d'inference",
  section 1, "La solution : rejouer plutot que sauvegarder", "La fusion").
* ``backward`` -- reverse mode of the token recurrence (training, the chunk
  kernel's other use: "Noyaux KDA et FlashKDA", "FlashKDA : le noyau par
  blocs"); the module ``chunk_reverse`` states the same backward in the
  chunk (WY) form, pinned against it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP if available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_max_threads.restype = I
            lib.oracle_kda_prefill.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, D, D, I, P, I]
            lib.oracle_kda_prefill.restype = I
            lib.oracle_segment_transition.argtypes = [I, I, I, I, P, P, P, P, D, P, P, I]
            lib.oracle_segment_transition.restype = I
            lib.oracle_segment_compose.argtypes = [I, I, I, I, P, P, P, P, P]
            lib.oracle_segment_compose.restype = I
            lib.oracle_unit_lower_inverse.argtypes = [I, P, P]
            lib.oracle_unit_lower_inverse.restype = I
            lib.oracle_chunk_form_head.argtypes = [I, I, I, I, P, P, P, P, P, P, P, D, D]
            lib.oracle_chunk_form_head.restype = I
            vargs = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, D, D, I, P, D, D]
            lib.oracle_kda_backward.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, D, D,
                                                I]
            lib.oracle_kda_backward.restype = I
            lib.oracle_decode_verify.argtypes = vargs + [I]
            lib.oracle_decode_verify.restype = I
            lib.oracle_decode_verify_ragged.argtypes = vargs[:13] + [P] + vargs[13:] + [I]
            lib.oracle_decode_verify_ragged.restype = I
            lib.oracle_decode_stepwise.argtypes = vargs
            lib.oracle_decode_stepwise.restype = I
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def prefill(q, k, v, g, beta, cu_seqlens, S0=None, scale=1.0, g_min=-5.0, erase=True,
            head_mask=None, nthreads=0):
    """Token-by-token gated delta rule.  Shapes: q,k,g [T,H,dk]; v [T,H,dv];
    beta [T,H]; cu_seqlens [N+1]; S0 [N,H,dk,dv] or None.
    Returns (o [T,H,dv], S_final [N,H,dk,dv]) as float64."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    S0 = None if S0 is None else _f64(S0).reshape(N, H, dk, dv)
    o = np.zeros((T, H, dv))
    Sf = np.zeros((N, H, dk, dv))
    hm = None if head_mask is None else np.ascontiguousarray(np.asarray(head_mask, dtype=np.uint8))
    rc = _load().oracle_kda_prefill(N, T, H, dk, dv, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                    _ptr(beta), _ptr(S0), _ptr(o), _ptr(Sf), float(scale),
                                    float(g_min), int(bool(erase)), _ptr(hm), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_kda_prefill rejected its arguments ({rc})")
    return o, Sf


def segment_transition(k, v, g, beta, g_min=-5.0, nthreads=0):
    """Transition (M [H,dk,dk], N [H,dk,dv]) of the token range given."""
    k, v, g, beta = map(_f64, (k, v, g, beta))
    T, H, dk = k.shape
    dv = v.shape[2]
    M = np.zeros((H, dk, dk))
    Nm = np.zeros((H, dk, dv))
    rc = _load().oracle_segment_transition(T, H, dk, dv, _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                           float(g_min), _ptr(M), _ptr(Nm), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_segment_transition rejected its arguments")
    return M, Nm


def segment_compose(M, Nm, S0=None):
    """M [P,H,dk,dk], Nm [P,H,dk,dv] -> (S_in [P,H,dk,dv], S_final [H,dk,dv])."""
    M, Nm = _f64(M), _f64(Nm)
    P, H, dk, dv = Nm.shape
    S0 = None if S0 is None else _f64(S0)
    S_in = np.zeros((P, H, dk, dv))
    Sf = np.zeros((H, dk, dv))
    rc = _load().oracle_segment_compose(P, H, dk, dv, _ptr(M), _ptr(Nm), _ptr(S0), _ptr(S_in), _ptr(Sf))
    if rc != 0:
        raise ValueError("oracle_segment_compose rejected its arguments")
    return S_in, Sf


def unit_lower_inverse(A):
    """(I + A)^{-1} for strictly lower-triangular A (forward substitution)."""
    A = _f64(A)
    n = A.shape[0]
    T = np.zeros((n, n))
    _load().oracle_unit_lower_inverse(n, _ptr(A), _ptr(T))
    return T


def backward(q, k, v, g, beta, cu_seqlens, do, S0=None, dS_final=None, scale=1.0, g_min=-5.0, nthreads=0):
    """Reverse mode of the token recurrence (prefill with erase).  Shapes as
    prefill; do [T,H,dv]; dS_final [N,H,dk,dv] or None.  Returns float64
    (dq, dk, dv, dg, dbeta, dS0): dg is w.r.t. the raw g (zero where
    g < g_min), dS0 w.r.t. the initial state."""
    q, k, v, g, beta, do = map(_f64, (q, k, v, g, beta, do))
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    S0 = None if S0 is None else _f64(S0).reshape(N, H, dk, dv)
    dS_final = None if dS_final is None else _f64(dS_final).reshape(N, H, dk, dv)
    dq, dkk, dg = (np.zeros((T, H, dk)) for _ in range(3))
    dvv = np.zeros((T, H, dv))
    db = np.zeros((T, H))
    dS0 = np.zeros((N, H, dk, dv))
    rc = _load().oracle_kda_backward(N, T, H, dk, dv, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(S0), _ptr(do), _ptr(dS_final), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg),
                                     _ptr(db), _ptr(dS0), float(scale), float(g_min), int(nthreads))
    if rc != 0:
        raise ValueError("oracle backward rejected its arguments")
    return dq, dkk, dvv, dg, db, dS0


def chunk_form_head(q, k, v, g, beta, S0=None, C=64, scale=1.0, g_min=-5.0):
    """Chunk (WY) form for one head: q,k,g [T,dk]; v [T,dv]; beta [T]."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((T, dv))
    _load().oracle_chunk_form_head(T, dk, dv, int(C), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(S), _ptr(o), float(scale), float(g_min))
    return o, S


def _verify_common(fn, stepwise, state, tail, conv_w, cached_qkv, cached_g, cached_b, accepted,
                   new_qkv, new_g, new_b, out_w, eps_in, eps_out, conv_act, scale, g_min, nthreads,
                   draft_len=None):
    state = _f64(state).copy()
    tail = _f64(tail).copy()
    conv_w, cached_qkv, cached_g, cached_b, new_qkv, new_g, new_b, out_w = map(
        _f64, (conv_w, cached_qkv, cached_g, cached_b, new_qkv, new_g, new_b, out_w))
    acc = np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
    R, H, dk, dv = state.shape
    W = conv_w.shape[1]
    Wd = new_qkv.shape[1] - 1
    if stepwise:
        o = np.zeros((R, H, dv))
    else:
        o = np.zeros((R, Wd + 1, H, dv))
    args = [R, H, dk, dv, W, Wd, _ptr(state), _ptr(tail), _ptr(conv_w), _ptr(cached_qkv),
            _ptr(cached_g), _ptr(cached_b), _ptr(acc), _ptr(new_qkv), _ptr(new_g), _ptr(new_b),
            _ptr(out_w), float(eps_in), float(eps_out), int(conv_act), _ptr(o), float(scale),
            float(g_min)]
    if draft_len is not None:
        dl = np.ascontiguousarray(np.asarray(draft_len, dtype=np.int32))
        args.insert(13, _ptr(dl))
    if not stepwise:
        args.append(int(nthreads))
    bad = fn(*args)
    if bad < 0:
        raise ValueError("oracle decode rejected its arguments")
    return state, tail, o, bad


def decode_verify(state, tail, conv_w, cached_qkv, cached_g, cached_b, accepted, new_qkv, new_g,
                  new_b, out_w, eps_in=1e-6, eps_out=1e-6, conv_act=1, scale=1.0, g_min=-5.0,
                  nthreads=0, draft_len=None):
    """Replay-based verify.  Returns (state', tail', o [R,Wd+1,H,dv], n_bad).
    draft_len [R] (ragged batches): request r has new rows 0..draft_len[r];
    its o rows past that stay zero."""
    if draft_len is None:
        return _verify_common(_load().oracle_decode_verify, False, state, tail, conv_w, cached_qkv,
                              cached_g, cached_b, accepted, new_qkv, new_g, new_b, out_w, eps_in,
                              eps_out, conv_act, scale, g_min, nthreads)
    return _verify_common(_load().oracle_decode_verify_ragged, False, state, tail, conv_w, cached_qkv,
                          cached_g, cached_b, accepted, new_qkv, new_g, new_b, out_w, eps_in,
                          eps_out, conv_act, scale, g_min, nthreads, draft_len=draft_len)


def decode_stepwise(state, tail, conv_w, cached_qkv, cached_g, cached_b, accepted, new_qkv, new_g,
                    new_b, out_w, eps_in=1e-6, eps_out=1e-6, conv_act=1, scale=1.0, g_min=-5.0):
    """One-token-at-a-time decoding of the accepted prefix and the bonus token.
    Returns (state', tail', o_bonus [R,H,dv], n_bad)."""
    return _verify_common(_load().oracle_decode_stepwise, True, state, tail, conv_w, cached_qkv,
                          cached_g, cached_b, accepted, new_qkv, new_g, new_b, out_w, eps_in,
                          eps_out, conv_act, scale, g_min, 0)
