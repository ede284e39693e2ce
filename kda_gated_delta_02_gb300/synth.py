"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws random tensors and nothing else: it holds none of the
recurrence's arithmetic, so the CUDA path and the oracle can both consume its
output.  Distributions (the workload recipe):

* q, k ~ N(0, 1), then L2-normalised per head over dk (prefill inputs);
* v ~ N(0, 1);
* g = max(-softplus(N(0, 1)), -5) per channel, fp32;
* beta = sigmoid(N(0, 1)), fp32;
* stored states ~ N(0, 0.02^2);
* decode: pre-conv q|k|v, raw g and raw beta ~ N(0, 1) (bf16), conv weights
  ~ N(0, 0.5^2), output-norm weight ~ N(1, 0.1^2), accepted length ~ U{0..Wd}.

Draw order is fixed: lengths -> q -> k -> v -> g -> beta -> S0, then for
decode: state -> conv tail -> conv_w -> w_o -> cached proj -> new proj ->
accepted lengths.  One torch.Generator seeded per workload; it lives on the
device the tensors are drawn on (CPU for small cases, CUDA for full sizes).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    N: int
    T: int  # total tokens (fixed length when lengths is None)
    H: int
    dk: int
    dv: int
    dtype: torch.dtype
    seed: int = 0
    len_range: tuple | None = None  # (lo, hi) per-sequence lengths, varlen
    stored_state: bool = False
    cp: bool = False


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    R: int
    H: int
    dk: int
    dv: int
    W: int = 4
    Wd: int = 7
    seed: int = 0


# The five workloads (sizes as stated by the pages' configs).
TINY = PrefillWorkload("tiny prefill T=256 H=4 d=64 fp32", 1, 256, 4, 64, 64, torch.float32)
PREFILL_32K = PrefillWorkload("prefill T=32768 H=96 d=128 bf16", 1, 32768, 96, 128, 128, torch.bfloat16)
VARLEN = PrefillWorkload("varlen prefix-continuation 16 seqs U[1K,8K] H=96 d=128 bf16", 16, 0, 96, 128,
                         128, torch.bfloat16, seed=2, len_range=(1024, 8192), stored_state=True)
ULTRA_LONG = PrefillWorkload("ultra-long T=1048576 H=12 d=128 bf16 (context-parallel)", 1, 1 << 20, 12,
                             128, 128, torch.bfloat16, seed=3, cp=True)
VERIFY = DecodeWorkload("verify-replay R=256 H=96 d=128 W=4 window 7", 256, 96, 128, 128, seed=4)


def state_bytes(layers: int, heads: int, dk: int, dv: int, bytes_per_elem: int) -> int:
    """Bytes of one request's recurrent state over all KDA layers."""
    return layers * heads * dk * dv * bytes_per_elem


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, gen, device, std=1.0, mean=0.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def _l2norm_(x):
    x.div_(torch.linalg.vector_norm(x, dim=-1, keepdim=True))
    return x


def make_prefill(w: PrefillWorkload, device="cpu", T_override: int | None = None,
                 H_override: int | None = None):
    """Returns dict(q, k, v, g, beta, cu_seqlens, S0) on `device`.
    q,k,v in w.dtype; g, beta, S0 fp32; cu_seqlens int32."""
    gen = _gen(w.seed, device)
    H = H_override or w.H
    if w.len_range is not None:
        lo, hi = w.len_range
        lens = torch.randint(lo, hi + 1, (w.N,), generator=gen, device=device)
        lens = lens.cpu()
    else:
        T = T_override or w.T
        lens = torch.full((w.N,), T // w.N, dtype=torch.int64)
    cu = torch.zeros(w.N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    T = int(cu[-1])
    q = _l2norm_(_randn((T, H, w.dk), gen, device)).to(w.dtype)
    k = _l2norm_(_randn((T, H, w.dk), gen, device)).to(w.dtype)
    v = _randn((T, H, w.dv), gen, device).to(w.dtype)
    g = _randn((T, H, w.dk), gen, device)
    g = torch.clamp_min(-torch.nn.functional.softplus(g), -5.0)
    beta = torch.sigmoid(_randn((T, H), gen, device))
    S0 = _randn((w.N, H, w.dk, w.dv), gen, device, std=0.02) if w.stored_state else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=cu.to(device), S0=S0)


def make_decode(w: DecodeWorkload, device="cpu", R_override: int | None = None,
                H_override: int | None = None, accepted=None):
    """Returns dict of decode-verify inputs on `device` (bf16 activations/state,
    fp32 weights, int32 accepted lengths)."""
    gen = _gen(w.seed, device)
    R = R_override or w.R
    H = H_override or w.H
    Cq = H * (2 * w.dk + w.dv)
    bf = torch.bfloat16
    state = _randn((R, H, w.dk, w.dv), gen, device, std=0.02).to(bf)
    tail = _randn((R, w.W - 1, Cq), gen, device).to(bf)
    conv_w = _randn((Cq, w.W), gen, device, std=0.5)
    out_w = _randn((w.dv,), gen, device, std=0.1, mean=1.0)
    cached_qkv = _randn((R, w.Wd, Cq), gen, device).to(bf)
    cached_g = _randn((R, w.Wd, H * w.dk), gen, device).to(bf)
    cached_b = _randn((R, w.Wd, H), gen, device).to(bf)
    new_qkv = _randn((R, w.Wd + 1, Cq), gen, device).to(bf)
    new_g = _randn((R, w.Wd + 1, H * w.dk), gen, device).to(bf)
    new_b = _randn((R, w.Wd + 1, H), gen, device).to(bf)
    if accepted is None:
        acc = torch.randint(0, w.Wd + 1, (R,), generator=gen, device=device).to(torch.int32)
    else:
        acc = torch.as_tensor(accepted, dtype=torch.int32, device=device)
    return dict(state=state, tail=tail, conv_w=conv_w, out_w=out_w, cached_qkv=cached_qkv,
                cached_g=cached_g, cached_b=cached_b, new_qkv=new_qkv, new_g=new_g, new_b=new_b,
                accepted=acc)
