"""Reverse mode of the chunk (WY) form, fp64 (test infrastructure only).

Only ``tests/`` may import this module; the CUDA path never does.  It writes
out, with numpy matrix products and one library inverse per chunk, the
backward of the chunk form of the prefill -- the algebra a chunked backward
on the tensor cores runs -- so that such a kernel has a checked statement to
follow.  It is pinned against the token-level reverse mode
(``oracle.backward``, itself pinned by finite differences of the forward
oracle), not against any GPU output.

Chunk form followed ("Dentro de los esfuerzos de optimizacion de Kimi K3",
"Nota tecnica: Precision del KDA y memoria on-chip"; the backward as the
chunk kernel's training use: "Noyaux KDA et FlashKDA", "FlashKDA : le noyau
par blocs").  For a chunk of L tokens entered with state S0, with
gamma_t = sum_{r<=t} max(g_r, g_min) (per key channel), Gam = e^gamma and
GamC = Gam of the chunk's last token:

    Kt = K * Gam      Kb = K / Gam      Kh = K * GamC / Gam      Qt = Q * Gam
    A  = strict_lower(diag(beta) Kt Kb^T)        B = lower(Qt Kb^T)
    Tm = (I + A)^-1   R = diag(beta) (V - Kt S0)    U = Tm R
    O  = scale (Qt S0 + B U)                      S_C = diag(GamC) S0 + Kh^T U

(u_t is beta_t (v_t - p_t) of the token recurrence; A_ts carries beta_t.)
Given dO and dS_C the reverse pass is, step by step in the opposite order:

    dU  = scale B^T dO + Kh dS_C            dB = scale lower(dO U^T)
    dQt = scale dO S0^T                     dS0 = scale Qt^T dO + diag(GamC) dS_C
    dKh = U dS_C^T                          dgamma_C += GamC * rowsum(dS_C * S0)
    dR  = Tm^T dU                           dTm = dU R^T
    dA  = strict_lower(-Tm^T dTm Tm^T)
    dV  = diag(beta) dR                     dbeta = rowsum((V - Kt S0) * dR)
    dKt = -diag(beta) dR S0^T               dS0 -= Kt^T diag(beta) dR
    dM  = diag(beta) dA  (M = Kt Kb^T)      dbeta += rowsum(dA * M)
    dKt += dM Kb                            dKb = dM^T Kt
    dQt += lower(dB) Kb                     dKb += lower(dB)^T Qt
    dK  = dKt Gam + dKb / Gam + dKh GamC / Gam          dQ = dQt Gam
    dgamma_t = dKt Kt - dKb Kb - dKh Kh + dQt Qt   (+ sum_t dKh Kh and
               the dgamma_C term on the chunk's last token)
    dg'_r = sum_{t >= r} dgamma_t;   dg = 0 where g < g_min, else dg'

and dS0 of a chunk is dS_C of the chunk before it.  In fp64 the factors
1/Gam stay finite (gamma >= 64 g_min = -320 within a chunk of 64).  A NaN g
takes the floor, as an IEEE maximum does, and gets the gradient of g = g_min
(the pages say nothing of NaN).
"""
from __future__ import annotations

import numpy as np


def _chunk_forward(q, k, v, gp, beta, S0, scale, mm=np.matmul):
    gam = np.cumsum(gp, axis=0)
    Gam = np.exp(gam)
    GamC = Gam[-1]
    Kt, Kb, Kh, Qt = k * Gam, k / Gam, k * (GamC / Gam), q * Gam
    L = k.shape[0]
    M = mm(Kt, Kb.T)
    A = np.tril(beta[:, None] * M, -1)
    B = np.tril(mm(Qt, Kb.T))
    Tm = np.linalg.inv(np.eye(L) + A)
    Vres = v - mm(Kt, S0)
    R = beta[:, None] * Vres
    U = mm(Tm, R)
    O = scale * (mm(Qt, S0) + mm(B, U))
    SC = GamC[:, None] * S0 + mm(Kh.T, U)
    return dict(Gam=Gam, GamC=GamC, Kt=Kt, Kb=Kb, Kh=Kh, Qt=Qt, M=M, B=B, Tm=Tm, Vres=Vres, R=R, U=U,
                O=O, SC=SC)


def _chunk_reverse(f, S0, beta, dO, dSC, scale, mm=np.matmul):
    Gam, GamC, Kt, Kb, Kh, Qt = f["Gam"], f["GamC"], f["Kt"], f["Kb"], f["Kh"], f["Qt"]
    M, B, Tm, Vres, R, U = f["M"], f["B"], f["Tm"], f["Vres"], f["R"], f["U"]
    # O = scale (Qt S0 + B U);  S_C = diag(GamC) S0 + Kh^T U
    dU = scale * mm(B.T, dO) + mm(Kh, dSC)
    dB = scale * np.tril(mm(dO, U.T))
    dQt = scale * mm(dO, S0.T)
    dS0 = scale * mm(Qt.T, dO) + GamC[:, None] * dSC
    dKh = mm(U, dSC.T)
    dgamC = GamC * np.sum(dSC * S0, axis=1)
    # U = Tm R;  Tm = (I + A)^-1
    dR = mm(Tm.T, dU)
    dTm = mm(dU, R.T)
    dA = np.tril(-mm(mm(Tm.T, dTm), Tm.T), -1)
    # R = diag(beta) (V - Kt S0)
    dV = beta[:, None] * dR
    dbeta = np.sum(Vres * dR, axis=1)
    dKt = -mm(beta[:, None] * dR, S0.T)
    dS0 -= mm(Kt.T, beta[:, None] * dR)
    # A = strict_lower(diag(beta) M), M = Kt Kb^T
    dM = beta[:, None] * dA
    dbeta += np.sum(dA * M, axis=1)
    dKt += mm(dM, Kb)
    dKb = mm(dM.T, Kt)
    # B = lower(Qt Kb^T)
    dQt += mm(np.tril(dB), Kb)
    dKb += mm(np.tril(dB).T, Qt)
    # Kt = K Gam, Kb = K / Gam, Kh = K GamC / Gam, Qt = Q Gam (Gam = e^gamma)
    dK = dKt * Gam + dKb / Gam + dKh * (GamC / Gam)
    dQ = dQt * Gam
    dgam = dKt * Kt - dKb * Kb - dKh * Kh + dQt * Qt
    dgam[-1] += dgamC + np.sum(dKh * Kh, axis=0)
    # gamma = cumsum(g'): the gradient of g'_r sums those of gamma_t, t >= r
    dgp = np.cumsum(dgam[::-1], axis=0)[::-1]
    return dQ, dK, dV, dgp, dbeta, dS0


def chunk_form_backward_head(q, k, v, g, beta, do, S0=None, dS_final=None, C=64, scale=1.0, g_min=-5.0,
                             mm=np.matmul):
    """One head: q, k, g [T, dk]; v, do [T, dv]; beta [T]; S0, dS_final
    [dk, dv] or None (zero).  Returns (o, S_final, dq, dk, dv, dg, dbeta,
    dS0), fp64; dg is with respect to the raw g (zero where g < g_min).
    `mm` computes every matrix product (a test can round its operands to
    study a reduced-precision kernel); the inverse stays fp64."""
    q, k, v, g, beta, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, do))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    gp = np.fmax(g, g_min)
    bounds = [(c0, min(c0 + C, T)) for c0 in range(0, T, C)]
    starts, fwd = [], []
    o = np.zeros((T, dv))
    for c0, c1 in bounds:
        starts.append(S)
        f = _chunk_forward(q[c0:c1], k[c0:c1], v[c0:c1], gp[c0:c1], beta[c0:c1], S, scale, mm)
        fwd.append(f)
        o[c0:c1] = f["O"]
        S = f["SC"]
    S_final = S
    dq, dkk, dgp = np.zeros((T, dk)), np.zeros((T, dk)), np.zeros((T, dk))
    dvv, db = np.zeros((T, dv)), np.zeros(T)
    dS = np.zeros((dk, dv)) if dS_final is None else np.array(dS_final, dtype=np.float64)
    for (c0, c1), S_in, f in reversed(list(zip(bounds, starts, fwd))):
        dQ, dK, dV, dG, dB, dS = _chunk_reverse(f, S_in, beta[c0:c1], do[c0:c1], dS, scale, mm)
        dq[c0:c1], dkk[c0:c1], dvv[c0:c1], dgp[c0:c1], db[c0:c1] = dQ, dK, dV, dG, dB
    dg = np.where(g < g_min, 0.0, dgp)
    return o, S_final, dq, dkk, dvv, dg, db, dS


def state_gradient_chain(q, k, v, g, beta, do, S0=None, dS_final=None, C=64, scale=1.0, g_min=-5.0):
    """The serial part of the chunked backward on its own, one head: the
    chunk-start states S_in[c] and the state gradients dS_C[c] arriving at the
    end of each chunk c (chunk order).  It is the adjoint of the forward's
    state walk (U = Tm R = Tm diag(beta) V - W S0, O = scale (Qt S0 + B U),
    S_C = diag(GamC) S0 + Kh^T U, with W = Tm diag(beta) Kt) and uses the
    same chunk-local operands:

        dU      = scale B^T dO + Kh dS_C
        dS_prev = scale Qt^T dO + diag(GamC) dS_C - W^T dU

    Given S_in[c] and dS_C[c], every chunk's token gradients are independent of
    the other chunks (``chunk_token_gradients``)."""
    q, k, v, g, beta, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, do))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    gp = np.fmax(g, g_min)
    bounds = [(c0, min(c0 + C, T)) for c0 in range(0, T, C)]
    S_in, fwd = [], []
    for c0, c1 in bounds:
        S_in.append(S)
        f = _chunk_forward(q[c0:c1], k[c0:c1], v[c0:c1], gp[c0:c1], beta[c0:c1], S, scale)
        fwd.append(f)
        S = f["SC"]
    dS_C = [None] * len(bounds)
    dS = np.zeros((dk, dv)) if dS_final is None else np.array(dS_final, dtype=np.float64)
    for c in range(len(bounds) - 1, -1, -1):
        c0, c1 = bounds[c]
        f = fwd[c]
        dS_C[c] = dS
        W = f["Tm"] @ (beta[c0:c1, None] * f["Kt"])
        dU = scale * f["B"].T @ do[c0:c1] + f["Kh"] @ dS
        dS = scale * f["Qt"].T @ do[c0:c1] + f["GamC"][:, None] * dS - W.T @ dU
    return bounds, S_in, dS_C, dS


def chunk_token_gradients(q, k, v, g, beta, do, S_in, dS_C, scale=1.0, g_min=-5.0):
    """One chunk's token gradients (dq, dk, dv, dg, dbeta) and its dS0 from the
    chunk's rows, its start state S_in and the state gradient dS_C at its end."""
    q, k, v, g, beta, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, do))
    f = _chunk_forward(q, k, v, np.fmax(g, g_min), beta, S_in, scale)
    dQ, dK, dV, dgp, dB, dS0 = _chunk_reverse(f, S_in, beta, do, dS_C, scale)
    # dg' of the chunk's tokens is local: gamma restarts at every chunk
    return dQ, dK, dV, np.where(g < g_min, 0.0, dgp), dB, dS0


def chunk_form_backward(q, k, v, g, beta, cu_seqlens, do, S0=None, dS_final=None, C=64, scale=1.0,
                        g_min=-5.0):
    """Packed sequences (cu_seqlens [N+1]) and heads: q, k, g [T, H, dk]; v, do
    [T, H, dv]; beta [T, H]; S0, dS_final [N, H, dk, dv] or None.  Chunks restart
    at every sequence start.  Returns (o, S_final, dq, dk, dv, dg, dbeta, dS0)."""
    q, k, v, g, beta, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, do))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, H, dk = k.shape
    dv = v.shape[2]
    N = cu.shape[0] - 1
    o, dq, dkk, dvv, dg = (np.zeros_like(x) for x in (v, q, k, v, g))
    db = np.zeros((T, H))
    S_final, dS0 = np.zeros((N, H, dk, dv)), np.zeros((N, H, dk, dv))
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            s0 = None if S0 is None else S0[n, h]
            dsf = None if dS_final is None else dS_final[n, h]
            if b == a:
                S_final[n, h] = 0.0 if s0 is None else s0
                dS0[n, h] = 0.0 if dsf is None else dsf
                continue
            r = chunk_form_backward_head(q[a:b, h], k[a:b, h], v[a:b, h], g[a:b, h], beta[a:b, h],
                                         do[a:b, h], s0, dsf, C=C, scale=scale, g_min=g_min)
            o[a:b, h], S_final[n, h] = r[0], r[1]
            dq[a:b, h], dkk[a:b, h], dvv[a:b, h], dg[a:b, h], db[a:b, h], dS0[n, h] = r[2:]
    return o, S_final, dq, dkk, dvv, dg, db, dS0


# ---------------------------------------------------------------------------
# fp32 with block anchoring.  In fp32 the factors 1/Gam overflow inside a
# chunk of 64 held at the floor (e^{320}).  The forward avoids them by
# splitting e^{gamma_t - gamma_s} = e^{gamma_t - gamma_a} e^{gamma_a - gamma_s}
# with the anchor a = the last token of the 16-token block of s: the column
# factor lies in [e^{-75}, 1] and the row factor in [0, e^{75}] (rows of later
# blocks are <= 1), both inside fp32.  The same split carries the gradients of
# M = Kt Kb^T and B = Qt Kb^T, the only products that need 1/Gam:
#     row part  dK_t += e^{gamma_t - gamma_a} (dM_t,blk  (k_blk e^{gamma_a - gamma_blk}))
#     col part  dK_s += e^{gamma_a - gamma_s} (dM_rows,s^T (k_rows e^{gamma_rows - gamma_a}))
# and the log-decay gradient takes k (or q) times the row part minus k times
# the column part.  Every other factor (e^{gamma}, e^{gamma_C - gamma}) is at
# most 1 and may only underflow where the true term is below fp32's range.

_BLK = 16


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def _anchored_tiles(x_rows, k, gam, L, strict):
    """Lower(-triangular) products x_rows_t . k_s e^{gamma_t - gamma_s} in fp32,
    built per 16-token column block with its anchor, and the per-block factors."""
    P = np.zeros((L, L), dtype=np.float32)
    blocks = []
    for j0 in range(0, L, _BLK):
        j1 = min(j0 + _BLK, L)
        a = j1 - 1
        col = np.exp(gam[a] - gam[j0:j1])          # <= 1, >= e^{-75}
        row = np.exp(gam[j0:] - gam[a])            # <= e^{75}
        kc = k[j0:j1] * col
        xr = x_rows[j0:] * row
        P[j0:, j0:j1] = xr @ kc.T
        blocks.append((j0, j1, row, col))
    mask = np.tril(np.ones((L, L), dtype=bool), -1 if strict else 0)
    return np.where(mask, P, np.float32(0)), blocks


def chunk_form_backward_head_f32(q, k, v, g, beta, do, S0=None, dS_final=None, C=64, scale=1.0, g_min=-5.0):
    """The chunk-form reverse pass in fp32 (numpy float32 products and
    elementwise work; fp32 inverse), with the block anchoring above.  Same
    arguments and results as ``chunk_form_backward_head``, as float64 arrays
    holding fp32 values."""
    q, k, v, g, beta, do = (_f32(x) for x in (q, k, v, g, beta, do))
    T, dk = k.shape
    dv = v.shape[1]
    scale = np.float32(scale)
    S = np.zeros((dk, dv), np.float32) if S0 is None else _f32(S0).copy()
    gp = np.fmax(g, np.float32(g_min))
    bounds = [(c0, min(c0 + C, T)) for c0 in range(0, T, C)]
    starts, fwd = [], []
    o = np.zeros((T, dv), np.float32)
    for c0, c1 in bounds:
        L = c1 - c0
        kk, qq, vv, bb = k[c0:c1], q[c0:c1], v[c0:c1], beta[c0:c1]
        gam = np.cumsum(gp[c0:c1], axis=0, dtype=np.float32)
        Gam = np.exp(gam)
        GamC = Gam[-1]
        Kt, Qt, Kh = kk * Gam, qq * Gam, kk * np.exp(gam[-1] - gam)
        M, blocks = _anchored_tiles(kk, kk, gam, L, strict=True)
        B, _ = _anchored_tiles(qq, kk, gam, L, strict=False)
        A = bb[:, None] * M
        Tm = np.linalg.inv(np.eye(L, dtype=np.float32) + A).astype(np.float32)
        Vres = vv - Kt @ S
        R = bb[:, None] * Vres
        U = Tm @ R
        o[c0:c1] = scale * (Qt @ S + B @ U)
        starts.append(S)
        fwd.append(dict(gam=gam, Gam=Gam, GamC=GamC, Kt=Kt, Qt=Qt, Kh=Kh, M=M, B=B, blocks=blocks, Tm=Tm,
                        Vres=Vres, R=R, U=U))
        S = GamC[:, None] * S + Kh.T @ U
    S_final = S
    dq, dkk, dgp = (np.zeros((T, dk), np.float32) for _ in range(3))
    dvv, db = np.zeros((T, dv), np.float32), np.zeros(T, np.float32)
    dS = np.zeros((dk, dv), np.float32) if dS_final is None else _f32(dS_final).copy()
    for (c0, c1), S_in, f in reversed(list(zip(bounds, starts, fwd))):
        kk, qq, bb, dO = k[c0:c1], q[c0:c1], beta[c0:c1], do[c0:c1]
        Gam, GamC, Kt, Qt, Kh = f["Gam"], f["GamC"], f["Kt"], f["Qt"], f["Kh"]
        M, B, Tm, Vres, R, U = f["M"], f["B"], f["Tm"], f["Vres"], f["R"], f["U"]
        dU = scale * (B.T @ dO) + Kh @ dS
        dB = scale * np.tril(dO @ U.T)
        dQs = scale * (dO @ S_in.T)                   # through Qt S0
        dS0 = scale * (Qt.T @ dO) + GamC[:, None] * dS
        dKh = U @ dS.T
        dgamC = GamC * np.sum(dS * S_in, axis=1)
        dR = Tm.T @ dU
        dTm = dU @ R.T
        dA = np.tril(-(Tm.T @ dTm @ Tm.T), -1)
        dvv[c0:c1] = bb[:, None] * dR
        dbeta = np.sum(Vres * dR, axis=1) + np.sum(dA * M, axis=1)
        dKs = -(bb[:, None] * dR) @ S_in.T            # through Kt S0
        dS0 -= Kt.T @ (bb[:, None] * dR)
        dM = bb[:, None] * dA
        # M and B through the anchored blocks: row and column parts
        Krow, Kcol, Qrow = (np.zeros_like(kk) for _ in range(3))
        for j0, j1, row, col in f["blocks"]:
            kc = kk[j0:j1] * col
            Krow[j0:] += row * (dM[j0:, j0:j1] @ kc)
            Qrow[j0:] += row * (dB[j0:, j0:j1] @ kc)
            Kcol[j0:j1] += col * (dM[j0:, j0:j1].T @ (kk[j0:] * row) + dB[j0:, j0:j1].T @ (qq[j0:] * row))
        dkk[c0:c1] = dKs * Gam + Krow + Kcol + dKh * np.exp(f["gam"][-1] - f["gam"])
        dq[c0:c1] = dQs * Gam + Qrow
        dgam = dKs * Kt + dQs * Qt - dKh * Kh + kk * Krow + qq * Qrow - kk * Kcol
        dgam[-1] += dgamC + np.sum(dKh * Kh, axis=0)
        dgp[c0:c1] = np.cumsum(dgam[::-1], axis=0, dtype=np.float32)[::-1]
        db[c0:c1] = dbeta
        dS = dS0
    dg = np.where(g < np.float32(g_min), np.float32(0), dgp)
    out = (o, S_final, dq, dkk, dvv, dg, db, dS)
    return tuple(np.asarray(x, dtype=np.float64) for x in out)
