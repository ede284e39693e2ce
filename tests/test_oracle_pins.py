"""Pins for the fp64 oracle: each checks it against something other than itself.

* brute-force products of the explicit dk x dk transition matrices (tiny sizes)
* the delta-rule store invariant, closed forms for the beta = 0 and no-erase
  limits (decayed / plain linear attention, against numpy's matmul)
* the pages' worked examples (tests/golden/): dependency inverse, affine
  composition, state-size arithmetic
* numpy.linalg.inv for the triangular inverse, numpy's logaddexp / a direct
  logistic for the gates, identity and shift convolution kernels
* structural invariants: head permutation, sequence independence, replay
  equals one-token-at-a-time decoding bit for bit
"""
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden

G_MIN = -5.0


def rand_inputs(rng, T, H, dk, dv, beta_zero=False, unit_k=True, g_scale=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -np.logaddexp(0.0, g_scale * rng.standard_normal((T, H, dk)))
    beta = np.zeros((T, H)) if beta_zero else 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


def explicit_A(k, g, beta):
    """(I - b k k^T) Diag(exp(max(g, g_min))) as an explicit matrix."""
    dk = k.shape[0]
    D = np.diag(np.exp(np.maximum(g, G_MIN)))
    return (np.eye(dk) - beta * np.outer(k, k)) @ D


def brute_force_head(q, k, v, g, beta, S0):
    """S_t = A_t ... A_1 S0 + sum_s A_t ... A_{s+1} b_s k_s v_s^T, o_t = S_t^T q_t."""
    T = q.shape[0]
    As = [explicit_A(k[t], g[t], beta[t]) for t in range(T)]
    outs, states = [], []
    for t in range(T):
        prod = np.eye(k.shape[1])
        for r in range(t + 1):
            prod = As[r] @ prod
        St = prod @ S0
        for s in range(t + 1):
            P = np.eye(k.shape[1])
            for r in range(s + 1, t + 1):
                P = As[r] @ P
            St = St + P @ (beta[s] * np.outer(k[s], v[s]))
        outs.append(St.T @ q[t])
        states.append(St)
    return np.array(outs), states


# --------------------------------------------------------------------------- recurrence
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_recurrence_matches_brute_force_products(oracle, seed):
    rng = np.random.default_rng(seed)
    T, H, dk, dv = 7, 2, 4, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv, unit_k=False)
    g[2, 0, 1] = -7.5  # below the floor: must act as -5
    g[4, 1, :] = -5.0
    S0 = rng.standard_normal((1, H, dk, dv))
    o, Sf = oracle.prefill(q, k, v, g, beta, [0, T], S0=S0)
    for h in range(H):
        ob, states = brute_force_head(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], S0[0, h])
        np.testing.assert_allclose(o[:, h], ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(Sf[0, h], states[-1], rtol=0, atol=1e-13)


def test_floor_applies_per_token_per_channel(oracle):
    rng = np.random.default_rng(5)
    T, H, dk, dv = 6, 1, 3, 2
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    g_low = g.copy()
    g_low[1, 0, 0] = -40.0
    g_low[3, 0, 2] = -5.5
    g_clamped = np.maximum(g_low, -5.0)
    a = oracle.prefill(q, k, v, g_low, beta, [0, T])
    b = oracle.prefill(q, k, v, g_clamped, beta, [0, T])
    np.testing.assert_array_equal(a[0], b[0])
    c = oracle.prefill(q, k, v, g_low, beta, [0, T], g_min=-100.0)
    assert np.max(np.abs(c[0] - a[0])) > 1e-6  # the floor is not a no-op here


def test_delta_rule_store_invariant(oracle):
    """beta = 1 and unit k: the state maps k_t exactly onto v_t, S_t^T k_t = v_t."""
    rng = np.random.default_rng(11)
    T, H, dk, dv = 9, 3, 8, 5
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    beta[:] = 1.0
    S0 = rng.standard_normal((1, H, dk, dv))
    o, _ = oracle.prefill(k, k, v, g, beta, [0, T], S0=S0)  # read out with q = k
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-13)


def test_beta_zero_is_pure_decay(oracle):
    """beta = 0: S_t = Diag(Gamma_t) S0 and o_t = (Diag(Gamma_t) S0)^T q_t."""
    rng = np.random.default_rng(3)
    T, H, dk, dv = 10, 2, 6, 4
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv, beta_zero=True)
    S0 = rng.standard_normal((1, H, dk, dv))
    o, Sf = oracle.prefill(q, k, v, g, beta, [0, T], S0=S0)
    gam = np.cumsum(np.maximum(g, G_MIN), axis=0)  # [T,H,dk]
    for h in range(H):
        for t in range(T):
            St = np.exp(gam[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(Sf[0, h], np.exp(gam[-1, h])[:, None] * S0[0, h], rtol=1e-13)


def test_no_erase_is_decayed_linear_attention(oracle):
    """Without the erase term: o_t = S0^T Gamma_t q_t + sum_{s<=t} ((q_t . Gamma_t/Gamma_s) k_s) b_s v_s."""
    rng = np.random.default_rng(4)
    T, H, dk, dv = 12, 2, 5, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    o, _ = oracle.prefill(q, k, v, g, beta, [0, T], S0=S0, erase=False)
    gam = np.cumsum(np.maximum(g, G_MIN), axis=0)
    for h in range(H):
        for t in range(T):
            ref = S0[0, h].T @ (np.exp(gam[t, h]) * q[t, h])
            for s in range(t + 1):
                ref = ref + np.dot(q[t, h] * np.exp(gam[t, h] - gam[s, h]), k[s, h]) * beta[s, h] * v[s, h]
            np.testing.assert_allclose(o[t, h], ref, rtol=1e-12, atol=1e-13)


def test_no_erase_zero_decay_is_plain_linear_attention(oracle):
    """g = 0 and no erase: O = (causal(Q K^T)) (diag(b) V), a plain matmul."""
    rng = np.random.default_rng(6)
    T, H, dk, dv = 16, 2, 8, 8
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    g[:] = 0.0
    o, _ = oracle.prefill(q, k, v, g, beta, [0, T], erase=False)
    for h in range(H):
        scores = np.tril(q[:, h] @ k[:, h].T)
        np.testing.assert_allclose(o[:, h], scores @ (beta[:, h, None] * v[:, h]), rtol=1e-12, atol=1e-13)


def test_zero_decay_zero_beta_is_identity_readout(oracle):
    """g = 0, beta = 0 (literal rule): the state never changes, o_t = S0^T q_t."""
    rng = np.random.default_rng(7)
    T, H, dk, dv = 5, 1, 4, 4
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv, beta_zero=True)
    g[:] = 0.0
    S0 = rng.standard_normal((1, H, dk, dv))
    o, Sf = oracle.prefill(q, k, v, g, beta, [0, T], S0=S0)
    np.testing.assert_allclose(o[:, 0], q[:, 0] @ S0[0, 0], rtol=1e-14)
    np.testing.assert_array_equal(Sf, S0)


def test_scale_multiplies_output(oracle):
    rng = np.random.default_rng(8)
    q, k, v, g, beta = rand_inputs(rng, 6, 1, 4, 4)
    o1, _ = oracle.prefill(q, k, v, g, beta, [0, 6])
    o2, _ = oracle.prefill(q, k, v, g, beta, [0, 6], scale=0.25)
    np.testing.assert_allclose(o2, 0.25 * o1, rtol=1e-15)


def test_heads_are_independent(oracle):
    rng = np.random.default_rng(9)
    T, H, dk, dv = 8, 4, 4, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    perm = np.array([2, 0, 3, 1])
    o, Sf = oracle.prefill(q, k, v, g, beta, [0, T], S0=S0)
    op, Sfp = oracle.prefill(q[:, perm], k[:, perm], v[:, perm], g[:, perm], beta[:, perm], [0, T],
                             S0=S0[:, perm])
    np.testing.assert_array_equal(op, o[:, perm])
    np.testing.assert_array_equal(Sfp, Sf[:, perm])


def test_packed_sequences_match_separate_runs(oracle):
    rng = np.random.default_rng(10)
    lens = [5, 1, 0, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, dk, dv = int(cu[-1]), 2, 4, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    o, Sf = oracle.prefill(q, k, v, g, beta, cu, S0=S0)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, Sn = oracle.prefill(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], [0, b - a], S0=S0[n:n + 1])
        np.testing.assert_array_equal(o[a:b], on)
        np.testing.assert_array_equal(Sf[n], Sn[0])
    np.testing.assert_array_equal(Sf[2], S0[2])  # empty sequence keeps its state


def test_head_mask_skips_heads(oracle):
    rng = np.random.default_rng(12)
    q, k, v, g, beta = rand_inputs(rng, 6, 3, 4, 4)
    o, Sf = oracle.prefill(q, k, v, g, beta, [0, 6])
    om, Sfm = oracle.prefill(q, k, v, g, beta, [0, 6], head_mask=[0, 1, 0])
    np.testing.assert_array_equal(om[:, 1], o[:, 1])
    assert np.all(om[:, 0] == 0) and np.all(om[:, 2] == 0)


# --------------------------------------------------------------------------- chunk algebra
def test_dependency_inverse_worked_example(oracle):
    rows = read_golden("dependency_inverse_example.txt")
    A = np.zeros((3, 3))
    T_ref = {}
    for name, r, c, num, den in rows:
        val = Fraction(int(num), int(den))
        if name == "A":
            A[int(r), int(c)] = float(val)
        else:
            T_ref[(int(r), int(c))] = val
    T = oracle.unit_lower_inverse(A)
    for (r, c), val in T_ref.items():
        assert T[r, c] == float(val), (r, c, T[r, c], val)  # exact in binary
    assert T[2, 0] == -1.0 / 16.0


@pytest.mark.parametrize("n", [1, 5, 16, 64])
def test_unit_lower_inverse_matches_numpy(oracle, n):
    rng = np.random.default_rng(n)
    A = np.tril(rng.standard_normal((n, n)) * 0.3, -1)
    T = oracle.unit_lower_inverse(A)
    np.testing.assert_allclose(T, np.linalg.inv(np.eye(n) + A), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(T @ (np.eye(n) + A), np.eye(n), atol=1e-12)
    assert np.all(np.triu(T, 1) == 0) and np.all(np.diag(T) == 1.0)


@pytest.mark.parametrize("T,C,floor_stress", [(64, 64, False), (200, 64, False), (37, 16, False),
                                              (128, 64, True)])
def test_chunk_form_matches_token_form(oracle, T, C, floor_stress):
    rng = np.random.default_rng(T + C)
    dk, dv = 8, 6
    q, k, v, g, beta = rand_inputs(rng, T, 1, dk, dv)
    if floor_stress:
        g[:] = -5.0
    S0 = 0.5 * rng.standard_normal((1, 1, dk, dv))
    o_ref, S_ref = oracle.prefill(q, k, v, g, beta, [0, T], S0=S0)
    o, S = oracle.chunk_form_head(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0=S0[0, 0], C=C)
    scale_o = np.max(np.abs(o_ref))
    np.testing.assert_allclose(o, o_ref[:, 0], rtol=0, atol=1e-12 * max(scale_o, 1.0))
    np.testing.assert_allclose(S, S_ref[0, 0], rtol=0, atol=1e-12 * max(np.max(np.abs(S_ref)), 1.0))


# --------------------------------------------------------------------------- segments
def test_affine_composition_worked_example(oracle):
    rows = {r[0]: [Fraction(int(r[1]), int(r[2])), Fraction(int(r[3]), int(r[4]))]
            for r in read_golden("affine_composition_example.txt")}
    M = np.array([float(rows["first"][0]), float(rows["second"][0])]).reshape(2, 1, 1, 1)
    N = np.array([float(rows["first"][1]), float(rows["second"][1])]).reshape(2, 1, 1, 1)
    Mc, Nc = rows["composed"]
    for s in [0.0, 1.0, -3.0, 8.5]:
        S_in, Sf = oracle.segment_compose(M, N, S0=np.array([[[s]]]))
        assert Sf[0, 0, 0] == float(Mc) * s + float(Nc)
        assert S_in[0, 0, 0, 0] == s
        assert S_in[1, 0, 0, 0] == float(rows["first"][0]) * s + float(rows["first"][1])


def test_segment_transition_matches_explicit_products(oracle):
    rng = np.random.default_rng(21)
    T, H, dk, dv = 6, 2, 4, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv, unit_k=False)
    M, N = oracle.segment_transition(k, v, g, beta)
    for h in range(H):
        P = np.eye(dk)
        for t in range(T):
            P = explicit_A(k[t, h], g[t, h], beta[t, h]) @ P
        np.testing.assert_allclose(M[h], P, rtol=0, atol=1e-14)
        _, states = brute_force_head(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], np.zeros((dk, dv)))
        np.testing.assert_allclose(N[h], states[-1], rtol=0, atol=1e-14)


@pytest.mark.parametrize("cuts", [[0, 7, 8, 20, 31], [0, 0, 5, 5, 31], [0, 31]])
def test_composed_segments_match_sequential(oracle, cuts):
    """Split [0, T) at `cuts` (length-1 and empty segments included); compose
    the independent transitions and compare with the sequential states."""
    rng = np.random.default_rng(len(cuts))
    T, H, dk, dv = 31, 2, 6, 5
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((H, dk, dv))
    Ms, Ns = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        M, N = oracle.segment_transition(k[a:b], v[a:b], g[a:b], beta[a:b])
        Ms.append(M)
        Ns.append(N)
    S_in, Sf = oracle.segment_compose(np.array(Ms), np.array(Ns), S0=S0)
    for p, a in enumerate(cuts[:-1]):
        _, Sa = oracle.prefill(q[:a], k[:a], v[:a], g[:a], beta[:a], [0, a], S0=S0[None])
        np.testing.assert_allclose(S_in[p], Sa[0], rtol=0, atol=1e-12)
    _, ST = oracle.prefill(q, k, v, g, beta, [0, T], S0=S0[None])
    np.testing.assert_allclose(Sf, ST[0], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- decode verify
def decode_inputs(rng, R, H, dk, dv, W=4, Wd=7, accepted=None, state_std=0.02):
    Cq = H * (2 * dk + dv)
    state = state_std * rng.standard_normal((R, H, dk, dv))
    tail = rng.standard_normal((R, W - 1, Cq))
    conv_w = 0.5 * rng.standard_normal((Cq, W))
    out_w = 1.0 + 0.1 * rng.standard_normal(dv)
    cached_qkv = rng.standard_normal((R, Wd, Cq))
    cached_g = rng.standard_normal((R, Wd, H * dk))
    cached_b = rng.standard_normal((R, Wd, H))
    new_qkv = rng.standard_normal((R, Wd + 1, Cq))
    new_g = rng.standard_normal((R, Wd + 1, H * dk))
    new_b = rng.standard_normal((R, Wd + 1, H))
    if accepted is None:
        accepted = rng.integers(0, Wd + 1, size=R)
    return dict(state=state, tail=tail, conv_w=conv_w, cached_qkv=cached_qkv, cached_g=cached_g,
                cached_b=cached_b, accepted=np.asarray(accepted, dtype=np.int32), new_qkv=new_qkv,
                new_g=new_g, new_b=new_b, out_w=out_w)


@pytest.mark.parametrize("conv_act", [0, 1])
def test_replay_equals_stepwise_decoding_bitwise(oracle, conv_act):
    rng = np.random.default_rng(30 + conv_act)
    R, H, dk, dv = 8, 2, 4, 3
    inp = decode_inputs(rng, R, H, dk, dv, accepted=list(range(8)))
    st_v, tl_v, o_v, bad_v = oracle.decode_verify(**inp, conv_act=conv_act)
    st_s, tl_s, o_s, bad_s = oracle.decode_stepwise(**inp, conv_act=conv_act)
    assert bad_v == 0 and bad_s == 0
    np.testing.assert_array_equal(st_v, st_s)
    np.testing.assert_array_equal(tl_v, tl_s)
    np.testing.assert_array_equal(o_v[:, 0], o_s)  # bonus-token output row


def test_ragged_windows_pin_the_token_count(oracle):
    """Ragged verify (a draft count per request, "Dentro de los esfuerzos de
    optimizacion de Kimi K3" section 5): with no drafts it is one-token-at-a-
    time decoding of the accepted rows and the bonus (an independent routine),
    bit for bit; padded draft rows (NaN here) never reach outputs, state or
    tail; a request's rows match the full window's rows (later drafts cannot
    change earlier outputs); out-of-range counts skip the request."""
    rng = np.random.default_rng(35)
    R, H, dk, dv, Wd = 8, 2, 4, 3, 7
    inp = decode_inputs(rng, R, H, dk, dv, accepted=list(range(8)))
    # no drafts == stepwise decoding
    zero = np.zeros(R, dtype=np.int32)
    st_r, tl_r, o_r, bad_r = oracle.decode_verify(**inp, draft_len=zero)
    st_s, tl_s, o_s, bad_s = oracle.decode_stepwise(**inp)
    assert bad_r == 0 and bad_s == 0
    np.testing.assert_array_equal(st_r, st_s)
    np.testing.assert_array_equal(tl_r, tl_s)
    np.testing.assert_array_equal(o_r[:, 0], o_s)
    assert np.all(o_r[:, 1:] == 0.0)
    # random counts, padding poisoned with NaN
    d = rng.integers(0, Wd + 1, size=R).astype(np.int32)
    poisoned = {k: v.copy() for k, v in inp.items()}
    for r in range(R):
        poisoned["new_qkv"][r, d[r] + 1:] = np.nan
        poisoned["new_g"][r, d[r] + 1:] = np.nan
        poisoned["new_b"][r, d[r] + 1:] = np.nan
    st_p, tl_p, o_p, bad_p = oracle.decode_verify(**poisoned, draft_len=d)
    st_u, tl_u, o_u, bad_u = oracle.decode_verify(**inp)  # every request with Wd drafts
    assert bad_p == 0 and bad_u == 0
    assert np.all(np.isfinite(st_p)) and np.all(np.isfinite(tl_p)) and np.all(np.isfinite(o_p))
    np.testing.assert_array_equal(st_p, st_u)  # the state is written back after the bonus
    np.testing.assert_array_equal(tl_p, tl_u)
    for r in range(R):
        np.testing.assert_array_equal(o_p[r, :d[r] + 1], o_u[r, :d[r] + 1])
        assert np.all(o_p[r, d[r] + 1:] == 0.0)
    # out-of-range counts: request skipped, counted
    bad_d = d.copy()
    bad_d[3] = Wd + 1
    bad_d[5] = -1
    st_b, tl_b, o_b, nb = oracle.decode_verify(**inp, draft_len=bad_d)
    assert nb == 2
    for r in (3, 5):
        np.testing.assert_array_equal(st_b[r], inp["state"][r])
        np.testing.assert_array_equal(tl_b[r], inp["tail"][r])
        assert np.all(o_b[r] == 0.0)


def test_conv_identity_and_shift_pin_tail_order(oracle):
    """beta = 0 and g = 0 freeze the state, so each output row reads out
    RMSNorm(S0^T normalize(conv q)).  Identity taps [0,0,0,1] give the token's
    own q; taps [1,0,0,0] give the q of the row three positions earlier."""
    rng = np.random.default_rng(40)
    R, H, dk, dv, W, Wd = 3, 2, 4, 4, 4, 7
    inp = decode_inputs(rng, R, H, dk, dv, accepted=[0, 2, 7], state_std=1.0)
    inp["cached_b"][:] = -800.0  # sigmoid -> 0 exactly
    inp["new_b"][:] = -800.0
    inp["cached_g"][:] = -800.0  # softplus -> 0 exactly, g = 0
    inp["new_g"][:] = -800.0
    Cq = H * (2 * dk + dv)

    def expected(rows_q, S0_rh):
        x = rows_q / np.sqrt(np.sum(rows_q ** 2) + 1e-6)
        o = S0_rh.T @ x
        return o / np.sqrt(np.mean(o ** 2) + 1e-6) * inp["out_w"]

    for taps, shift in [([0, 0, 0, 1], 0), ([1, 0, 0, 0], 3)]:
        cw = np.tile(np.array(taps, dtype=np.float64), (Cq, 1))
        st, tl, o, bad = oracle.decode_verify(**{**inp, "conv_w": cw}, conv_act=0)
        assert bad == 0
        np.testing.assert_array_equal(st, inp["state"])  # frozen
        for r in range(R):
            a = int(inp["accepted"][r])
            seq = list(inp["tail"][r]) + list(inp["cached_qkv"][r, :a]) + list(inp["new_qkv"][r])
            for j in range(Wd + 1):
                p = (W - 1) + a + j - shift
                for h in range(H):
                    ref = expected(seq[p][h * dk:(h + 1) * dk], inp["state"][r, h])
                    np.testing.assert_allclose(o[r, j, h], ref, rtol=1e-12, atol=1e-12)


def test_conv_silu_matches_library_silu(oracle):
    """The short-conv activation ("Noyaux d'inference" section 1, "La fusion":
    the pages name the short convolution but no activation; SiLU is the reading
    adopted, conv_act = 1) against torch.nn.functional.silu, a library routine.

    q branch: identity taps, beta = 0 and g = 0 (the state stays S0 = I),
    w_o = 1, so every output row is RMSNorm(normalise(silu(q_raw))).
    k and v branches: random taps over the cached tail, S0 = 0, beta = 1 and
    g = 0 with no accepted rows, so the state written back after the bonus
    token is normalise(silu(conv(k))) silu(conv(v))^T -- conv first, then the
    activation, then the norm."""
    torch = pytest.importorskip("torch")
    silu = lambda x: torch.nn.functional.silu(torch.from_numpy(np.asarray(x, dtype=np.float64))).numpy()
    rng = np.random.default_rng(45)
    R, H, d, W, Wd = 3, 2, 5, 4, 7
    Cq = H * 3 * d
    inp = decode_inputs(rng, R, H, d, d, accepted=[2, 0, 7], state_std=1.0)
    inp["state"] = np.broadcast_to(np.eye(d), (R, H, d, d)).copy()
    inp["cached_b"][:] = inp["new_b"][:] = -800.0  # logistic -> 0 exactly
    inp["cached_g"][:] = inp["new_g"][:] = -800.0  # softplus -> 0 exactly, g = 0
    inp["out_w"] = np.ones(d)
    cw = np.tile(np.array([0, 0, 0, 1.0]), (Cq, 1))
    _, _, o, bad = oracle.decode_verify(**{**inp, "conv_w": cw}, conv_act=1, eps_out=0.0)
    assert bad == 0
    for r in range(R):
        for j in range(Wd + 1):
            for h in range(H):
                y = silu(inp["new_qkv"][r, j, h * d:(h + 1) * d])
                qh = y / np.sqrt(np.sum(y ** 2) + 1e-6)
                np.testing.assert_allclose(o[r, j, h], qh / np.sqrt(np.mean(qh ** 2)), rtol=1e-12)

    inp = decode_inputs(rng, R, H, d, d, accepted=[0, 0, 0], state_std=1.0)
    inp["state"][:] = 0.0
    inp["new_b"][:] = 800.0  # logistic -> 1 exactly
    inp["new_g"][:] = -800.0
    st, _, _, bad = oracle.decode_verify(**inp, conv_act=1)
    assert bad == 0
    for r in range(R):
        rows = np.concatenate([inp["tail"][r], inp["new_qkv"][r, :1]], axis=0)  # W rows, oldest first
        conv = np.einsum("jc,cj->c", rows, inp["conv_w"])
        for h in range(H):
            kk = silu(conv[H * d + h * d:H * d + (h + 1) * d])
            kk = kk / np.sqrt(np.sum(kk ** 2) + 1e-6)
            vv = silu(conv[2 * H * d + h * d:2 * H * d + (h + 1) * d])
            np.testing.assert_allclose(st[r, h], np.outer(kk, vv), rtol=1e-12, atol=1e-15)


def test_gates_match_library_functions(oracle):
    """The written-back state exposes the gates: with S0 = 0 one bonus token
    gives S = b k v^T (b = logistic(b_raw)); with b = 0, S = Diag(e^g) S0 where
    g = max(-log(1 + e^{g_raw}), -5) (numpy.logaddexp)."""
    rng = np.random.default_rng(41)
    R, H, dk, dv = 2, 2, 4, 4
    inp = decode_inputs(rng, R, H, dk, dv, accepted=[0, 0], state_std=1.0)
    Cq = H * (2 * dk + dv)
    cw = np.tile(np.array([0, 0, 0, 1.0]), (Cq, 1))
    inp["new_g"][:, 0] = np.linspace(-12, 12, H * dk)  # includes floor-binding values
    # beta part
    z = {**inp, "state": np.zeros_like(inp["state"]), "conv_w": cw}
    st, _, _, _ = oracle.decode_verify(**z, conv_act=0)
    for r in range(R):
        for h in range(H):
            x = inp["new_qkv"][r, 0]
            kk = x[H * dk + h * dk:H * dk + (h + 1) * dk]
            kk = kk / np.sqrt(np.sum(kk ** 2) + 1e-6)
            vv = x[2 * H * dk + h * dv:2 * H * dk + (h + 1) * dv]
            b = 1.0 / (1.0 + np.exp(-inp["new_b"][r, 0, h]))
            np.testing.assert_allclose(st[r, h], b * np.outer(kk, vv), rtol=1e-13, atol=1e-15)
    # decay part
    d = {**inp, "conv_w": cw, "new_b": np.full_like(inp["new_b"], -800.0)}
    st, _, _, _ = oracle.decode_verify(**d, conv_act=0)
    for r in range(R):
        for h in range(H):
            graw = inp["new_g"][r, 0, h * dk:(h + 1) * dk]
            gexp = np.maximum(-np.logaddexp(0.0, graw), -5.0)
            np.testing.assert_allclose(st[r, h], np.exp(gexp)[:, None] * inp["state"][r, h], rtol=1e-13)


def test_output_rows_are_rms_normalised(oracle):
    rng = np.random.default_rng(42)
    R, H, dk, dv = 4, 2, 8, 8
    inp = decode_inputs(rng, R, H, dk, dv)
    inp["out_w"] = 1.0 + 0.2 * rng.standard_normal(dv)
    _, _, o, _ = oracle.decode_verify(**inp, eps_out=0.0)
    rms = np.sqrt(np.mean((o / inp["out_w"]) ** 2, axis=-1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-12)


def test_input_norm_unit_length(oracle):
    """Identity conv, state frozen at S0 = I (dk = dv), w_o = 1: the output row
    is RMSNorm(q_hat) so sum(o^2) = dv, and ||q_hat|| = 1 up to eps."""
    rng = np.random.default_rng(43)
    R, H, d = 2, 1, 6
    inp = decode_inputs(rng, R, H, d, d, accepted=[3, 0], state_std=1.0)
    inp["state"] = np.broadcast_to(np.eye(d), (R, H, d, d)).copy()
    inp["cached_b"][:] = inp["new_b"][:] = -800.0
    inp["cached_g"][:] = inp["new_g"][:] = -800.0
    inp["out_w"] = np.ones(d)
    Cq = H * 3 * d
    cw = np.tile(np.array([0, 0, 0, 1.0]), (Cq, 1))
    _, _, o, _ = oracle.decode_verify(**{**inp, "conv_w": cw}, conv_act=0, eps_out=0.0)
    for r in range(R):
        for j in range(8):
            row = inp["new_qkv"][r, j, :d]
            np.testing.assert_allclose(o[r, j, 0], row / np.sqrt(np.mean(row ** 2)), rtol=1e-10)


def test_invalid_accepted_length_skips_request(oracle):
    rng = np.random.default_rng(44)
    R, H, dk, dv = 4, 2, 4, 4
    inp = decode_inputs(rng, R, H, dk, dv, accepted=[2, 9, -1, 7])
    st, tl, o, bad = oracle.decode_verify(**inp)
    assert bad == 2
    for r in (1, 2):
        np.testing.assert_array_equal(st[r], inp["state"][r])
        np.testing.assert_array_equal(tl[r], inp["tail"][r])
        assert np.all(o[r] == 0)
    ok = {**inp, "accepted": np.array([2, 0, 0, 7], dtype=np.int32)}
    st2, tl2, o2, _ = oracle.decode_verify(**ok)
    for r in (0, 3):
        np.testing.assert_array_equal(st[r], st2[r])
        np.testing.assert_array_equal(o[r], o2[r])


def test_state_traffic_arithmetic():
    rows = dict((r[0], int(r[1])) for r in read_golden("state_traffic_example.txt"))
    from kda_gated_delta_02_gb300 import synth
    assert synth.state_bytes(rows["layers"], rows["heads"], rows["dk"], rows["dv"],
                             rows["bytes_per_elem"]) == rows["state_bytes_all_layers"]


# --------------------------------------------------------------------------- backward
def _fd_case(rng, lens, H=2, dk=3, dv=2, floor_frac=0.25):
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -np.abs(rng.standard_normal((T, H, dk)))  # above the floor, well away from it
    below = rng.random((T, H, dk)) < floor_frac
    g[below] = -5.0 - 0.5 - rng.random(int(below.sum()))  # under the floor by more than the step
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = 0.3 * rng.standard_normal((len(lens), H, dk, dv))
    Wo = rng.standard_normal((T, H, dv))
    Ws = rng.standard_normal((len(lens), H, dk, dv))
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, cu=cu), Wo, Ws


def test_backward_matches_central_differences(oracle):
    """The reverse-mode oracle against central differences of the forward
    oracle's loss <o, Wo> + <S_final, Ws> (h = 1e-6, fp64), for every element of
    q, k, v, g, beta and S0, on packed sequences (one of length 1) with part of
    g under the floor (derivative 0 there) and a scale."""
    rng = np.random.default_rng(90)
    x, Wo, Ws = _fd_case(rng, [5, 1, 4])
    scale = 0.7

    def loss(d):
        o, Sf = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], S0=d["S0"], scale=scale)
        return float(np.sum(o * Wo) + np.sum(Sf * Ws))

    dq, dk, dv, dg, db, dS0 = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], Wo,
                                              S0=x["S0"], dS_final=Ws, scale=scale)
    grads = dict(q=dq, k=dk, v=dv, g=dg, beta=db, S0=dS0)
    h = 1e-6
    for name, gr in grads.items():
        fd = np.zeros_like(gr)
        for idx in np.ndindex(gr.shape):
            xp = {kk: vv.copy() for kk, vv in x.items()}
            xm = {kk: vv.copy() for kk, vv in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (loss(xp) - loss(xm)) / (2 * h)
        err = np.max(np.abs(fd - gr)) / max(1e-3, np.max(np.abs(fd)))
        assert err < 1e-6, f"d{name}: relative error {err:.2e}"
    assert np.all(dg[x["g"] < -5.0] == 0.0)  # the floor passes no gradient


def test_backward_without_final_state_gradient_and_beta_zero(oracle):
    """With beta = 0 nothing is written: o_t = scale S_t^T q_t with
    S_t = D_t..D_1 S0, so dq, dS0 have closed forms and dk = dv = 0."""
    rng = np.random.default_rng(91)
    T, H, dk, dv = 4, 1, 3, 2
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -np.abs(rng.standard_normal((T, H, dk)))
    beta = np.zeros((T, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    do = rng.standard_normal((T, H, dv))
    dq, dkk, dvv, dg, db, dS0 = oracle.backward(q, k, v, g, beta, [0, T], do, S0=S0)
    np.testing.assert_array_equal(dkk, 0.0)
    np.testing.assert_array_equal(dvv, 0.0)
    decay = np.cumprod(np.exp(g[:, 0]), axis=0)  # [T, dk]: prod_{r<=t} e^{g_r}
    for t in range(T):
        St = decay[t][:, None] * S0[0, 0]
        np.testing.assert_allclose(dq[t, 0], St @ do[t, 0], rtol=1e-12, atol=1e-12)
    want = sum(np.outer(decay[t] * q[t, 0], do[t, 0]) for t in range(T))
    np.testing.assert_allclose(dS0[0, 0], want, rtol=1e-12, atol=1e-12)


def test_nan_log_decay_takes_the_floor(oracle):
    """A NaN log-decay acts exactly as g = g_min (the floor takes the non-NaN
    operand, as an IEEE maximum does): prefill, segment transitions, the
    backward (dg included) and the chunk-form reverse pass give identical
    results; in verify a NaN raw gate acts as +inf (whose decay 1 / (1 + e^g)
    is 0, floored to e^{g_min})."""
    from oracle import chunk_reverse
    rng = np.random.default_rng(97)
    T, H, dk, dv = 40, 2, 6, 5
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    nan = rng.random(g.shape) < 0.2
    g_nan, g_flr = g.copy(), g.copy()
    g_nan[nan] = np.nan
    g_flr[nan] = G_MIN
    cu = np.array([0, 25, T], dtype=np.int32)
    S0 = 0.1 * rng.standard_normal((2, H, dk, dv))
    for a, b in zip(oracle.prefill(q, k, v, g_nan, beta, cu, S0=S0), oracle.prefill(q, k, v, g_flr, beta, cu, S0=S0)):
        np.testing.assert_array_equal(a, b)
    for a, b in zip(oracle.segment_transition(k[:, :1], v[:, :1], g_nan[:, :1], beta[:, :1]),
                    oracle.segment_transition(k[:, :1], v[:, :1], g_flr[:, :1], beta[:, :1])):
        np.testing.assert_array_equal(a, b)
    do = rng.standard_normal((T, H, dv))
    bn = oracle.backward(q, k, v, g_nan, beta, cu, do, S0=S0)
    bf = oracle.backward(q, k, v, g_flr, beta, cu, do, S0=S0)
    for a, b in zip(bn, bf):
        np.testing.assert_array_equal(a, b)
    assert np.all(np.isfinite(bn[3]))
    rn = chunk_reverse.chunk_form_backward_head(q[:, 0], k[:, 0], v[:, 0], g_nan[:, 0], beta[:, 0], do[:, 0], C=16)
    rf = chunk_reverse.chunk_form_backward_head(q[:, 0], k[:, 0], v[:, 0], g_flr[:, 0], beta[:, 0], do[:, 0], C=16)
    for a, b in zip(rn, rf):
        np.testing.assert_array_equal(a, b)
    inp = decode_inputs(rng, 4, 2, 4, 3)
    i_nan, i_inf = dict(inp), dict(inp)
    for key in ("cached_g", "new_g"):
        m = rng.random(inp[key].shape) < 0.3
        i_nan[key] = np.where(m, np.nan, inp[key])
        i_inf[key] = np.where(m, np.inf, inp[key])
    for a, b in zip(oracle.decode_verify(**i_nan), oracle.decode_verify(**i_inf)):
        np.testing.assert_array_equal(a, b)
