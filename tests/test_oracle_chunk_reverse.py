"""The chunk (WY) form of the backward (oracle/chunk_reverse.py) against the
token-level reverse mode of the oracle (itself pinned by central differences
of the forward oracle), and its forward half against the forward oracle.

CPU only: packed ragged sequences, chunk lengths that split them into many
chunks (with a partial last chunk), one chunk per sequence, one token per
chunk (then A = 0 and the chunk form is the token recurrence), part of g
under the floor and some exactly at it.
"""
import numpy as np
import pytest

from oracle import chunk_reverse

G_MIN = -5.0
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def _case(rng, lens, H, dk, dv, below=0.1, at=0.05):
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -np.logaddexp(0.0, rng.standard_normal((T, H, dk)))
    u = rng.random((T, H, dk))
    g[u < below] = -5.5 - rng.random(int((u < below).sum()))
    g[(u >= below) & (u < below + at)] = G_MIN
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    N = len(lens)
    S0 = 0.05 * rng.standard_normal((N, H, dk, dv))
    do = rng.standard_normal((T, H, dv))
    dSf = 0.1 * rng.standard_normal((N, H, dk, dv))
    return q, k, v, g, beta, cu, S0, do, dSf


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("C,lens", [(16, [37, 0, 64, 5]), (64, [130, 64]), (8, [23]), (1, [9, 4]),
                                    (256, [100, 0, 3])])
def test_chunk_reverse_matches_token_reverse(oracle, C, lens):
    rng = np.random.default_rng(C * 7 + len(lens))
    H, dk, dv = 2, 8, 6
    q, k, v, g, beta, cu, S0, do, dSf = _case(rng, lens, H, dk, dv)
    got = chunk_reverse.chunk_form_backward(q, k, v, g, beta, cu, do, S0=S0, dS_final=dSf, C=C, scale=0.7)
    ref = oracle.backward(q, k, v, g, beta, cu, do, S0=S0, dS_final=dSf, scale=0.7)
    for name, a, b in zip(NAMES, got[2:], ref):
        assert _rel(a, b) <= 1e-10, f"{name}: {_rel(a, b):.2e}"
    # the floor: no gradient below it, gradient at it
    assert np.all(got[5][g < G_MIN] == 0.0)
    o_ref, S_ref = oracle.prefill(q, k, v, g, beta, cu, S0=S0, scale=0.7)
    assert _rel(got[0], o_ref) <= 1e-11
    assert _rel(got[1], S_ref) <= 1e-11


def test_chunk_reverse_absent_states_d128(oracle):
    """d = 128, two chunks of 64 and a partial one, no initial state and no
    final-state gradient."""
    rng = np.random.default_rng(5)
    q, k, v, g, beta, cu, _, do, _ = _case(rng, [150], 1, 128, 128)
    got = chunk_reverse.chunk_form_backward(q, k, v, g, beta, cu, do, C=64)
    ref = oracle.backward(q, k, v, g, beta, cu, do)
    for name, a, b in zip(NAMES, got[2:], ref):
        assert _rel(a, b) <= 1e-10, f"{name}: {_rel(a, b):.2e}"


def test_chunk_reverse_gradient_of_a_chunk_boundary_state(oracle):
    """dS0 of the second chunk is the state gradient the first chunk receives:
    splitting a sequence's reverse pass at a chunk boundary by hand (second
    half first, its dS0 fed to the first half as dS_final) gives the same
    gradients as one pass."""
    rng = np.random.default_rng(9)
    q, k, v, g, beta, cu, S0, do, dSf = _case(rng, [48], 1, 8, 8)
    h = 0
    full = chunk_reverse.chunk_form_backward_head(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], do[:, h],
                                                  S0[0, h], dSf[0, h], C=16)
    _, S1 = oracle.prefill(q[:32], k[:32], v[:32], g[:32], beta[:32], [0, 32], S0=S0)
    second = chunk_reverse.chunk_form_backward_head(q[32:, h], k[32:, h], v[32:, h], g[32:, h], beta[32:, h],
                                                    do[32:, h], S1[0, h], dSf[0, h], C=16)
    first = chunk_reverse.chunk_form_backward_head(q[:32, h], k[:32, h], v[:32, h], g[:32, h], beta[:32, h],
                                                   do[:32, h], S0[0, h], second[7], C=16)
    for idx, name in zip(range(2, 7), NAMES[:5]):
        joined = np.concatenate([first[idx], second[idx]])
        assert _rel(joined, full[idx]) <= 1e-12, name
    assert _rel(first[7], full[7]) <= 1e-12


def test_serial_chain_then_independent_chunks(oracle):
    """The decomposition a chunked kernel would use: the state-gradient chain
    alone (serial over chunks), then every chunk's token gradients from its
    (S_in, dS_C) pair in any order, equal the whole reverse pass."""
    rng = np.random.default_rng(17)
    q, k, v, g, beta, cu, S0, do, dSf = _case(rng, [150], 1, 16, 8)
    h = 0
    args = (q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], do[:, h])
    full = chunk_reverse.chunk_form_backward_head(*args, S0=S0[0, h], dS_final=dSf[0, h], C=32, scale=0.9)
    bounds, S_in, dS_C, dS0 = chunk_reverse.state_gradient_chain(*args, S0=S0[0, h], dS_final=dSf[0, h], C=32,
                                                                 scale=0.9)
    assert _rel(dS0, full[7]) <= 1e-12
    parts = {}
    for c in reversed(range(len(bounds))):  # any order; reversed to show no hidden carry
        c0, c1 = bounds[c]
        parts[c] = chunk_reverse.chunk_token_gradients(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h], g[c0:c1, h],
                                                       beta[c0:c1, h], do[c0:c1, h], S_in[c], dS_C[c], scale=0.9)
    for idx, name in enumerate(NAMES[:5]):
        joined = np.concatenate([parts[c][idx] for c in range(len(bounds))])
        assert _rel(joined, full[2 + idx]) <= 1e-12, name


def _bf16(x):
    """Round to bfloat16 (nearest even) and back."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def test_bf16_operand_error_budget(oracle):
    """Error budget of a tensor-core chunked backward: every product of the
    chunk-form reverse pass with both operands rounded to bf16 and fp32
    accumulation (the inverse exact) stays within 1e-2 of the fp64 gradients
    at d = 128 over 256 tokens (four chunks); with exact products the
    agreement is 1e-10, so the gap is the operand rounding alone."""
    rng = np.random.default_rng(23)
    q, k, v, g, beta, cu, _, do, _ = _case(rng, [256], 1, 128, 128, below=0.0, at=0.0)
    q, k, v, do = (_bf16(x) for x in (q, k, v, do))
    mm16 = lambda a, b: (_bf16(a).astype(np.float32) @ _bf16(b).astype(np.float32)).astype(np.float64)
    h = 0
    got = chunk_reverse.chunk_form_backward_head(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], do[:, h],
                                                 C=64, mm=mm16)
    ref = oracle.backward(q, k, v, g, beta, cu, do)
    errs = {n: _rel(a, np.asarray(b)[:, 0] if np.asarray(b).ndim > 1 and np.asarray(b).shape[0] == 256 else b[0])
            for n, a, b in zip(NAMES, got[2:], ref)}
    assert all(e <= 1e-2 for e in errs.values()), errs
    assert max(errs.values()) >= 1e-4, errs  # the rounding is really applied


@pytest.mark.parametrize("floor_chunks", [False, True])
def test_f32_anchored_matches_f64(oracle, floor_chunks):
    """The fp32 chunk-form reverse pass with 16-token block anchoring against
    the fp64 reverse mode, d = 128 over 200 tokens (a partial last chunk).  With
    two chunks held at the floor (gamma down to -320 inside a chunk, where
    1/e^gamma overflows fp32) everything stays finite and within 2e-5 (fp32
    rounding; measured about 1e-6)."""
    rng = np.random.default_rng(29 + floor_chunks)
    q, k, v, g, beta, cu, S0, do, dSf = _case(rng, [200], 1, 128, 128, below=0.0, at=0.0)
    if floor_chunks:
        g[0:64] = G_MIN
        g[128:192] = G_MIN - 0.5
        gam = np.cumsum(np.maximum(g[0:64, 0], G_MIN), axis=0).astype(np.float32)
        with np.errstate(over="ignore", divide="ignore"):
            assert not np.all(np.isfinite(np.float32(1.0) / np.exp(gam)))  # the naive factor overflows
    h = 0
    got = chunk_reverse.chunk_form_backward_head_f32(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], do[:, h],
                                                     S0[0, h], dSf[0, h], C=64, scale=0.8)
    ref = chunk_reverse.chunk_form_backward_head(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], do[:, h],
                                                 S0[0, h], dSf[0, h], C=64, scale=0.8)
    for name, a, b in zip(("o", "S_final") + NAMES, got, ref):
        assert np.all(np.isfinite(a)), name
        assert _rel(a, b) <= 2e-5, f"{name}: {_rel(a, b):.2e}"
    if floor_chunks:
        assert np.all(got[5][128:192] == 0.0)  # below the floor: no gradient


def test_bf16_rounding_helper_matches_the_pages_example():
    """The bf16 rounding the error-budget test applies reproduces the pages'
    example (tests/golden/bf16_rounding_example.txt): 256.5 rounds to 256 in
    bf16, so the fp32 difference with 256 drops from 0.5 to 0; values bf16
    holds exactly are kept and ties go to even."""
    from conftest import read_golden
    rows = {r[0]: [float(x) for x in r[1:]] for r in read_golden("bf16_rounding_example.txt")}
    a, b, diff = rows["fp32"]
    assert np.float32(a) - np.float32(b) == diff
    ra, rb, rdiff = rows["bf16"]
    assert _bf16(np.array([a]))[0] == ra and _bf16(np.array([b]))[0] == rb
    assert np.float32(_bf16(np.array([a]))[0]) - np.float32(_bf16(np.array([b]))[0]) == rdiff
    # exact values stay; the tie 1 + 2^-8 goes to even (1), 1 + 3 * 2^-8 to 1 + 2^-6
    assert _bf16(np.array([1.5, -3.25, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8])).tolist() == [1.5, -3.25, 1.0,
                                                                                         1 + 2.0 ** -6]


def test_state_gradient_chain_composes_over_segments(oracle):
    """The state-gradient chain is affine in the gradient at a segment's end:
    dS_start = M^T dS_end + r, with M the forward transition of the segment
    (oracle.segment_transition) and r the chain from dS_end = 0.  Composing
    (M^T, r) over segments, last to first, gives the chain's value at every
    segment start, the backward counterpart of the forward's context-parallel
    composition; each segment can then be reversed on its own."""
    rng = np.random.default_rng(31)
    T, seg, C = 192, 64, 32
    q, k, v, g, beta, cu, S0, do, dSf = _case(rng, [T], 1, 16, 8, below=0.05, at=0.02)
    h = 0
    args = lambda a, b: (q[a:b, h], k[a:b, h], v[a:b, h], g[a:b, h], beta[a:b, h], do[a:b, h])
    _, S_in, dS_C, dS0 = chunk_reverse.state_gradient_chain(*args(0, T), S0=S0[0, h], dS_final=dSf[0, h], C=C,
                                                            scale=0.6)
    # the chain's value at each chunk start is dS_C of the chunk before (dS0 at 0)
    at_start = {0: dS0}
    for c in range(1, T // C):
        at_start[c * C] = dS_C[c - 1]
    bounds = [(a, a + seg) for a in range(0, T, seg)]
    maps = []
    for a, b in bounds:
        M, _ = oracle.segment_transition(k[a:b], v[a:b], g[a:b], beta[a:b])
        # the segment's own start state (from the forward), then its chain from zero
        Sa = S_in[a // C]
        r = chunk_reverse.state_gradient_chain(*args(a, b), S0=Sa, dS_final=None, C=C, scale=0.6)[3]
        maps.append((M[h], r))
    dS = dSf[0, h]
    for (a, b), (M, r) in reversed(list(zip(bounds, maps))):
        dS = M.T @ dS + r
        assert _rel(dS, at_start[a]) <= 1e-12, a
