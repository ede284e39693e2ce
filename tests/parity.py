"""Error measures for GPU-vs-oracle parity.

Normwise relative error of one slice: max|x - y| / max|y| (y = oracle).  A
tensor's error is the maximum over its per-head slices.  Bars (fixed in the
tests that use them): 2e-2 for bf16 / normalised outputs, 1e-2 for states.
"""
import numpy as np

OUT_TOL = 2e-2
STATE_TOL = 1e-2


def normwise_err(x, y, head_axis):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert x.shape == y.shape, (x.shape, y.shape)
    if x.size == 0:
        return 0.0
    xs = np.moveaxis(x, head_axis, 0).reshape(x.shape[head_axis], -1)
    ys = np.moveaxis(y, head_axis, 0).reshape(y.shape[head_axis], -1)
    num = np.max(np.abs(xs - ys), axis=1)
    den = np.maximum(np.max(np.abs(ys), axis=1), 1e-30)
    assert np.all(np.isfinite(xs)), "non-finite GPU values"
    return float(np.max(num / den))


def to64(t):
    return t.detach().to("cpu").double().numpy()


def _align256(n):
    return (n + 255) // 256 * 256


def pipe_wanted(T, H, units, one_piece, sms=152):
    return not one_piece and T // 64 + units >= 64 and units * H < sms


def split_layout(T, H, units, room, one_piece, sms=152):
    """Pieces of the two-kernel prefill with room for the operand blobs of
    `room` chunk slots, as the library lays them out: (slots per piece, blob
    buffers, pieces, bytes of the area: slot list, item counters, two carry
    states, blobs).  All slots form one piece when they fit and the call does
    not pipeline (few slots (< 64), walks with a CTA for every SM, or a
    context-parallel call); otherwise two buffers of at most a quarter of the
    slots each, so the pieces pipeline."""
    n = T // 64 + units
    want = -(-n // 4) if pipe_wanted(T, H, units, one_piece, sms) else n
    piece, nbuf = 0, 1
    if room >= n and want >= n:
        piece = n
    elif room >= 2:
        piece, nbuf = min(want, room // 2), 2
    elif room >= 1:
        piece = 1
    pieces = 0
    if piece:
        pieces = -(-n // piece)
        piece = -(-n // pieces)
        if pieces == 1:
            nbuf = 1
    else:
        nbuf = 0
    fixed = _align256(n * 8) + _align256(n * 4) + _align256(2 * 2 * H * 128 * 128 * 4)
    return piece, nbuf, pieces, fixed + _align256(nbuf * piece * H * 66048)


def split_wanted_room(T, H, units, one_piece, sms=152):
    """Blob room (slots) kda_chunk_fwd_prep_workspace_size asks for."""
    n = T // 64 + units
    want = 2 * -(-n // 4) if pipe_wanted(T, H, units, one_piece, sms) else n
    cap = (16384 << 20) // (H * 66048)
    return min(want, max(cap, 1))
