"""Philox4x32-10 counter-based generator and the uniforms / Gumbel variates the
method draws from it.  Test infrastructure only (see oracle/__init__.py).

Generator: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
1, 2, 3", SC'11, section 4 (the Philox S-box: two 32x32->64 multiplies per
round, Weyl-sequence key schedule, 10 rounds for the 4x32 variant).  Written
here from that definition; pinned by the generator's published known-answer
vectors in tests/golden/philox4x32_10_kat.txt.

The pages draw random numbers in sampling, acceptance and residual sampling
(DeepSpec walkthrough, section 3.2 "sample_block_tokens" and section 8.2
"verify_draft_tokens") without saying how; the reading used here keys every
draw by (seed, request b, position k, index, stream):

    counter = (index >> 2, k, b, stream),  key = (seed & 0xffffffff, seed >> 32)
    word    = output word (index & 3)

Streams separate the independent draws of one round (see STREAM_* below).
"""
import numpy as np

_MASK = np.uint64(0xFFFFFFFF)
_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)

# One stream per independent draw of a round.
STREAM_DRAFT_TOKEN = 0     # Gumbel noise of the draft sample x_k, one word per vocabulary index
STREAM_ACCEPT = 1          # acceptance uniform u of the rejection test (index 0)
STREAM_VERIFY_TOKEN = 2    # Gumbel noise of the token the verifier emits: the residual draw at the
                           # rejected position, the bonus draw from p_t at row l* + 1, or the draw
                           # from p_t when a residual has no mass (only one of them per request)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox4x32 rounds on counters (c0..c3) under key (k0, k1).

    Every argument is an integer or an integer array of 32-bit values; the
    four returned arrays are the output words.  Each round multiplies c0 by
    0xD2511F53 and c2 by 0xCD9E8D57 (full 64-bit products), then forms
    (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0));
    the key is bumped by (0x9E3779B9, 0xBB67AE85) between rounds.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK for c in (c0, c1, c2, c3))
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for _ in range(10):
        p0 = _M0 * c0            # < 2**64: exact in uint64
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + _W0) & _MASK
        k1 = (k1 + _W1) & _MASK
    return c0, c1, c2, c3


def draw_words(seed, b, k, stream, index):
    """The 32-bit word for (seed, request b, position k, stream, index).

    b and index may be arrays (broadcast together); k and stream are scalars.
    """
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    index = np.asarray(index, dtype=np.uint64)
    b = np.asarray(b, dtype=np.uint64)
    index, b = np.broadcast_arrays(index, b)
    words = philox4x32_10(index >> np.uint64(2), np.uint64(k), b, np.uint64(stream),
                          seed & 0xFFFFFFFF, seed >> 32)
    sel = (index & np.uint64(3)).astype(np.int64)
    out = np.choose(sel, words)
    return out.astype(np.uint64)


def row_words(seed, b, k, stream, V):
    """[R, V] words of requests b[R] at position k for indices 0 .. V-1: the same
    values as draw_words, with each Philox block computed once for its four words."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    b = np.atleast_1d(np.asarray(b, dtype=np.uint64))
    nq = -(-int(V) // 4)
    c0 = np.arange(nq, dtype=np.uint64)[None, :]
    words = philox4x32_10(c0, np.uint64(k), b[:, None], np.uint64(stream), seed & 0xFFFFFFFF, seed >> 32)
    out = np.stack(words, axis=-1).reshape(b.shape[0], nq * 4)     # word v & 3 of block v >> 2
    return out[:, :int(V)]


def uniform_open(words):
    """u in (0, 1): ((w >> 9) + 1/2) * 2**-23, an odd multiple of 2**-24."""
    w = np.asarray(words, dtype=np.uint64)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def uniform_accept(words):
    """u in [0, 1): (w >> 8) * 2**-24, the acceptance test's uniform."""
    w = np.asarray(words, dtype=np.uint64)
    return (w >> np.uint64(8)).astype(np.float64) * 2.0 ** -24


def gumbel(u):
    """Standard Gumbel variate -ln(-ln u) for u in (0, 1), in float64."""
    u = np.asarray(u, dtype=np.float64)
    return -np.log(-np.log(u))
