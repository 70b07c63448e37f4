"""Pins for oracle.philox: the published known-answer vectors of Philox4x32-10
and the distribution of the uniforms and Gumbel variates drawn from it."""
import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append([int(x, 16) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat_rows())
def test_known_answer_vectors(row):
    c, k, expect = row[0:4], row[4:6], row[6:10]
    out = philox.philox4x32_10(*c, *k)
    assert [int(x) for x in out] == expect


def test_draw_words_layout():
    # index -> counter (index >> 2, k, b, stream), word index & 3
    seed = 0x0123456789ABCDEF
    w = philox.draw_words(seed, 5, 3, 2, np.arange(8))
    blk0 = philox.philox4x32_10(0, 3, 5, 2, seed & 0xFFFFFFFF, seed >> 32)
    blk1 = philox.philox4x32_10(1, 3, 5, 2, seed & 0xFFFFFFFF, seed >> 32)
    assert [int(x) for x in w] == [int(x) for x in blk0] + [int(x) for x in blk1]


def test_row_words_equal_draw_words():
    # the per-row fast path computes each Philox block once; the words are the same
    seed = 0xFEEDFACE00C0FFEE
    b = np.array([0, 3, 1023])
    for V in (1, 5, 8, 37):
        rows = philox.row_words(seed, b, 6, philox.STREAM_VERIFY_TOKEN, V)
        ref = philox.draw_words(seed, b[:, None], 6, philox.STREAM_VERIFY_TOKEN, np.arange(V)[None, :])
        assert rows.shape == (3, V) and np.array_equal(rows, ref)


def test_uniform_ranges_exact():
    w = np.array([0, 0xFFFFFFFF, 0x00000200, 0x80000000], dtype=np.uint64)
    u = philox.uniform_open(w)
    assert u[0] == 2.0 ** -24 and u[1] == 1.0 - 2.0 ** -24
    assert np.all((u > 0) & (u < 1))
    # each value is an odd multiple of 2^-24: exactly representable in float32
    assert np.all(u.astype(np.float32).astype(np.float64) == u)
    ua = philox.uniform_accept(w)
    assert ua[0] == 0.0 and ua[1] == 1.0 - 2.0 ** -24 and ua[3] == 0.5
    assert np.all(ua.astype(np.float32).astype(np.float64) == ua)


def test_uniform_and_gumbel_distributions():
    w = philox.draw_words(7, np.arange(200000) // 1000, 1, philox.STREAM_DRAFT_TOKEN,
                          np.arange(200000) % 1000)
    u = philox.uniform_open(w)
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    g = philox.gumbel(u)
    assert stats.kstest(g, "gumbel_r").pvalue > 1e-3
    # a sign or nesting slip (e.g. -ln u, an exponential) is far off
    assert stats.kstest(-np.log(u), "gumbel_r").pvalue < 1e-6


def test_streams_and_keys_independent():
    a = philox.draw_words(1, 0, 1, 0, np.arange(4096))
    b = philox.draw_words(1, 0, 1, 1, np.arange(4096))
    c = philox.draw_words(2, 0, 1, 0, np.arange(4096))
    d = philox.draw_words(1, 1, 1, 0, np.arange(4096))
    e = philox.draw_words(1, 0, 2, 0, np.arange(4096))
    for other in (b, c, d, e):
        assert np.mean(a == other) < 0.01
