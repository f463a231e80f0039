"""The joint-training attention mask (GravityOCR review §3.1 "Joint
AR-Diffusion Training"; the Trillion Labs blog's three-stream figure).

* the oracle's mask, written entry by entry from the rule text, has the
  structure the pages state (clean rows never read the corrupted streams;
  a corrupted block reads its whole block and only earlier clean blocks;
  the two corrupted streams never read each other);
* the library's per-row key intervals (gocr_three_stream_ranges, host code
  of the C ABI, no GPU) reproduce that mask exactly, edge sizes included.
"""
import numpy as np
import pytest

import oracle


def _mask_from_ranges(lim, lo2, hi2):
    k = np.arange(len(lim))[None, :]
    return (k <= lim[:, None]) | ((k >= lo2[:, None]) & (k <= hi2[:, None]))


@pytest.mark.parametrize("P,N,B", [(3, 10, 4), (0, 7, 3), (5, 8, 8), (4, 9, 32), (2, 6, 1), (6, 0, 4), (16, 40, 8)])
def test_library_ranges_equal_the_oracle_mask(P, N, B):
    from self_speculative_block_gb300 import gocr
    lim, lo2, hi2, pos = gocr.three_stream_ranges(P, N, B)
    want = oracle.three_stream_mask(P, N, B)
    assert np.array_equal(_mask_from_ranges(lim, lo2, hi2), want)
    # rotary positions: the prefix at 0..P-1, each stream's response token i at P + i
    if N:
        np.testing.assert_array_equal(pos, np.concatenate([np.arange(P)] + [P + np.arange(N)] * 3))


def test_mask_structure_from_the_pages():
    P, N, B = 3, 11, 4
    m = oracle.three_stream_mask(P, N, B)
    pre, cl = slice(0, P), slice(P, P + N)
    c1, c2 = slice(P + N, P + 2 * N), slice(P + 2 * N, P + 3 * N)
    # every stream reads the whole prefix causally / fully; the prefix reads nothing else
    assert m[:P, P:].sum() == 0 and m[P:, pre].all()
    # the clean stream is causal and never reads a corrupted stream
    assert np.array_equal(m[cl, cl], np.tril(np.ones((N, N), bool))) and not m[cl, P + N:].any()
    # the corrupted streams never read each other
    assert not m[c1, c2].any() and not m[c2, c1].any()
    for s in (c1, c2):
        blk = np.arange(N) // B
        same = blk[:, None] == blk[None, :]
        assert np.array_equal(m[s, s], same)                    # own block, bidirectional
        assert np.array_equal(m[s, cl], blk[None, :] < blk[:, None])  # earlier clean blocks only
    # every row reads at least itself
    assert np.diag(m).all()


def test_one_block_and_unit_blocks():
    P, N = 2, 6
    m = oracle.three_stream_mask(P, N, N)  # one block: a corrupted stream reads all of itself and no clean token
    c1 = slice(P + N, P + 2 * N)
    assert m[c1, c1].all() and not m[c1, P:P + N].any()
    m1 = oracle.three_stream_mask(P, N, 1)  # unit blocks: token i reads clean tokens before i and itself
    assert np.array_equal(m1[c1, P:P + N], np.tril(np.ones((N, N), bool), -1))
    assert np.array_equal(m1[c1, c1], np.eye(N, dtype=bool))
