"""Pins for the oracle's Top-K: the selected set is characterised without
sorting (every selected score beats every unselected one, ties going to the
lower position), checked exhaustively over small tie patterns, against a
library lexicographic sort on random rows, and on closed-form special cases."""
import itertools

import numpy as np


def _check_characterisation(scores, n, K, sel):
    m = min(K, n)
    got = [int(i) for i in sel if i >= 0]
    assert len(got) == m and all(i == -1 for i in sel[m:])
    assert got == sorted(got) and len(set(got)) == m
    S = set(got)
    for i in S:
        assert 0 <= i < n
        for j in range(n):
            if j in S:
                continue
            assert scores[i] > scores[j] or (scores[i] == scores[j] and i < j), (scores, K, got)


def test_topk_exhaustive_tie_patterns(orc):
    vals = [-1.0, -0.0, 0.0, 1.0, 2.5]
    for n in range(0, 6):
        rows = np.array(list(itertools.product(vals, repeat=n)) or [[]], np.float32).reshape(-1, max(n, 1))
        if n == 0:
            rows = np.zeros((1, 1), np.float32)
        for K in range(1, 7):
            lens = np.full(rows.shape[0], n, np.int32)
            out = orc.topk_rows(rows, lens, K)
            for r in range(rows.shape[0]):
                _check_characterisation(rows[r], n, K, out[r])


def test_topk_matches_library_sort(orc):
    rng = np.random.default_rng(5)
    for n, K in [(1000, 17), (4096, 2048), (3000, 5000), (777, 777)]:
        s = rng.standard_normal(n).astype(np.float32)
        s[::7] = s[3]                    # many exact ties
        s[::11] = 0.0
        s[5::11] = -0.0
        out = orc.topk_rows(s[None, :], np.array([n], np.int32), K)[0]
        # library: sort by (-score, position); -0 and +0 compare equal
        key = np.where(s == 0, np.float32(0), s)
        order = np.lexsort((np.arange(n), -key.astype(np.float64)))
        want = np.sort(order[:min(K, n)])
        assert np.array_equal(out[:min(K, n)], want)
        assert np.all(out[min(K, n):] == -1)


def test_topk_special_cases(orc):
    s = np.full((1, 50), 3.25, np.float32)
    out = orc.topk_rows(s, np.array([50], np.int32), 8)[0]
    assert list(out) == list(range(8))                       # all equal -> lowest positions
    out = orc.topk_rows(s, np.array([5], np.int32), 8)[0]
    assert list(out) == [0, 1, 2, 3, 4, -1, -1, -1]          # K >= n -> every valid position
    s = np.arange(50, dtype=np.float32)[None, :]
    out = orc.topk_rows(s, np.array([50], np.int32), 3)[0]
    assert list(out) == [47, 48, 49]
    out = orc.topk_rows(-s, np.array([50], np.int32), 3)[0]
    assert list(out) == [0, 1, 2]
