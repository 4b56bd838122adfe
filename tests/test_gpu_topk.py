"""GPU Top-K from given fp32 scores: bit-exact against the oracle's full-sort
selection on the same scores, over ragged lengths, exact ties (in buckets
too large and small enough for the final in-bucket ranking), signed zeros
and every cluster size."""
import numpy as np
import pytest
import torch

from _util import dev

pytestmark = pytest.mark.gpu


def _scores(rng, R, N, ties):
    s = rng.standard_normal((R, N)).astype(np.float32)
    if ties:
        s = np.round(s * 4).astype(np.float32) / 4       # few distinct values: many exact ties
        s[:, ::13] = -0.0
        s[:, 5::13] = 0.0
    return s


@pytest.mark.parametrize("R,N,K,ties", [(3, 1, 1, False), (5, 127, 16, True), (4, 129, 128, False),
                                        (6, 1000, 256, True), (3, 4096, 2048, False), (2, 40000, 2048, True),
                                        (2, 131072, 2048, False), (3, 300, 1000, True)])
def test_topk_from_scores_bit_exact(orc, R, N, K, ties):
    import indexer_top_sparse_gb300 as d
    rng = np.random.default_rng(R * 1000 + N + K)
    s = _scores(rng, R, N, ties)
    lens = rng.integers(0, N + 1, size=R).astype(np.int32)
    lens[0] = N
    ref = orc.topk_rows(s, lens, K)
    got = d.dsa_topk_from_scores(dev(s), dev(lens), K).cpu().numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_topk_every_cluster_size(orc, C):
    import indexer_top_sparse_gb300 as d
    rng = np.random.default_rng(C)
    s = _scores(rng, 4, 5000, True)
    lens = np.array([5000, 4999, 2049, 17], np.int32)
    d.set_tuning("topk_cluster", C)
    try:
        got = d.dsa_topk_from_scores(dev(s), dev(lens), 2048).cpu().numpy()
    finally:
        d.set_tuning("topk_cluster", 0)
    assert np.array_equal(got, orc.topk_rows(s, lens, 2048))


@pytest.mark.parametrize("C", [1, 4, 16])
@pytest.mark.parametrize("K", [1, 333, 2048])
def test_topk_ties_inside_small_bucket(orc, C, K):
    # scores on a 1/1024 grid in [0, 3): a bucket of the top 16 key bits spans
    # 8 grid values, about 50 keys at this length, each value ~7 times, so the
    # threshold bucket is ranked directly and its ties split by position
    import indexer_top_sparse_gb300 as d
    rng = np.random.default_rng(70 + C + K)
    s = (rng.integers(0, 3072, size=(3, 20000)) / 1024.0).astype(np.float32)
    lens = np.array([20000, 19999, 4097], np.int32)
    d.set_tuning("topk_cluster", C)
    try:
        got = d.dsa_topk_from_scores(dev(s), dev(lens), K).cpu().numpy()
    finally:
        d.set_tuning("topk_cluster", 0)
    assert np.array_equal(got, orc.topk_rows(s, lens, K))


def test_topk_all_equal_takes_lowest_positions(orc):
    import indexer_top_sparse_gb300 as d
    s = np.full((2, 3000), 1.5, np.float32)
    s[1] = -0.0
    s[1, ::2] = 0.0
    got = d.dsa_topk_from_scores(dev(s), dev(np.array([3000, 3000], np.int32)), 100).cpu().numpy()
    assert np.array_equal(got[0], np.arange(100)) and np.array_equal(got[1], np.arange(100))
