"""GPU fused indexer + Top-K against the oracle: scores within 1e-3 relative
(of the score's natural magnitude), selection bit-exact on the GPU's own
scores, and Top-K sets equal to the oracle's except at near-threshold
positions.  Covers ragged decode lengths, page permutation, tiny and
page-boundary lengths, prefill and chunked prefill, every cluster size and
ring depth, and the all-equal-scores tie rule."""
import numpy as np
import pytest
import torch

from _util import check_index_sets, logical_rows, score_magnitude, to_device
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu


def _run(wl, K, ld=None):
    import indexer_top_sparse_gb300 as d
    t = to_device(wl)
    ld = ld or int(wl.seq_lens.max())
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device="cuda")
    ws = d.Workspace(256)
    idx, sc = d.dsa_index_scores(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"], K,
                                 scores, workspace=ws)
    ws.check()
    idx2 = d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"], K,
                            workspace=ws)
    ws.check()
    idx, idx2, sc = idx.cpu().numpy(), idx2.cpu().numpy(), sc.cpu().numpy()
    assert np.array_equal(idx, idx2), "scores hook must not change the selection"
    return idx, sc


def _check(orc, wl, K, rows=None):
    idx, sc = _run(wl, K)
    pos = wl.query_pos()
    rows = range(wl.T) if rows is None else rows
    ref_idx, ref_sc = orc.index_topk(wl.q_idx, wl.head_w, wl.k_idx, wl.page_table, wl.seq_lens, wl.cu_q, K,
                                     wl.page_size, rows=np.array(list(rows), np.int32), want_scores=True,
                                     ld_scores=sc.shape[1])
    near = 0
    for r, t in enumerate(rows):
        n = int(pos[t]) + 1
        b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
        mag = score_magnitude(wl.q_idx[t], wl.head_w[t], logical_rows(wl.k_idx, wl.page_table[b], wl.page_size, n))
        err = np.abs(sc[t, :n].astype(np.float64) - ref_sc[r, :n])
        tol = 1e-3 * np.maximum(np.abs(ref_sc[r, :n]), mag) + 1e-30
        assert np.all(err <= tol), f"row {t}: worst score error {np.max(err / tol):.3g} x tolerance"
        # the kernel's selection is exactly the Top-K of the kernel's own scores
        own = orc.topk_rows(sc[t:t + 1, :n], np.array([n], np.int32), K)[0]
        assert np.array_equal(idx[t], own), f"row {t}: selection differs from Top-K of the kernel's scores"
        near += check_index_sets(idx[t], ref_idx[r], ref_sc[r], n, K)
    return near


def test_decode_ragged_paged(orc):
    lens = [1, 63, 64, 65, 129, 1000, 2047, 2048, 2049, 5000]
    wl = make_workload("ragged", lens, [1] * len(lens), H=16, K=256, page_size=64, seed=1, with_kv=False)
    _check(orc, wl, 256)


def test_decode_small_contiguous(orc):
    wl = make_workload("b1n2048", [2048], [1], H=16, K=256, page_size=2048, permute=False, seed=2, with_kv=False)
    _check(orc, wl, 256)


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_every_cluster_size(orc, C):
    import indexer_top_sparse_gb300 as d
    wl = make_workload("c", [3000, 700, 64], [1, 1, 1], H=16, K=512, page_size=128, seed=3 + C, with_kv=False)
    d.set_tuning("indexer_cluster", C)
    try:
        _check(orc, wl, 512)
    finally:
        d.set_tuning("indexer_cluster", 0)


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_ring_depths(orc, stages):
    # (3 runs as 2: the ring depth is even, two threads issue alternate tiles)
    import indexer_top_sparse_gb300 as d
    wl = make_workload("s", [4100, 2500], [1, 1], H=16, K=300, page_size=64, seed=9, with_kv=False)
    d.set_tuning("indexer_stages", stages)
    try:
        _check(orc, wl, 300)
    finally:
        d.set_tuning("indexer_stages", 0)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_prefill_causal(orc, G):
    import indexer_top_sparse_gb300 as d
    wl = make_workload("prefill", [333], [333], H=16, K=64, page_size=64, permute=False, seed=11, with_kv=False)
    d.set_tuning("indexer_group", G)
    try:
        _check(orc, wl, 64)
    finally:
        d.set_tuning("indexer_group", 0)


def test_chunked_prefill_multi_sequence(orc):
    # chunks of different sequences: their queries are the last positions
    wl = make_workload("chunks", [700, 130, 2200], [200, 7, 65], H=16, K=128, page_size=64, seed=12, with_kv=False)
    _check(orc, wl, 128, rows=list(range(0, wl.T, 3)) + [wl.T - 1])


def test_all_equal_scores_take_lowest_positions():
    import indexer_top_sparse_gb300 as d
    wl = make_workload("zeros", [3000, 77], [1, 1], H=16, K=256, page_size=64, seed=13, with_kv=False)
    wl.q_idx[:] = 0
    idx, sc = _run(wl, 256)
    assert np.all(sc[0, :3000] == 0)
    assert np.array_equal(idx[0], np.arange(256))
    assert np.array_equal(idx[1, :77], np.arange(77)) and np.all(idx[1, 77:] == -1)


def test_bad_page_is_reported():
    import indexer_top_sparse_gb300 as d
    wl = make_workload("bad", [500], [1], H=16, K=64, page_size=64, seed=14, with_kv=False)
    t = to_device(wl)
    pt = t["page_table"].clone()
    pt[0, 3] = 10_000
    ws = d.Workspace(256)
    d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], pt, t["seq_lens"], t["cu_q"], 64, workspace=ws)
    with pytest.raises(d.DSAError) as e:
        ws.check()
    assert e.value.code == 4
    ws.check()  # the error word was cleared


@pytest.mark.parametrize("G", [1, 4])
def test_grid_order_gives_the_same_indices(orc, G):
    # the longest-first row order is a scheduling choice only: with the rows
    # taken in plain grid order the indices are the same, bit for bit (and
    # match the oracle)
    import indexer_top_sparse_gb300 as d
    from _util import tuning
    wl = make_workload("order", [900, 300, 2500], [40, 17, 3], H=16, K=256, page_size=64, seed=71, with_kv=False)
    with tuning(indexer_group=G):
        base, _ = _run(wl, 256)
        with tuning(indexer_order=-1):
            plain, _ = _run(wl, 256)
        _check(orc, wl, 256)
    assert np.array_equal(base, plain)
