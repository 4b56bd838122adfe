"""GPU flat bf16 indexer (one CTA per SM scores an even share of all rows'
tiles; the CTA that completes a row selects it) against the oracle.

Its selection must be exactly the Top-K of the scores the cluster kernel
produces for the same inputs (the two kernels score with the same MMA shape
and epilogue), and its index sets must match the oracle's up to
near-threshold positions.  Covers ragged decode rows, rows shorter than K,
more CTAs than tiles, several rows per CTA, rows at the staging limit, a
causal prefill forced onto the flat kernel, contiguous pages, the tie rule
and a bad page id."""
import numpy as np
import pytest
import torch

from _util import check_index_sets, logical_rows, score_magnitude, to_device, tuning
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu


def _flat(wl, K, force=True):
    import indexer_top_sparse_gb300 as d
    t = to_device(wl)
    maxp = wl.page_table.shape[1]
    with tuning(indexer_flat=1 if force else 0):
        n = d.index_topk_workspace_size(wl.B, wl.T, K, maxp, wl.page_size)
        assert n > 256, "the flat indexer applies to this shape"
        ws = d.Workspace(n)
        idx = d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"], K,
                               workspace=ws)
        ws.check()
        # a second call in the same workspace gives the same indices
        idx2 = d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"],
                                K, workspace=ws)
        ws.check()
    idx, idx2 = idx.cpu().numpy(), idx2.cpu().numpy()
    assert np.array_equal(idx, idx2)
    return idx


def _cluster_scores(wl, K):
    import indexer_top_sparse_gb300 as d
    t = to_device(wl)
    ld = int(wl.query_pos().max()) + 1
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device="cuda")
    ws = d.Workspace(256)
    with tuning(indexer_flat=-1):
        idx, sc = d.dsa_index_scores(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"],
                                     t["cu_q"], K, scores, workspace=ws)
    ws.check()
    return idx.cpu().numpy(), sc.cpu().numpy()


def _check(orc, wl, K, rows=None, force=True):
    idx = _flat(wl, K, force)
    cidx, sc = _cluster_scores(wl, K)
    pos = wl.query_pos()
    rows = list(range(wl.T)) if rows is None else rows
    for t in range(wl.T):
        n = int(pos[t]) + 1
        own = orc.topk_rows(sc[t:t + 1, :n], np.array([n], np.int32), K)[0]
        assert np.array_equal(idx[t], own), f"row {t}: flat selection differs from the Top-K of the scores"
    assert np.array_equal(idx, cidx)
    ref_idx, ref_sc = orc.index_topk(wl.q_idx, wl.head_w, wl.k_idx, wl.page_table, wl.seq_lens, wl.cu_q, K,
                                     wl.page_size, rows=np.array(rows, np.int32), want_scores=True,
                                     ld_scores=sc.shape[1])
    for r, t in enumerate(rows):
        n = int(pos[t]) + 1
        b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
        mag = score_magnitude(wl.q_idx[t], wl.head_w[t], logical_rows(wl.k_idx, wl.page_table[b], wl.page_size, n))
        err = np.abs(sc[t, :n].astype(np.float64) - ref_sc[r, :n])
        assert np.all(err <= 1e-3 * np.maximum(np.abs(ref_sc[r, :n]), mag) + 1e-30)
        check_index_sets(idx[t], ref_idx[r], ref_sc[r], n, K)
    return idx


def test_flat_decode_ragged(orc):
    lens = [1, 63, 64, 65, 127, 128, 129, 1000, 2047, 2048, 2049, 5000]
    wl = make_workload("flat_ragged", lens, [1] * len(lens), H=16, K=256, page_size=64, seed=81, with_kv=False)
    _check(orc, wl, 256)


def test_flat_fewer_tiles_than_ctas(orc):
    wl = make_workload("flat_tiny", [100, 300, 40], [1, 1, 1], H=16, K=64, page_size=64, seed=82, with_kv=False)
    _check(orc, wl, 64)


def test_flat_many_rows_per_cta(orc):
    rng = np.random.default_rng(83)
    lens = rng.integers(1, 700, size=400)
    wl = make_workload("flat_many", lens, [1] * len(lens), H=16, K=128, page_size=64, seed=83, with_kv=False)
    _check(orc, wl, 128, rows=list(range(0, 400, 37)) + [399])


def test_flat_long_rows(orc):
    # 32768-position rows (the decode benchmark's length), K = 2048
    wl = make_workload("flat_long", [32768, 32700, 20000, 32768], [1] * 4, H=16, K=2048, page_size=64, seed=84,
                       with_kv=False)
    _check(orc, wl, 2048, rows=[0, 2])


def test_flat_staging_limit(orc):
    # rows as long as the selection can stage (the query slots and a five-tile ring)
    wl = make_workload("flat_limit", [49152, 300], [1, 1], H=16, K=1024, page_size=64, seed=85, with_kv=False)
    _check(orc, wl, 1024, rows=[0, 1])


def test_flat_forced_on_a_causal_prefill(orc):
    wl = make_workload("flat_prefill", [700], [300], H=16, K=128, page_size=128, permute=False, seed=86,
                       with_kv=False)
    _check(orc, wl, 128, rows=[0, 1, 63, 64, 127, 128, 299])


def test_flat_contiguous_page(orc):
    wl = make_workload("flat_b1", [2048], [1], H=16, K=256, page_size=2048, permute=False, seed=87, with_kv=False)
    _check(orc, wl, 256)


def test_flat_all_equal_scores_take_lowest_positions():
    wl = make_workload("flat_zeros", [3000, 77], [1, 1], H=16, K=256, page_size=64, seed=88, with_kv=False)
    wl.q_idx[:] = 0
    idx = _flat(wl, 256)
    assert np.array_equal(idx[0], np.arange(256))
    assert np.array_equal(idx[1, :77], np.arange(77)) and np.all(idx[1, 77:] == -1)


def test_flat_bad_page_is_reported(orc):
    import indexer_top_sparse_gb300 as d
    wl = make_workload("flat_bad", [500, 900], [1, 1], H=16, K=64, page_size=64, seed=89, with_kv=False)
    t = to_device(wl)
    pt = t["page_table"].clone()
    pt[0, 3] = 10_000
    with tuning(indexer_flat=1):
        ws = d.Workspace(d.index_topk_workspace_size(wl.B, wl.T, 64, wl.page_table.shape[1], wl.page_size))
        d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], pt, t["seq_lens"], t["cu_q"], 64, workspace=ws)
        with pytest.raises(d.DSAError) as e:
            ws.check()
        assert e.value.code == 4
        ws.check()
        # the same workspace then serves a correct call
        idx = d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"], 64,
                               workspace=ws).cpu().numpy()
        ws.check()
    ref_idx, ref_sc = orc.index_topk(wl.q_idx, wl.head_w, wl.k_idx, wl.page_table, wl.seq_lens, wl.cu_q, 64,
                                     wl.page_size, rows=np.array([0, 1], np.int32), want_scores=True)
    for r in range(2):
        check_index_sets(idx[r], ref_idx[r], ref_sc[r], int(wl.seq_lens[r]), 64)


def test_small_workspace_keeps_the_cluster_kernel(orc):
    # a workspace of only the error block runs the cluster kernel (same result)
    import indexer_top_sparse_gb300 as d
    wl = make_workload("flat_ws", [3000, 1200], [1, 1], H=16, K=256, page_size=64, seed=90, with_kv=False)
    t = to_device(wl)
    ws = d.Workspace(256)
    idx = d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"], 256,
                           workspace=ws).cpu().numpy()
    ws.check()
    assert np.array_equal(idx, _flat(wl, 256))
