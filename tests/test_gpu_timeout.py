"""Failure detection without a GPU fault.

Every pipeline wait inside the kernels is bounded.  When one runs out, the
kernel records DSA_ERR_TIMEOUT in the workspace error word, stops its
pipeline, lets its own copies and tensor-core work finish, frees its tensor
memory and returns (the indexer's CTAs still pass every cluster barrier
together), so the context stays usable.  A test-only wait limit of one
microsecond (dsa_workspace_set_wait_limit) makes the waits of the fused
indexer (its cluster and flat forms) and of the sparse MLA run out on purpose: nothing is left unset,
every wait simply gives up early.  The same call with the default limit is
then correct again, checked against the oracle.  No kernel is made to fault
or hang."""
import numpy as np
import pytest

from _util import check_index_sets, dev, to_device, tuning
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu

TIMEOUT = 6


def _expect_timeout(d, ws):
    with pytest.raises(d.DSAError) as e:
        ws.check()
    assert e.value.code == TIMEOUT
    ws.check()  # the error word was cleared


@pytest.mark.parametrize("flat", [1, -1], ids=["flat", "cluster"])
def test_indexer_wait_runs_out_then_recovers(orc, flat):
    import indexer_top_sparse_gb300 as d
    wl = make_workload("timeout_idx", [32768] * 8, [1] * 8, H=16, K=2048, page_size=64, seed=61, with_kv=False)
    t = to_device(wl)
    with tuning(indexer_flat=flat):
        ws = d.Workspace(d.index_topk_workspace_size(wl.B, wl.T, wl.K, wl.max_pages, wl.page_size))
        ws.set_wait_limit(1)
        d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"], wl.K,
                         workspace=ws)
        _expect_timeout(d, ws)
        ws.set_wait_limit(0)
        idx = d.dsa_index_topk(t["q_idx"], t["head_w"], t["k_idx"], t["page_table"], t["seq_lens"], t["cu_q"],
                               wl.K, workspace=ws)
        ws.check()
    idx = idx.cpu().numpy()
    rows = np.array([0, 5], np.int32)
    ref_idx, ref_sc = orc.index_topk(wl.q_idx, wl.head_w, wl.k_idx, wl.page_table, wl.seq_lens, wl.cu_q, wl.K,
                                     wl.page_size, rows=rows, want_scores=True)
    for r, t_ in enumerate(rows):
        check_index_sets(idx[t_], ref_idx[r], ref_sc[r], int(wl.seq_lens[t_]), wl.K)


def test_sparse_mla_wait_runs_out_then_recovers(orc):
    import indexer_top_sparse_gb300 as d
    rng = np.random.default_rng(62)
    wl = make_workload("timeout_mla", [6000] * 16, [1] * 16, H=128, K=2048, page_size=64, seed=62, with_idx=False)
    idx = np.full((wl.T, wl.K), -1, np.int32)
    for r in range(wl.T):
        idx[r] = np.sort(rng.choice(int(wl.seq_lens[r]), wl.K, replace=False))
    t = to_device(wl)
    idx_d = dev(idx)
    # the default decode form: independent 64-head CTAs on the split grid
    with tuning(mla_dsplit=-1, mla_stream_k=-1, mla_pair=-1):
        ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, wl.K))
        ws.set_wait_limit(1)
        d.dsa_sparse_mla(t["q"], t["kv"], t["page_table"], t["seq_lens"], t["cu_q"], idx_d, wl.scale, workspace=ws)
        _expect_timeout(d, ws)
        ws.set_wait_limit(0)
        out = d.dsa_sparse_mla(t["q"], t["kv"], t["page_table"], t["seq_lens"], t["cu_q"], idx_d, wl.scale,
                               workspace=ws)
        ws.check()
    rows = np.array([0, 9, 15], np.int32)
    ref, _ = orc.sparse_mla(wl.q, wl.kv, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size, rows=rows)
    np.testing.assert_allclose(out.float().cpu().numpy()[rows], ref, atol=2e-2, rtol=1e-2)
