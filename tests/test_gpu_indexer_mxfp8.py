"""GPU fused indexer + Top-K on MXFP8 index operands against the oracle.  Both
sides read the same E4M3 codes and E8M0 block scales (made on the CPU by the
oracle's quantiser); scores must agree within 1e-3 relative of the score's
natural magnitude, the selection must be exactly the Top-K of the kernel's
own scores, and the Top-K sets must equal the oracle's except at
near-threshold positions."""
import numpy as np
import pytest
import torch

from _util import check_index_sets, dev
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu


def _quantised(orc, wl):
    q, qs = orc.quant_mxfp8(wl.q_idx)
    k, ks = orc.quant_mxfp8(wl.k_idx)
    return q, qs, k, ks


def _dequant(orc, codes, scales):
    lut = np.array([orc.e4m3_to_f64(c) for c in range(256)])
    slut = np.array([orc.e8m0_to_f64(c) for c in range(256)])
    v = lut[codes].reshape(codes.shape[:-1] + (-1, 32))
    return (v * slut[scales][..., None]).reshape(codes.shape)


def _run(wl, q, qs, k, ks, K):
    import indexer_top_sparse_gb300 as d
    ld = int(wl.seq_lens.max())
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device="cuda")
    ws = d.Workspace(256)
    args = (dev(q), dev(wl.head_w), dev(k), dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q), K)
    kw = dict(q_idx_scale=dev(qs), k_idx_scale=dev(ks), dtype="mxfp8", workspace=ws)
    idx, sc = d.dsa_index_scores(*args, scores, **kw)
    ws.check()
    idx2 = d.dsa_index_topk(*args, **kw)
    ws.check()
    idx, idx2, sc = idx.cpu().numpy(), idx2.cpu().numpy(), sc.cpu().numpy()
    assert np.array_equal(idx, idx2), "scores hook must not change the selection"
    return idx, sc


def _check(orc, wl, K):
    q, qs, k, ks = _quantised(orc, wl)
    idx, sc = _run(wl, q, qs, k, ks, K)
    ref_idx, ref_sc = orc.index_topk(q, wl.head_w, k, wl.page_table, wl.seq_lens, wl.cu_q, K, wl.page_size,
                                     dtype=orc.IDX_MXFP8, q_scale=qs, k_scale=ks, want_scores=True,
                                     ld_scores=sc.shape[1])
    qf = _dequant(orc, q, qs)
    kf = _dequant(orc, k, ks).reshape(-1, 128)
    pos = wl.query_pos()
    near = 0
    for t in range(wl.T):
        n = int(pos[t]) + 1
        b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
        rows = np.array([wl.page_table[b, s // wl.page_size] * wl.page_size + s % wl.page_size for s in range(n)])
        mag = (np.maximum(kf[rows] @ qf[t].T, 0) * np.abs(wl.head_w[t].astype(np.float64))[None, :]).sum(1)
        err = np.abs(sc[t, :n].astype(np.float64) - ref_sc[t, :n])
        tol = 1e-3 * np.maximum(np.abs(ref_sc[t, :n]), mag) + 1e-30
        assert np.all(err <= tol), f"row {t}: worst score error {np.max(err / tol):.3g} x tolerance"
        own = orc.topk_rows(sc[t:t + 1, :n], np.array([n], np.int32), K)[0]
        assert np.array_equal(idx[t], own), f"row {t}: selection differs from Top-K of the kernel's scores"
        near += check_index_sets(idx[t], ref_idx[t], ref_sc[t], n, K)
    return near


def test_mxfp8_decode_ragged_paged(orc):
    lens = [1, 63, 64, 65, 129, 1000, 2047, 2048, 2049, 5000]
    wl = make_workload("ragged", lens, [1] * len(lens), H=16, K=256, page_size=64, seed=11, with_kv=False)
    _check(orc, wl, 256)


@pytest.mark.parametrize("C", [1, 2, 8, 16])
def test_mxfp8_cluster_sizes(orc, C):
    import indexer_top_sparse_gb300 as d
    wl = make_workload("c", [3000, 700, 64], [1, 1, 1], H=16, K=512, page_size=128, seed=20 + C, with_kv=False)
    d.set_tuning("indexer_cluster", C)
    try:
        _check(orc, wl, 512)
    finally:
        d.set_tuning("indexer_cluster", 0)


@pytest.mark.parametrize("stages", [2, 4, 5])
def test_mxfp8_ring_depths(orc, stages):
    # (5 runs as 4: the ring depth is even, two threads issue alternate tiles)
    import indexer_top_sparse_gb300 as d
    wl = make_workload("s", [4100, 333], [1, 1], H=16, K=256, page_size=64, seed=30 + stages, with_kv=False)
    d.set_tuning("indexer_stages", stages)
    try:
        _check(orc, wl, 256)
    finally:
        d.set_tuning("indexer_stages", 0)


@pytest.mark.parametrize("G", [1, 2, 3])
def test_mxfp8_prefill_causal(orc, G):
    # G query rows of a sequence per cluster share each key tile (their
    # queries stacked in the MMA's N: 192 with three rows, whose query scales
    # fill six TMEM columns); 17 rows leave a last group of one (G = 2) or two
    # (G = 3)
    import indexer_top_sparse_gb300 as d
    from _util import tuning
    wl = make_workload("p", [700, 300, 2100], [40, 17, 9], H=16, K=256, page_size=64, seed=41, with_kv=False)
    with tuning(indexer_group=G):
        _check(orc, wl, 256)


def test_mxfp8_scales_required():
    import indexer_top_sparse_gb300 as d
    wl = make_workload("r", [128], [1], H=16, K=64, page_size=64, seed=5, with_kv=False)
    q = torch.zeros((1, 64, 128), dtype=torch.uint8, device="cuda")
    k = torch.zeros((wl.page_table.max() + 1, 64, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(TypeError):
        d.dsa_index_topk(q, dev(wl.head_w), k, dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q), 64,
                         dtype="mxfp8")


@pytest.mark.parametrize("lens,nq", [([1, 63, 1000, 2049, 40000], [1, 1, 1, 1, 1]), ([700, 300], [40, 17])])
def test_mxfp8_query_quantised_in_the_kernel(orc, lens, nq):
    # dtype "mxfp8_qbf16": q_idx goes in as bf16 and the fused indexer
    # quantises it itself.  Its codes and scales are the standalone
    # quantiser's, so scores and indices equal those of the pre-quantised
    # call bit for bit; they are also checked against the oracle.
    import indexer_top_sparse_gb300 as d
    from _util import dev_bf16
    wl = make_workload("qq", lens, nq, H=16, K=512, page_size=64, seed=51, with_kv=False)
    q, qs, k, ks = _quantised(orc, wl)
    idx_ref, sc_ref = _run(wl, q, qs, k, ks, 512)
    ld = int(wl.seq_lens.max())
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device="cuda")
    ws = d.Workspace(256)
    args = (dev_bf16(wl.q_idx), dev(wl.head_w), dev(k), dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q), 512)
    idx, sc = d.dsa_index_scores(*args, scores, k_idx_scale=dev(ks), dtype="mxfp8_qbf16", workspace=ws)
    ws.check()
    idx2 = d.dsa_index_topk(*args, k_idx_scale=dev(ks), dtype="mxfp8_qbf16", workspace=ws)
    ws.check()
    idx, idx2, sc = idx.cpu().numpy(), idx2.cpu().numpy(), sc.cpu().numpy()
    assert np.array_equal(idx, idx_ref) and np.array_equal(idx2, idx_ref)
    fin = ~np.isnan(sc_ref)
    assert np.array_equal(sc[fin].view(np.uint32), sc_ref[fin].view(np.uint32))
    _check(orc, wl, 512)
