"""Device-detected input errors on the attention kernels.

A selected index outside 0..pos(t), a page-table entry outside
[0, num_pages), and a sequence longer than its page-table row
(seq_lens[b] > max_pages_per_seq * page_size, so that a valid index would need
a page-table entry past the row) are reported through the workspace error
word (DSA_ERR_BAD_INDEX / DSA_ERR_BAD_PAGE from dsa_get_error) and the access
is skipped.  Each kernel form is covered: 64-head CTAs on the split grid,
the 64-head pair that shares gathered rows, stream-K, the 128-head dims-split CTA pair, and the FP8 cache.  After each
error the same call on valid inputs is correct again (the GPU and the
context are unaffected), checked against the oracle.  The inputs are made on
the host; no kernel is made to fault."""
import numpy as np
import pytest
import torch

from _util import dev, to_device, tuning
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu

BAD_PAGE, BAD_INDEX = 4, 5
FORMS = {"split64": dict(mla_dsplit=-1, mla_stream_k=-1, mla_splits=2),
         "pair64": dict(mla_dsplit=-1, mla_stream_k=-1, mla_pair=1, mla_splits=2),
         "stream_k": dict(mla_dsplit=-1, mla_stream_k=1),
         "dsplit": dict(mla_dsplit=1, mla_splits=2),
         "fp8": dict(mla_stream_k=-1, mla_splits=2)}


def _indices(rng, wl):
    pos = wl.query_pos()
    idx = np.full((wl.T, wl.K), -1, np.int32)
    for t in range(wl.T):
        n = int(pos[t]) + 1
        m = min(wl.K, n)
        idx[t, :m] = np.sort(rng.choice(n, m, replace=False))
    return idx


def _setup(form):
    # 12 decode rows of 1010..3000 positions, K = 1000, 128 heads: a shape on
    # which stream-K applies when forced (every CTA gets 2+ key tiles)
    rng = np.random.default_rng(41)
    lens = rng.integers(1010, 3000, size=12)
    wl = make_workload(f"err_{form}", lens, [1] * 12, H=128, K=1000, page_size=64, seed=41, with_idx=False)
    return wl, _indices(rng, wl)


def _call(d, wl, t, idx_d, pt, sl, form, ws, cache):
    kw = {}
    kv = t["kv"]
    if form == "fp8":
        kv = cache[0]
        kw = dict(kv_rope=cache[1], kv_scale=cache[2], dtype="fp8_rowscale")
    with tuning(**FORMS[form]):
        return d.dsa_sparse_mla(t["q"], kv, pt, sl, t["cu_q"], idx_d, wl.scale, workspace=ws, **kw)


def _ws(d, wl):
    with tuning(mla_stream_k=1):
        n = d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)
    return d.Workspace(max(n, d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)))


def _expect(d, ws, code):
    with pytest.raises(d.DSAError) as e:
        ws.check()
    assert e.value.code == code
    ws.check()  # the error word was cleared


def _good_call_matches_oracle(orc, d, wl, t, idx, ws, form, cache):
    out = _call(d, wl, t, dev(idx), t["page_table"], t["seq_lens"], form, ws, cache)
    ws.check()
    if form == "fp8":
        rn, rr, rs = orc.quant_fp8_rows(wl.kv)
        want, _ = orc.sparse_mla(wl.q, rn, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size,
                                 dtype=orc.KV_FP8_ROWSCALE, kv_rope=rr, kv_scale=rs)
    else:
        want, _ = orc.sparse_mla(wl.q, wl.kv, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size)
    np.testing.assert_allclose(out.float().cpu().numpy(), want, atol=2e-2, rtol=1e-2)


def _fp8_cache(d, t, form):
    return d.dsa_quant_fp8_rows(t["kv"]) if form == "fp8" else None


@pytest.mark.parametrize("form", list(FORMS))
def test_index_beyond_the_causal_bound_is_reported(orc, form):
    import indexer_top_sparse_gb300 as d
    wl, idx = _setup(form)
    t = to_device(wl)
    cache = _fp8_cache(d, t, form)
    ws = _ws(d, wl)
    bad = idx.copy()
    pos = wl.query_pos()
    bad[1, 3] = int(pos[1]) + 1          # one past the query's own position
    bad[2, 500] = int(pos[2]) + 4000     # far past the sequence
    _call(d, wl, t, dev(bad), t["page_table"], t["seq_lens"], form, ws, cache)
    _expect(d, ws, BAD_INDEX)
    _good_call_matches_oracle(orc, d, wl, t, idx, ws, form, cache)


@pytest.mark.parametrize("form", list(FORMS))
def test_page_id_out_of_range_is_reported(orc, form):
    import indexer_top_sparse_gb300 as d
    wl, idx = _setup(form)
    t = to_device(wl)
    cache = _fp8_cache(d, t, form)
    ws = _ws(d, wl)
    pt = t["page_table"].clone()
    page = int(idx[0, 7]) // wl.page_size    # a page that row 0 selects
    pt[0, page] = wl.num_pages + 3
    pt[2, int(idx[2, 100]) // wl.page_size] = -5
    _call(d, wl, t, dev(idx), pt, t["seq_lens"], form, ws, cache)
    _expect(d, ws, BAD_PAGE)
    _good_call_matches_oracle(orc, d, wl, t, idx, ws, form, cache)


@pytest.mark.parametrize("form", list(FORMS))
def test_sequence_longer_than_its_page_row_is_reported(orc, form):
    # seq_lens of sequence 1 claims more positions than its page-table row
    # maps; an index past the row must not read the next row (or past the
    # table) but is reported as a bad page
    import indexer_top_sparse_gb300 as d
    wl, idx = _setup(form)
    t = to_device(wl)
    cache = _fp8_cache(d, t, form)
    ws = _ws(d, wl)
    max_len = wl.max_pages * wl.page_size
    sl = t["seq_lens"].clone()
    sl[1] = max_len + 200
    bad = idx.copy()
    bad[1, 0] = max_len + 150            # causal for the claimed length, past the page row
    _call(d, wl, t, dev(bad), t["page_table"], sl, form, ws, cache)
    _expect(d, ws, BAD_PAGE)
    _good_call_matches_oracle(orc, d, wl, t, idx, ws, form, cache)


def test_cache_append_past_the_page_row_is_reported():
    import indexer_top_sparse_gb300 as d
    wl = make_workload("err_append", [300, 200], [2, 1], H=16, K=64, page_size=64, seed=43)
    t = to_device(wl)
    ws = d.Workspace(256)
    sl = t["seq_lens"].clone()
    sl[1] = wl.max_pages * wl.page_size + 64     # its new token would sit past its page row
    k_cache, kv_cache = t["k_idx"].clone(), t["kv"].clone()
    k_new = torch.zeros((3, 128), dtype=torch.bfloat16, device="cuda")
    kv_new = torch.zeros((3, 576), dtype=torch.bfloat16, device="cuda")
    d.dsa_cache_append(t["page_table"], sl, t["cu_q"], k_new=k_new, kv_new=kv_new, k_cache=k_cache,
                       kv_cache=kv_cache, workspace=ws)
    _expect(d, ws, BAD_PAGE)
    # sequence 0's two tokens were written, nothing else changed
    rows = [int(wl.page_table[0, p // 64]) * 64 + p % 64 for p in (298, 299)]
    kc = k_cache.view(-1, 128)
    assert torch.count_nonzero(kc[rows].float()) == 0
    keep = torch.ones(kc.shape[0], dtype=torch.bool, device="cuda")
    keep[rows] = False
    assert torch.equal(kc[keep], t["k_idx"].view(-1, 128)[keep])
