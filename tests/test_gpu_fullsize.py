"""Full-size parity: each workload of the measurement table runs through the
C-ABI exactly as the benchmark launches it (default tuning, whole batch in
one call), and query rows are checked against the oracle row by row: every
row of the 32 x 32768 decode, 128 seeded rows of the 16k prefill (short rows,
rows around the 2048-key boundary, ragged tiles, the last rows), the first, a
middle and the last 4096-token chunk of the 131072-token FP8 prefill, and the
one-sequence 2048-position decode on its single 2048-row page.  Index sets
must agree except at near-threshold positions (1e-3 relative of the K-th
oracle score); attention, fed the GPU's own indices, must match the oracle
within 2e-2 / 1e-2 (bf16) or 6e-2 / 3e-2 (FP8).  FP8 caches (one scale per
row, or per 128-dim tile) are made by each side's own quantiser from the same
bf16 draws (the two quantisers agree bit for bit, see test_gpu_quant.py).

Every row of the 16k prefill is also checked against the oracle on each
128-head kernel form, two heads per row (one from each 64-head half, a
different pair on every row), so that a fault confined to some rows or to one
half of the heads cannot hide between sampled rows.

The oracle is single-threaded C; independent rows run on a thread pool (its
calls release the interpreter lock), which changes nothing in its
arithmetic."""
import concurrent.futures as cf
import os

import numpy as np
import pytest

from _util import check_index_sets, dev, dev_bf16, tuning
from indexer_top_sparse_gb300.inputs import decode_b32_n32k, decode_b64_mixed, decode_small, make_workload, prefill

pytestmark = pytest.mark.gpu

_WORKERS = max(1, min(16, os.cpu_count() or 1))


def _pmap(fn, items):
    with cf.ThreadPoolExecutor(max_workers=_WORKERS) as ex:
        return list(ex.map(fn, items))


def _gpu_path(wl, fp8=False, kv_fmt="fp8_rowscale"):
    """The production calls on the whole batch; returns indices and out."""
    import indexer_top_sparse_gb300 as d
    pt, sl, cq = dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q)
    ws = d.Workspace(max(d.index_topk_workspace_size(wl.B, wl.T, wl.K, wl.max_pages, wl.page_size),
                         d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)))
    if fp8:
        # MXFP8 index keys; the bf16 index query is quantised inside the indexer
        k_idx, k_sc = d.dsa_quant_mxfp8(dev_bf16(wl.k_idx))
        idx = d.dsa_index_topk(dev_bf16(wl.q_idx), dev(wl.head_w), k_idx, pt, sl, cq, wl.K, workspace=ws,
                               k_idx_scale=k_sc, dtype="mxfp8_qbf16")
        del k_idx, k_sc
        quant = d.dsa_quant_fp8_tiles if kv_fmt == "fp8_tile128" else d.dsa_quant_fp8_rows
        nope, rope, rsc = quant(dev_bf16(wl.kv))
        out = d.dsa_sparse_mla(dev_bf16(wl.q), nope, pt, sl, cq, idx, wl.scale, workspace=ws, kv_rope=rope,
                               kv_scale=rsc, dtype=kv_fmt)
    else:
        idx = d.dsa_index_topk(dev_bf16(wl.q_idx), dev(wl.head_w), dev_bf16(wl.k_idx), pt, sl, cq, wl.K,
                               workspace=ws)
        out = d.dsa_sparse_mla(dev_bf16(wl.q), dev_bf16(wl.kv), pt, sl, cq, idx, wl.scale, workspace=ws)
    ws.check()
    return idx.cpu().numpy(), out.float().cpu().numpy()


def _sequence_view(orc, wl, b, fp8, kv_fmt):
    """The oracle's inputs for the query rows of sequence b: its pages copied
    into a compact cache with an identity page table (data movement only),
    quantised by the oracle's own quantisers for the FP8 formats."""
    n_pages = (int(wl.seq_lens[b]) + wl.page_size - 1) // wl.page_size
    pages = wl.page_table[b, :n_pages]
    nq = int(wl.cu_q[b + 1] - wl.cu_q[b])
    view = {"k_idx": wl.k_idx[pages], "kv": wl.kv[pages], "pt": np.arange(n_pages, dtype=np.int32)[None, :],
            "sl": wl.seq_lens[b:b + 1].copy(), "cq": np.array([0, nq], np.int32),
            "rows": slice(int(wl.cu_q[b]), int(wl.cu_q[b + 1]))}
    if fp8:
        view["k8"] = orc.quant_mxfp8(view["k_idx"])
        tiles = kv_fmt == "fp8_tile128"
        view["kv8"] = (orc.quant_fp8_tiles if tiles else orc.quant_fp8_rows)(view["kv"])
        view["kvdt"] = orc.KV_FP8_TILE128 if tiles else orc.KV_FP8_ROWSCALE
    return view


def _oracle_row(orc, wl, v, t, g_idx_rows, fp8):
    """Oracle indices, scores and attention output of query row t of the
    sequence whose view is v (attention fed the GPU's indices)."""
    r = np.array([t - v["rows"].start], np.int32)
    q_idx, q = wl.q_idx[v["rows"]], wl.q[v["rows"]]
    g_idx = g_idx_rows[v["rows"]]
    if fp8:
        q8, qs = orc.quant_mxfp8(q_idx[r[0]:r[0] + 1])
        k8, ks = v["k8"]
        cq1 = np.array([0, 1], np.int32)
        sl1 = np.array([int(v["sl"][0]) - (int(v["cq"][1]) - 1 - int(r[0]))], np.int32)
        ref_idx, ref_sc = orc.index_topk(q8, wl.head_w[v["rows"]][r[0]:r[0] + 1], k8, v["pt"], sl1, cq1, wl.K,
                                         wl.page_size, dtype=orc.IDX_MXFP8, q_scale=qs, k_scale=ks,
                                         want_scores=True, ld_scores=int(v["sl"][0]))
        nope, rope, rsc = v["kv8"]
        ref_out, _ = orc.sparse_mla(q, nope, v["pt"], v["cq"], g_idx, wl.scale, wl.page_size, dtype=v["kvdt"],
                                    kv_rope=rope, kv_scale=rsc, rows=r)
    else:
        ref_idx, ref_sc = orc.index_topk(q_idx, wl.head_w[v["rows"]], v["k_idx"], v["pt"], v["sl"], v["cq"],
                                         wl.K, wl.page_size, rows=r, want_scores=True)
        ref_out, _ = orc.sparse_mla(q, v["kv"], v["pt"], v["cq"], g_idx, wl.scale, wl.page_size, rows=r)
    return ref_idx[0], ref_sc[0], ref_out[0]


def _check_rows(orc, wl, rows, idx, out, fp8=False, kv_fmt="fp8_rowscale"):
    pos = wl.query_pos()
    atol, rtol = (6e-2, 3e-2) if fp8 else (2e-2, 1e-2)
    seq = {int(t): int(np.searchsorted(wl.cu_q, t, side="right") - 1) for t in rows}
    views = dict(zip(sorted(set(seq.values())),
                     _pmap(lambda b: _sequence_view(orc, wl, b, fp8, kv_fmt), sorted(set(seq.values())))))
    refs = _pmap(lambda t: _oracle_row(orc, wl, views[seq[int(t)]], int(t), idx, fp8), list(rows))
    near = 0
    for t, (ref_idx, ref_sc, ref_out) in zip(rows, refs):
        near += check_index_sets(idx[t], ref_idx, ref_sc, int(pos[t]) + 1, wl.K)
        np.testing.assert_allclose(out[t], ref_out, atol=atol, rtol=rtol, err_msg=f"query row {t}")
    return near


def test_decode_b1_n2048_contiguous_bf16(orc):
    # one sequence of 2048 positions on a single 2048-row page, K = 256, 16 MLA heads
    wl = decode_small(0)
    assert wl.page_size == 2048 and wl.page_table.shape == (1, 1)
    idx, out = _gpu_path(wl)
    _check_rows(orc, wl, [0], idx, out)


def test_decode_b32_n32768_bf16_every_row(orc):
    wl = decode_b32_n32k(0)
    idx, out = _gpu_path(wl)
    _check_rows(orc, wl, list(range(wl.T)), idx, out)


@pytest.mark.parametrize("kv_fmt", ["fp8_rowscale", "fp8_tile128"])
def test_decode_b64_mixed_lengths_fp8(orc, kv_fmt):
    wl = decode_b64_mixed(0)
    idx, out = _gpu_path(wl, fp8=True, kv_fmt=kv_fmt)
    lens = wl.seq_lens
    order = np.argsort(lens)
    rows = sorted({int(order[0]), int(order[1]), int(order[-1]), int(order[-2]), 37, 0, 63})
    _check_rows(orc, wl, rows, idx, out, fp8=True, kv_fmt=kv_fmt)


def _prefill_rows(T, n=128, seed=11):
    """Seeded rows of a causal prefill covering every class: rows with a
    handful of valid keys, rows at 64-key tile edges, rows around the
    2048-key boundary, a ragged last tile, and the last rows."""
    fixed = [0, 1, 2, 7, 31, 62, 63, 64, 65, 127, 128, 1000, 2045, 2046, 2047, 2048, 2049, 2111, 2112, 4095, 4096,
             8191, 8192, 8256, T - 4, T - 3, T - 2, T - 1]
    fixed = sorted({t for t in fixed if 0 <= t < T})
    rng = np.random.default_rng(seed)
    rest = rng.choice(np.setdiff1d(np.arange(T), fixed), max(0, n - len(fixed)), replace=False)
    return sorted(fixed + [int(t) for t in rest])


def test_prefill_16k_bf16(orc):
    wl = prefill(16384, seed=0)
    idx, out = _gpu_path(wl)
    rows = _prefill_rows(wl.T)
    assert len(rows) >= 128
    _check_rows(orc, wl, rows, idx, out)


@pytest.mark.parametrize("chunk", [0, 15, 31])
def test_prefill_131k_chunks_fp8(orc, chunk):
    # chunk c of a 131072-token sequence prefilled 4096 tokens at a time: its
    # queries are the last 4096 of 4096 (c + 1) cached positions (permuted pages)
    n = 4096 * (chunk + 1)
    wl = make_workload(f"prefill_131072_chunk{chunk}_fp8", [n], [4096], H=128, K=2048, page_size=64, permute=True,
                       seed=3 + chunk)
    idx, out = _gpu_path(wl, fp8=True)
    _check_rows(orc, wl, [0, 1, 2047, 2048, 4095], idx, out, fp8=True)


def _heads_per_row(T, H):
    """Two heads for every row: one in each 64-head half, a different pair on
    each row (all heads of a half appear every 64 rows)."""
    h = np.empty((T, 2), np.int64)
    t = np.arange(T)
    h[:, 0] = t % (H // 2)
    h[:, 1] = H // 2 + (t * 37 + 11) % (H // 2)
    return h


def _oracle_two_heads(orc, wl, idx, heads, fp8_cache=None):
    """Oracle attention of every row for its two heads (q restricted to them),
    rows split over the thread pool."""
    q2 = np.ascontiguousarray(np.take_along_axis(wl.q, heads[:, :, None], axis=1))
    chunks = np.array_split(np.arange(wl.T, dtype=np.int32), 4 * _WORKERS)

    def run(rows):
        if fp8_cache is None:
            o, _ = orc.sparse_mla(q2, wl.kv, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size, rows=rows)
        else:
            nope, rope, rsc = fp8_cache
            o, _ = orc.sparse_mla(q2, nope, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size,
                                  dtype=orc.KV_FP8_ROWSCALE, kv_rope=rope, kv_scale=rsc, rows=rows)
        return o

    return np.concatenate(_pmap(run, chunks))


def test_prefill_16k_every_row_every_kernel_form(orc):
    # Every query row of the 16k prefill (rows with a handful of valid keys,
    # ragged last tiles, full 2048-key rows) on each 128-head kernel form --
    # the dims-split pair, the 64-head pair (which forwards gathered rows to
    # its peer) and independent 64-head CTAs; FP8 rows on the 64-head pair and
    # independent CTAs -- against the oracle fed the same indices.
    import indexer_top_sparse_gb300 as d
    wl = prefill(16384, seed=0)
    pt, sl, cq = dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q)
    ws = d.Workspace(max(d.index_topk_workspace_size(wl.B, wl.T, wl.K, wl.max_pages, wl.page_size),
                         d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)))
    idx_d = d.dsa_index_topk(dev_bf16(wl.q_idx), dev(wl.head_w), dev_bf16(wl.k_idx), pt, sl, cq, wl.K, workspace=ws)
    idx = idx_d.cpu().numpy()
    heads = _heads_per_row(wl.T, wl.H)
    hsel = dev(heads)
    q, kv = dev_bf16(wl.q), dev_bf16(wl.kv)
    ref = _oracle_two_heads(orc, wl, idx, heads)
    rows = np.arange(wl.T)[:, None]
    for name, knobs in (("dsplit", dict(mla_dsplit=1)), ("pair64", dict(mla_dsplit=-1, mla_pair=1)),
                        ("indep64", dict(mla_dsplit=-1, mla_pair=-1))):
        with tuning(**knobs):
            out = d.dsa_sparse_mla(q, kv, pt, sl, cq, idx_d, wl.scale, workspace=ws)
        ws.check()
        got = out[dev(rows), hsel].float().cpu().numpy()
        np.testing.assert_allclose(got, ref, atol=2e-2, rtol=1e-2, err_msg=name)
        del out
    nope, rope, rsc = d.dsa_quant_fp8_rows(kv)
    ref8 = _oracle_two_heads(orc, wl, idx, heads, fp8_cache=orc.quant_fp8_rows(wl.kv))
    for name, pair in (("pair64", 1), ("indep64", -1)):
        with tuning(mla_pair=pair):
            out = d.dsa_sparse_mla(q, nope, pt, sl, cq, idx_d, wl.scale, workspace=ws, kv_rope=rope, kv_scale=rsc,
                                   dtype="fp8_rowscale")
        ws.check()
        got = out[dev(rows), hsel].float().cpu().numpy()
        np.testing.assert_allclose(got, ref8, atol=6e-2, rtol=3e-2, err_msg=f"fp8 {name}")
        del out
