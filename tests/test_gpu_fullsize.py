"""Full-size parity: each workload of the measurement table runs through the
C-ABI exactly as the benchmark launches it (default tuning, whole batch in
one call), and sampled query rows are checked against the oracle row by row.
Index sets must agree except at near-threshold positions (1e-3 relative of
the K-th oracle score); attention, fed the GPU's own indices, must match the
oracle within 2e-2 / 1e-2 (bf16) or 6e-2 / 3e-2 (FP8).  FP8 caches (one scale
per row, or per 128-dim tile) are made by each side's own quantiser from the
same bf16 draws (the two quantisers agree bit for bit, see test_gpu_quant.py)."""
import numpy as np
import pytest
import torch

from _util import check_index_sets, dev, dev_bf16
from indexer_top_sparse_gb300.inputs import decode_b32_n32k, decode_b64_mixed, make_workload, prefill

pytestmark = pytest.mark.gpu


def _gpu_path(wl, fp8=False, kv_fmt="fp8_rowscale"):
    """The production calls on the whole batch; returns indices and out."""
    import indexer_top_sparse_gb300 as d
    pt, sl, cq = dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q)
    ws = d.Workspace(max(d.index_topk_workspace_size(wl.B, wl.T, wl.K, wl.max_pages, wl.page_size),
                         d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)))
    if fp8:
        q_idx, q_sc = d.dsa_quant_mxfp8(dev_bf16(wl.q_idx))
        k_idx, k_sc = d.dsa_quant_mxfp8(dev_bf16(wl.k_idx))
        idx = d.dsa_index_topk(q_idx, dev(wl.head_w), k_idx, pt, sl, cq, wl.K, workspace=ws,
                               q_idx_scale=q_sc, k_idx_scale=k_sc, dtype="mxfp8")
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


def _sequence_view(wl, t):
    """The oracle's inputs for query row t alone: its sequence's pages copied
    into a compact cache with an identity page table (data movement only)."""
    b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
    n_pages = (int(wl.seq_lens[b]) + wl.page_size - 1) // wl.page_size
    pages = wl.page_table[b, :n_pages]
    nq = int(wl.cu_q[b + 1] - wl.cu_q[b])
    view = {"k_idx": wl.k_idx[pages], "kv": wl.kv[pages], "pt": np.arange(n_pages, dtype=np.int32)[None, :],
            "sl": wl.seq_lens[b:b + 1].copy(), "cq": np.array([0, nq], np.int32),
            "rows": slice(int(wl.cu_q[b]), int(wl.cu_q[b + 1])), "r": t - int(wl.cu_q[b])}
    return view


def _check_rows(orc, wl, rows, idx, out, fp8=False, kv_fmt="fp8_rowscale"):
    pos = wl.query_pos()
    atol, rtol = (6e-2, 3e-2) if fp8 else (2e-2, 1e-2)
    near = 0
    for t in rows:
        v = _sequence_view(wl, t)
        r = np.array([v["r"]], np.int32)
        q_idx, q = wl.q_idx[v["rows"]], wl.q[v["rows"]]
        g_idx = idx[v["rows"]]
        if fp8:
            q8, qs = orc.quant_mxfp8(q_idx)
            k8, ks = orc.quant_mxfp8(v["k_idx"])
            ref_idx, ref_sc = orc.index_topk(q8, wl.head_w[v["rows"]], k8, v["pt"], v["sl"], v["cq"], wl.K,
                                             wl.page_size, dtype=orc.IDX_MXFP8, q_scale=qs, k_scale=ks, rows=r,
                                             want_scores=True)
            tiles = kv_fmt == "fp8_tile128"
            nope, rope, rsc = (orc.quant_fp8_tiles if tiles else orc.quant_fp8_rows)(v["kv"])
            ref_out, _ = orc.sparse_mla(q, nope, v["pt"], v["cq"], g_idx, wl.scale, wl.page_size,
                                        dtype=orc.KV_FP8_TILE128 if tiles else orc.KV_FP8_ROWSCALE,
                                        kv_rope=rope, kv_scale=rsc, rows=r)
        else:
            ref_idx, ref_sc = orc.index_topk(q_idx, wl.head_w[v["rows"]], v["k_idx"], v["pt"], v["sl"], v["cq"],
                                             wl.K, wl.page_size, rows=r, want_scores=True)
            ref_out, _ = orc.sparse_mla(q, v["kv"], v["pt"], v["cq"], g_idx, wl.scale, wl.page_size, rows=r)
        near += check_index_sets(idx[t], ref_idx[0], ref_sc[0], int(pos[t]) + 1, wl.K)
        np.testing.assert_allclose(out[t], ref_out[0], atol=atol, rtol=rtol, err_msg=f"query row {t}")
    return near


def test_decode_b32_n32768_bf16(orc):
    wl = decode_b32_n32k(0)
    idx, out = _gpu_path(wl)
    _check_rows(orc, wl, [0, 13, 31], idx, out)


@pytest.mark.parametrize("kv_fmt", ["fp8_rowscale", "fp8_tile128"])
def test_decode_b64_mixed_lengths_fp8(orc, kv_fmt):
    wl = decode_b64_mixed(0)
    idx, out = _gpu_path(wl, fp8=True, kv_fmt=kv_fmt)
    lens = wl.seq_lens
    rows = [int(np.argmin(lens)), int(np.argmax(lens)), 37]
    _check_rows(orc, wl, rows, idx, out, fp8=True, kv_fmt=kv_fmt)


def test_prefill_16k_bf16(orc):
    wl = prefill(16384, seed=0)
    idx, out = _gpu_path(wl)
    _check_rows(orc, wl, [0, 1, 2047, 2048, 9001, 16383], idx, out)


def test_prefill_131k_last_chunk_fp8(orc):
    # the last 4096-token chunk of a 131072-token sequence: its queries are the
    # last positions, every history position is cached
    wl = make_workload("prefill_131072_chunk31_fp8", [131072], [4096], H=128, K=2048, page_size=64,
                       permute=True, seed=3)
    idx, out = _gpu_path(wl, fp8=True)
    _check_rows(orc, wl, [0, 2048, 4095], idx, out, fp8=True)


def _max_excess(a, b, atol, rtol, rows=1024):
    """max over all elements of |a - b| - (atol + rtol |b|), on the GPU in
    row blocks (positive: out of tolerance somewhere)."""
    worst = -float("inf")
    for r0 in range(0, a.shape[0], rows):
        x, y = a[r0:r0 + rows].float(), b[r0:r0 + rows].float()
        worst = max(worst, ((x - y).abs() - (atol + rtol * y.abs())).max().item())
    return worst


def test_prefill_16k_every_row_on_every_kernel_form():
    # Every query row of the 16k prefill (rows with a handful of valid keys,
    # ragged last tiles, full 2048-key rows) on each 128-head kernel form: the
    # dims-split pair, the 64-head pair (which forwards gathered rows to its
    # peer) and independent 64-head CTAs; FP8 rows on the 64-head pair and
    # independent CTAs.  Each form is within the attention tolerance of the
    # oracle (sampled rows above), so any two agree within twice that.
    import indexer_top_sparse_gb300 as d
    from _util import tuning
    wl = prefill(16384, seed=0)
    pt, sl, cq = dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q)
    ws = d.Workspace(max(d.index_topk_workspace_size(wl.B, wl.T, wl.K, wl.max_pages, wl.page_size),
                         d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)))
    idx = d.dsa_index_topk(dev_bf16(wl.q_idx), dev(wl.head_w), dev_bf16(wl.k_idx), pt, sl, cq, wl.K, workspace=ws)
    q, kv = dev_bf16(wl.q), dev_bf16(wl.kv)
    outs = {}
    for name, knobs in (("dsplit", dict(mla_dsplit=1)), ("pair64", dict(mla_dsplit=-1, mla_pair=1)),
                        ("indep64", dict(mla_dsplit=-1, mla_pair=-1))):
        with tuning(**knobs):
            outs[name] = d.dsa_sparse_mla(q, kv, pt, sl, cq, idx, wl.scale, workspace=ws)
        ws.check()
    for other in ("pair64", "indep64"):
        assert _max_excess(outs[other], outs["dsplit"], 4e-2, 2e-2) <= 0, other
    del outs
    nope, rope, rsc = d.dsa_quant_fp8_rows(kv)
    f8 = {}
    for name, pair in (("pair64", 1), ("indep64", -1)):
        with tuning(mla_pair=pair):
            f8[name] = d.dsa_sparse_mla(q, nope, pt, sl, cq, idx, wl.scale, workspace=ws, kv_rope=rope, kv_scale=rsc,
                                        dtype="fp8_rowscale")
        ws.check()
    assert _max_excess(f8["pair64"], f8["indep64"], 4e-2, 2e-2) <= 0
