"""GPU sparse MLA against the oracle on the same indices: outputs within
2e-2 absolute / 1e-2 relative (bf16 path), lse within 1e-3; covers 16, 64 and
128 heads, -1 padding, a single selected key, rows with no valid key, every
split count, and the paged gather.  128-head bf16 cases run on both kernels:
the CTA pair that splits the latent dims (KERNELS "dsplit", the automatic
choice) and two 64-head CTAs per query ("heads64")."""
import math

import numpy as np
import pytest
import torch

from _util import dev, dev_bf16, to_device, tuning
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2
# value of the "mla_dsplit" knob for each 128-head bf16 kernel
KERNELS = {"dsplit": 1, "heads64": -1}


def _random_indices(rng, wl, K, pad_frac=0.0):
    pos = wl.query_pos()
    idx = np.full((wl.T, K), -1, np.int32)
    for t in range(wl.T):
        n = int(pos[t]) + 1
        m = min(K, n)
        sel = np.sort(rng.choice(n, m, replace=False)).astype(np.int32)
        if pad_frac:
            sel[rng.random(m) < pad_frac] = -1
        idx[t, :m] = sel
    return idx


def _run(wl, idx, want_lse=True):
    import indexer_top_sparse_gb300 as d
    t = to_device(wl)
    lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda") if want_lse else None
    ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, idx.shape[1]))
    out = d.dsa_sparse_mla(t["q"], t["kv"], t["page_table"], t["seq_lens"], t["cu_q"], dev(idx), wl.scale, lse=lse,
                           workspace=ws)
    ws.check()
    return out.float().cpu().numpy(), (lse.cpu().numpy() if want_lse else None)


def _compare(orc, wl, idx, rows=None):
    out, lse = _run(wl, idx)
    rows = np.arange(wl.T, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    ref, ref_lse = orc.sparse_mla(wl.q, wl.kv, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size, rows=rows)
    np.testing.assert_allclose(out[rows], ref, atol=ATOL, rtol=RTOL)
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[rows][fin], ref_lse[fin], rtol=1e-3, atol=1e-3)
    assert np.all(np.isneginf(lse[rows][~fin]))


@pytest.mark.parametrize("H,kernel", [(16, "heads64"), (64, "heads64"), (128, "dsplit"), (128, "heads64")])
def test_decode_heads(orc, H, kernel):
    rng = np.random.default_rng(H)
    wl = make_workload("mla", [3000, 513, 70], [1, 1, 1], H=H, K=512, page_size=64, seed=H, with_idx=False)
    with tuning(mla_dsplit=KERNELS[kernel]):
        _compare(orc, wl, _random_indices(rng, wl, 512))


@pytest.mark.parametrize("H,kernel", [(64, "heads64"), (128, "dsplit"), (128, "heads64")])
@pytest.mark.parametrize("splits", [1, 2, 3, 8])
def test_every_split_count(orc, splits, H, kernel):
    rng = np.random.default_rng(100 + splits)
    wl = make_workload("mla", [4000, 900], [1, 1], H=H, K=1000, page_size=64, seed=splits, with_idx=False)
    idx = _random_indices(rng, wl, 1000, pad_frac=0.1)
    with tuning(mla_splits=splits, mla_dsplit=KERNELS[kernel]):
        _compare(orc, wl, idx)


def test_padding_single_key_and_empty_rows(orc):
    wl = make_workload("mla", [300, 300, 300, 50], [1, 1, 1, 1], H=16, K=64, page_size=32, seed=5, with_idx=False)
    idx = np.full((4, 64), -1, np.int32)
    idx[0, :40] = np.arange(0, 400, 10)[:40] % 300
    idx[0] = np.where(np.arange(64) % 3 == 0, -1, idx[0])
    idx[1, 17] = 123                      # a single selected key
    # row 2: no valid key
    idx[3, :50] = np.arange(50)           # every position of a short sequence
    _compare(orc, wl, idx)
    out, lse = _run(wl, idx)
    v = wl.kv.reshape(-1, 576)[wl.page_table[1][123 // 32] * 32 + 123 % 32, :512]
    from indexer_top_sparse_gb300.inputs import bf16_to_f32
    np.testing.assert_allclose(out[1], np.broadcast_to(bf16_to_f32(v), (16, 512)), atol=1e-2, rtol=1e-2)
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))


def test_dsplit_padding_single_key_empty_rows_and_ragged_tiles(orc):
    # 128 heads on the dims-split pair: a row with -1 padding and a ragged last
    # tile (K = 100), a single selected key, a row with no valid key, and a
    # short sequence selected in full; one and two key splits
    wl = make_workload("mla", [300, 300, 300, 50], [1, 1, 1, 1], H=128, K=100, page_size=32, seed=6, with_idx=False)
    idx = np.full((4, 100), -1, np.int32)
    idx[0, :90] = np.arange(0, 900, 10)[:90] % 300
    idx[0] = np.where(np.arange(100) % 3 == 0, -1, idx[0])
    idx[1, 77] = 123
    idx[3, :50] = np.arange(50)
    for splits in (1, 2):
        with tuning(mla_splits=splits, mla_dsplit=1):
            _compare(orc, wl, idx)
            out, lse = _run(wl, idx)
        v = wl.kv.reshape(-1, 576)[wl.page_table[1][123 // 32] * 32 + 123 % 32, :512]
        from indexer_top_sparse_gb300.inputs import bf16_to_f32
        np.testing.assert_allclose(out[1], np.broadcast_to(bf16_to_f32(v), (128, 512)), atol=1e-2, rtol=1e-2)
        assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))


def test_dsplit_prefill_rows(orc):
    # many query rows of one sequence (more clusters than fit at once)
    rng = np.random.default_rng(8)
    wl = make_workload("mla_prefill", [700], [700], H=128, K=256, page_size=64, permute=True, seed=8, with_idx=False)
    with tuning(mla_dsplit=1):
        _compare(orc, wl, _random_indices(rng, wl, 256, pad_frac=0.02), rows=[0, 1, 63, 64, 255, 256, 500, 699])


def test_prefill_rows(orc):
    rng = np.random.default_rng(7)
    wl = make_workload("mla_prefill", [400], [400], H=16, K=128, page_size=64, permute=False, seed=7, with_idx=False)
    _compare(orc, wl, _random_indices(rng, wl, 128), rows=[0, 1, 2, 127, 128, 129, 255, 399])


def test_heads_32(orc):
    rng = np.random.default_rng(32)
    wl = make_workload("mla32", [2000, 300], [1, 1], H=32, K=700, page_size=64, seed=32, with_idx=False)
    _compare(orc, wl, _random_indices(rng, wl, 700, pad_frac=0.05))


@pytest.mark.parametrize("H,kernel", [(64, "heads64"), (128, "dsplit"), (128, "heads64")])
@pytest.mark.parametrize("order", ["rising", "falling"])
def test_reference_max_moves_across_tiles(orc, order, H, kernel):
    # logits that grow (or shrink) strongly from one 128-key tile to the next,
    # so that the running maximum moves by far more than 2^8 between tiles
    from indexer_top_sparse_gb300.inputs import bf16_bits, bf16_to_f32
    n, K = 1024, 1024
    wl = make_workload("mla_rescale", [n], [1], H=H, K=K, page_size=64, permute=True, seed=41, with_idx=False)
    kv = bf16_to_f32(wl.kv).reshape(-1, 576)
    q = bf16_to_f32(wl.q).reshape(H, 576)
    qdir = q[0] / np.linalg.norm(q[0])
    for s in range(n):
        row = wl.page_table[0][s // 64] * 64 + s % 64
        tile = s // 128
        f = (tile + 1) if order == "rising" else (8 - tile)
        kv[row, :] = 0.3 * kv[row, :] + 2.0 * f * qdir
    wl.kv = bf16_bits(kv.reshape(wl.kv.shape).astype(np.float32))
    wl.scale = 1.0
    idx = np.arange(K, dtype=np.int32)[None, :]
    with tuning(mla_splits=1, mla_dsplit=KERNELS[kernel]):
        _compare(orc, wl, idx)


@pytest.mark.parametrize("pair,kernel", [(1, "heads64"), (-1, "heads64"), (0, "auto")])
def test_128_heads_over_several_waves(orc, pair, kernel):
    # 200 query rows x 2 head groups: more CTAs than SMs (several waves); the
    # 64-head kernel with its head groups paired (1) or independent (-1), and
    # the automatic choice (the dims-split pair at this size)
    rng = np.random.default_rng(129)
    wl = make_workload("mla", [600, 300], [120, 80], H=128, K=192, page_size=64, seed=129, with_idx=False)
    with tuning(mla_pair=pair, mla_dsplit=KERNELS.get(kernel, 0)):
        _compare(orc, wl, _random_indices(rng, wl, 192, pad_frac=0.05))


@pytest.mark.parametrize("fp8", [False, True])
def test_paired_128_heads_matches(orc, fp8):
    # the two 64-head CTAs of a 128-head query as a cluster sharing each row
    import indexer_top_sparse_gb300 as d
    rng = np.random.default_rng(128)
    wl = make_workload("mla", [3000, 700], [1, 1], H=128, K=1024, page_size=64, seed=128, with_idx=False)
    if fp8:
        nope, rope, sc = orc.quant_fp8_rows(wl.kv)
        idx = _random_indices(rng, wl, 1024, pad_frac=0.05)
        d.set_tuning("mla_pair", 1)
        try:
            ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, idx.shape[1]))
            out = d.dsa_sparse_mla(dev_bf16(wl.q), dev(nope), dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q),
                                   dev(idx), wl.scale, workspace=ws, kv_rope=dev_bf16(rope), kv_scale=dev(sc),
                                   dtype="fp8_rowscale")
            ws.check()
        finally:
            d.set_tuning("mla_pair", 0)
        ref, _ = orc.sparse_mla(wl.q, nope, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size,
                                dtype=orc.KV_FP8_ROWSCALE, kv_rope=rope, kv_scale=sc)
        np.testing.assert_allclose(out.float().cpu().numpy(), ref, atol=ATOL, rtol=RTOL)
        return
    with tuning(mla_pair=1, mla_dsplit=-1):
        _compare(orc, wl, _random_indices(rng, wl, 1024, pad_frac=0.05))


@pytest.mark.parametrize("case", ["k1000_h128", "k1000_h64", "k2048_h128"])
@pytest.mark.parametrize("fp8", [False, True])
def test_stream_k_matches(orc, case, fp8):
    # one CTA per SM sharing all (row, head group, key tile) units: runs cross
    # into the next (row, head group) every few tiles, the last tile of a row
    # is ragged (K = 1000) and some indices are -1
    import indexer_top_sparse_gb300 as d
    K, H, T = {"k1000_h128": (1000, 128, 12), "k1000_h64": (1000, 64, 21), "k2048_h128": (2048, 128, 6)}[case]
    rng = np.random.default_rng(140 + K + H + fp8)
    lens = rng.integers(K + 10, 3 * K, size=T)
    wl = make_workload("sk", lens, [1] * T, H=H, K=K, page_size=64, seed=int(lens[0]), with_idx=False)
    idx = _random_indices(rng, wl, K, pad_frac=0.05)
    d.set_tuning("mla_stream_k", 1)
    d.set_tuning("mla_dsplit", -1)
    try:
        if fp8:
            nope, rope, sc = orc.quant_fp8_tiles(wl.kv)
            ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, K))
            out = d.dsa_sparse_mla(dev_bf16(wl.q), dev(nope), dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q),
                                   dev(idx), wl.scale, workspace=ws, kv_rope=dev_bf16(rope), kv_scale=dev(sc),
                                   dtype="fp8_tile128")
            ws.check()
            ref, _ = orc.sparse_mla(wl.q, nope, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size,
                                    dtype=orc.KV_FP8_TILE128, kv_rope=rope, kv_scale=sc)
            np.testing.assert_allclose(out.float().cpu().numpy(), ref, atol=ATOL, rtol=RTOL)
        else:
            _compare(orc, wl, idx)
    finally:
        d.set_tuning("mla_stream_k", 0)
        d.set_tuning("mla_dsplit", 0)


def test_stream_k_off_and_on_agree(orc):
    # a decode shape with one split per row and fewer CTAs than SMs, stream-K
    # forced on against the split grid: the same attention up to summation order
    import indexer_top_sparse_gb300 as d
    rng = np.random.default_rng(150)
    wl = make_workload("sk2", [4000] * 16, [1] * 16, H=128, K=2048, page_size=64, seed=150, with_idx=False)
    idx = dev(_random_indices(rng, wl, 2048))
    outs = []
    for mode in (1, -1):
        d.set_tuning("mla_stream_k", mode)
        d.set_tuning("mla_dsplit", -1)
        try:
            ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, 2048))
            lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
            o = d.dsa_sparse_mla(dev_bf16(wl.q), dev_bf16(wl.kv), dev(wl.page_table), dev(wl.seq_lens),
                                 dev(wl.cu_q), idx, wl.scale, workspace=ws, lse=lse)
            ws.check()
            outs.append((o.float().cpu().numpy(), lse.cpu().numpy()))
        finally:
            d.set_tuning("mla_stream_k", 0)
            d.set_tuning("mla_dsplit", 0)
    np.testing.assert_allclose(outs[0][0], outs[1][0], atol=1e-2, rtol=1e-2)
    np.testing.assert_allclose(outs[0][1], outs[1][1], atol=1e-4, rtol=1e-4)
    _every_row_against_oracle(orc, wl, idx.cpu().numpy(), outs)


def _every_row_against_oracle(orc, wl, idx, outs):
    """Both runs against the oracle on every row (rows on a thread pool: the
    oracle's calls release the interpreter lock)."""
    import concurrent.futures as cf
    import os
    rows = [np.array([t], np.int32) for t in range(wl.T)]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        refs = list(ex.map(lambda r: orc.sparse_mla(wl.q, wl.kv, wl.page_table, wl.cu_q, idx, wl.scale,
                                                    wl.page_size, rows=r), rows))
    ref = np.concatenate([o for o, _ in refs])
    ref_lse = np.concatenate([l for _, l in refs])
    for o, lse in outs:
        np.testing.assert_allclose(o, ref, atol=ATOL, rtol=RTOL)
        np.testing.assert_allclose(lse, ref_lse, atol=1e-3, rtol=1e-3)


def test_dsplit_and_heads64_agree_on_decode(orc):
    # the 32-row decode launch shape (two key splits) on both 128-head kernels:
    # the same attention up to summation order
    rng = np.random.default_rng(151)
    wl = make_workload("ds", [5000] * 32, [1] * 32, H=128, K=2048, page_size=64, seed=151, with_idx=False)
    idx = dev(_random_indices(rng, wl, 2048, pad_frac=0.01))
    import indexer_top_sparse_gb300 as d
    outs = []
    for kernel in ("dsplit", "heads64"):
        with tuning(mla_dsplit=KERNELS[kernel]):
            ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, 2048))
            lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
            o = d.dsa_sparse_mla(dev_bf16(wl.q), dev_bf16(wl.kv), dev(wl.page_table), dev(wl.seq_lens),
                                 dev(wl.cu_q), idx, wl.scale, workspace=ws, lse=lse)
            ws.check()
            outs.append((o.float().cpu().numpy(), lse.cpu().numpy()))
    np.testing.assert_allclose(outs[0][0], outs[1][0], atol=1e-2, rtol=1e-2)
    np.testing.assert_allclose(outs[0][1], outs[1][1], atol=1e-4, rtol=1e-4)
    _every_row_against_oracle(orc, wl, idx.cpu().numpy(), outs)
