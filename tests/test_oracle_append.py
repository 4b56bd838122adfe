"""Pins for the oracle's cache append: appended latent rows read back through
the oracle's attention (one selected key returns its value row, a pinned
property), index keys and quantised rows read back through the page table
equal the pinned codecs applied to the new rows, appending one decode step at
a time equals one prefill append, rows that are not appended stay untouched,
and a token whose page id is out of range writes nothing."""
import numpy as np
import pytest

from indexer_top_sparse_gb300.inputs import bf16_bits, make_page_table


def _batch(rng, lens, n_new, ps):
    lens = np.asarray(lens, np.int32)
    n_new = np.asarray(n_new, np.int32)
    pt, P = make_page_table(rng, lens, ps)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(n_new)
    T = int(cu[-1])
    k_new = bf16_bits(rng.standard_normal((T, 128)).astype(np.float32))
    kv_new = bf16_bits(rng.standard_normal((T, 576)).astype(np.float32))
    pos = np.concatenate([np.arange(l - n, l) for l, n in zip(lens, n_new)]).astype(np.int64)
    seq = np.repeat(np.arange(len(lens)), n_new)
    return lens, cu, pt, P, k_new, kv_new, pos, seq


def _rows(pt, ps, seq, pos):
    return np.array([pt[b, p // ps] * ps + p % ps for b, p in zip(seq, pos)])


def _caches(P, ps, idx_dtype, kv_dtype, orc, fill=0x55):
    k = np.full((P, ps, 128), fill, np.uint16 if idx_dtype == orc.IDX_BF16 else np.uint8)
    ks = np.full((P, ps, 4), fill, np.uint8)
    if kv_dtype == orc.KV_BF16:
        kv, rope, sc = np.full((P, ps, 576), fill, np.uint16), None, None
    else:
        kv = np.full((P, ps, 512), fill, np.uint8)
        rope = np.full((P, ps, 64), fill, np.uint16)
        sc = np.full((P, ps) if kv_dtype == orc.KV_FP8_ROWSCALE else (P, ps, 4), 7.0, np.float32)
    return k, ks, kv, rope, sc


def test_appended_rows_read_back_through_attention(orc):
    rng = np.random.default_rng(40)
    ps = 16
    lens, cu, pt, P, k_new, kv_new, pos, seq = _batch(rng, [300, 130, 64], [5, 1, 64], ps)
    kv = np.full((P, ps, 576), 0x7FC0, np.uint16)          # NaN everywhere not appended
    rc = orc.cache_append(pt, lens, cu, ps, kv_new=kv_new, kv_cache=kv)
    assert rc == 0
    q = bf16_bits(rng.standard_normal((1, 2, 576)).astype(np.float32))
    for t in range(len(pos)):
        cq = np.zeros(len(lens) + 1, np.int32)
        cq[seq[t] + 1:] = 1                                  # one query row, in sequence seq[t]
        out, lse = orc.sparse_mla(q, kv, pt, cq, np.array([[pos[t]]], np.int32), 0.3, ps)
        v = kv_new[t, :512].astype(np.uint32) << 16
        assert np.array_equal(out[0], np.broadcast_to(v.view(np.float32), out[0].shape)), t


@pytest.mark.parametrize("idx_dtype", ["bf16", "mxfp8"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "rows", "tiles"])
def test_appended_rows_equal_codecs(orc, idx_dtype, kv_dtype):
    idt = orc.IDX_BF16 if idx_dtype == "bf16" else orc.IDX_MXFP8
    kdt = {"bf16": orc.KV_BF16, "rows": orc.KV_FP8_ROWSCALE, "tiles": orc.KV_FP8_TILE128}[kv_dtype]
    rng = np.random.default_rng(41)
    ps = 8
    lens, cu, pt, P, k_new, kv_new, pos, seq = _batch(rng, [50, 17, 33], [3, 17, 1], ps)
    k, ks, kv, rope, sc = _caches(P, ps, idt, kdt, orc)
    assert orc.cache_append(pt, lens, cu, ps, k_new=k_new, kv_new=kv_new, idx_dtype=idt, k_cache=k, k_scale=ks,
                            kv_dtype=kdt, kv_cache=kv, kv_rope=rope, kv_scale=sc) == 0
    rows = _rows(pt, ps, seq, pos)
    flat = lambda a: a.reshape((P * ps,) + a.shape[2:])
    if idt == orc.IDX_BF16:
        assert np.array_equal(flat(k)[rows], k_new)
    else:
        c, e = orc.quant_mxfp8(k_new)
        assert np.array_equal(flat(k)[rows], c) and np.array_equal(flat(ks)[rows], e)
    if kdt == orc.KV_BF16:
        assert np.array_equal(flat(kv)[rows], kv_new)
    else:
        n, r, s = (orc.quant_fp8_rows if kdt == orc.KV_FP8_ROWSCALE else orc.quant_fp8_tiles)(kv_new)
        assert np.array_equal(flat(kv)[rows], n) and np.array_equal(flat(rope)[rows], r)
        assert np.array_equal(flat(sc)[rows], s)
    # every other row keeps its fill
    other = np.setdiff1d(np.arange(P * ps), rows)
    assert np.all(flat(kv)[other] == 0x55) and np.all(flat(k)[other] == 0x55)


@pytest.mark.parametrize("kv_dtype", ["bf16", "tiles"])
def test_decode_steps_equal_one_prefill_append(orc, kv_dtype):
    kdt = orc.KV_BF16 if kv_dtype == "bf16" else orc.KV_FP8_TILE128
    rng = np.random.default_rng(42)
    ps = 16
    lens = np.array([40, 23], np.int32)
    lens_, cu, pt, P, k_new, kv_new, pos, seq = _batch(rng, lens, lens, ps)   # every position is new
    a = _caches(P, ps, orc.IDX_MXFP8, kdt, orc)
    assert orc.cache_append(pt, lens, cu, ps, k_new=k_new, kv_new=kv_new, idx_dtype=orc.IDX_MXFP8, k_cache=a[0],
                            k_scale=a[1], kv_dtype=kdt, kv_cache=a[2], kv_rope=a[3], kv_scale=a[4]) == 0
    b = _caches(P, ps, orc.IDX_MXFP8, kdt, orc)
    for step in range(int(lens.max())):
        live = np.nonzero(lens > step)[0]
        sl = np.minimum(lens, step + 1).astype(np.int32)
        cq = np.zeros(len(lens) + 1, np.int32)
        cq[1:] = np.cumsum(lens > step)
        toks = np.array([cu[s] + step for s in live])
        assert orc.cache_append(pt, sl, cq, ps, k_new=k_new[toks], kv_new=kv_new[toks], idx_dtype=orc.IDX_MXFP8,
                                k_cache=b[0], k_scale=b[1], kv_dtype=kdt, kv_cache=b[2], kv_rope=b[3],
                                kv_scale=b[4]) == 0
    for x, y in zip(a, b):
        if x is not None:
            assert np.array_equal(x, y)


def test_bad_page_writes_nothing_for_that_token(orc):
    rng = np.random.default_rng(43)
    ps = 8
    lens, cu, pt, P, k_new, kv_new, pos, seq = _batch(rng, [20, 20], [2, 2], ps)
    pt = pt.copy()
    pt[1, (int(lens[1]) - 1) // ps] = P + 5                  # last page of sequence 1 out of range
    kv = np.full((P, ps, 576), 0x55, np.uint16)
    rc = orc.cache_append(pt, lens, cu, ps, kv_new=kv_new, kv_cache=kv)
    assert rc == -1
    rows = _rows(pt, ps, seq[:2], pos[:2])
    assert np.array_equal(kv.reshape(-1, 576)[rows], kv_new[:2])
    assert np.sum(kv.reshape(-1, 576)[:, 0] != 0x55) == 2
