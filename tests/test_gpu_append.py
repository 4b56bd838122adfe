"""GPU cache append against the oracle, bit for bit: new tokens' index keys
(bf16 or MXFP8) and latent rows (bf16, FP8 with row or tile scales) written
into their page slots for decode (one token per sequence), prefill (whole
sequences) and ragged batches; every other cache byte unchanged; an
out-of-range page reported through the workspace with nothing written for
that token."""
import zlib

import numpy as np
import pytest
import torch

from _util import dev
from indexer_top_sparse_gb300.inputs import bf16_bits, make_page_table

pytestmark = pytest.mark.gpu

IDX = {"bf16": 0, "mxfp8": 1}
KV = {"bf16": 0, "fp8_rowscale": 1, "fp8_tile128": 2}


def _batch(rng, lens, n_new, ps):
    lens = np.asarray(lens, np.int32)
    n_new = np.asarray(n_new, np.int32)
    pt, P = make_page_table(rng, lens, ps)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(n_new)
    T = int(cu[-1])
    k_new = bf16_bits(rng.standard_normal((T, 128)).astype(np.float32))
    kv_new = rng.standard_normal((T, 576)).astype(np.float32)
    kv_new[::7, :128] = 0.0                                   # zero blocks / tiles
    kv_new[1::5, 256:384] *= np.float32(1e-3)
    return lens, cu, pt, P, k_new, bf16_bits(kv_new)


def _caches(rng, P, ps, idx_dtype, kv_dtype):
    """Random initial cache bytes (the same on both sides)."""
    k = rng.integers(0, 256, size=(P, ps, 128 * (2 if idx_dtype == "bf16" else 1)), dtype=np.uint8)
    ks = rng.integers(0, 256, size=(P, ps, 4), dtype=np.uint8)
    if kv_dtype == "bf16":
        kv, rope, sc = rng.integers(0, 256, size=(P, ps, 1152), dtype=np.uint8), None, None
    else:
        kv = rng.integers(0, 256, size=(P, ps, 512), dtype=np.uint8)
        rope = rng.integers(0, 1 << 16, size=(P, ps, 64), dtype=np.uint16)
        sc = rng.standard_normal((P, ps) if kv_dtype == "fp8_rowscale" else (P, ps, 4)).astype(np.float32)
    return k, ks, kv, rope, sc


def _gpu(lens, cu, pt, k_new, kv_new, caches, idx_dtype, kv_dtype, ws=None):
    import indexer_top_sparse_gb300 as d
    k, ks, kv, rope, sc = caches
    gk = dev(k).view(torch.bfloat16) if idx_dtype == "bf16" else dev(k)
    gks = dev(ks) if idx_dtype == "mxfp8" else None
    gkv = dev(kv).view(torch.bfloat16) if kv_dtype == "bf16" else dev(kv)
    grope = None if rope is None else dev(rope.view(np.int16)).view(torch.bfloat16)
    gsc = None if sc is None else dev(sc)
    kn = None if k_new is None else dev(k_new.view(np.int16)).view(torch.bfloat16)
    vn = None if kv_new is None else dev(kv_new.view(np.int16)).view(torch.bfloat16)
    d.dsa_cache_append(dev(pt), dev(lens), dev(cu), k_new=kn, kv_new=vn, k_cache=gk, k_scale=gks, kv_cache=gkv,
                       kv_rope=grope, kv_scale=gsc, idx_dtype=idx_dtype, kv_dtype=kv_dtype, workspace=ws)
    torch.cuda.synchronize()
    out = (gk.view(torch.uint8).cpu().numpy(), None if gks is None else gks.cpu().numpy(),
           gkv.view(torch.uint8).cpu().numpy(), None if grope is None else grope.view(torch.int16).cpu().numpy(),
           None if gsc is None else gsc.cpu().numpy())
    return out


def _oracle(orc, lens, cu, pt, k_new, kv_new, caches, idx_dtype, kv_dtype):
    k, ks, kv, rope, sc = (None if c is None else c.copy() for c in caches)
    P, ps = kv.shape[0], kv.shape[1]
    kc = k.view(np.uint16) if idx_dtype == "bf16" else k
    vc = kv.view(np.uint16) if kv_dtype == "bf16" else kv
    rc = orc.cache_append(pt, lens, cu, ps, k_new=k_new, kv_new=kv_new, idx_dtype=IDX[idx_dtype], k_cache=kc,
                          k_scale=ks if idx_dtype == "mxfp8" else None, kv_dtype=KV[kv_dtype], kv_cache=vc,
                          kv_rope=rope, kv_scale=sc, num_pages=P)
    return rc, (k, ks if idx_dtype == "mxfp8" else None, kv, None if rope is None else rope.view(np.int16), sc)


CASES = {"decode": ([300, 65, 64, 1, 129], [1, 1, 1, 1, 1]),
         "prefill": ([700, 64], [700, 64]),
         "ragged": ([1000, 130, 77, 5], [37, 130, 1, 4])}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("kv_dtype", list(KV))
@pytest.mark.parametrize("idx_dtype", list(IDX))
def test_append_bit_exact(orc, idx_dtype, kv_dtype, case):
    rng = np.random.default_rng(zlib.crc32(f"{idx_dtype}/{kv_dtype}/{case}".encode()))
    ps = 64
    lens, cu, pt, P, k_new, kv_new = _batch(rng, *CASES[case], ps)
    caches = _caches(rng, P, ps, idx_dtype, kv_dtype)
    got = _gpu(lens, cu, pt, k_new, kv_new, caches, idx_dtype, kv_dtype)
    rc, ref = _oracle(orc, lens, cu, pt, k_new, kv_new, caches, idx_dtype, kv_dtype)
    assert rc == 0
    for name, g, r in zip(("k_cache", "k_scale", "kv_cache", "kv_rope", "kv_scale"), got, ref):
        if r is not None:
            assert np.array_equal(g, r), name


def test_append_one_cache_only(orc):
    rng = np.random.default_rng(5)
    ps = 16
    lens, cu, pt, P, k_new, kv_new = _batch(rng, [40, 17], [3, 2], ps)
    caches = _caches(rng, P, ps, "mxfp8", "fp8_tile128")
    got = _gpu(lens, cu, pt, k_new, None, caches, "mxfp8", "fp8_tile128")
    rc, ref = _oracle(orc, lens, cu, pt, k_new, None, caches, "mxfp8", "fp8_tile128")
    assert rc == 0
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    assert np.array_equal(got[2], caches[2]) and np.array_equal(got[4], caches[4])   # KV untouched


def test_append_bad_page_is_reported(orc):
    import indexer_top_sparse_gb300 as d
    rng = np.random.default_rng(6)
    ps = 16
    lens, cu, pt, P, k_new, kv_new = _batch(rng, [40, 40], [2, 2], ps)
    pt = pt.copy()
    pt[1, (int(lens[1]) - 1) // ps] = P + 3
    caches = _caches(rng, P, ps, "bf16", "fp8_rowscale")
    ws = d.Workspace(256)
    got = _gpu(lens, cu, pt, k_new, kv_new, caches, "bf16", "fp8_rowscale", ws=ws)
    with pytest.raises(d.DSAError, match="page"):
        ws.check()
    rc, ref = _oracle(orc, lens, cu, pt, k_new, kv_new, caches, "bf16", "fp8_rowscale")
    assert rc == -1
    for g, r in zip(got, ref):
        if r is not None:
            assert np.array_equal(g, r)
