"""Pins for the oracle's sparse MLA attention: selecting every position equals
dense softmax attention computed with torch (library softmax and matmul), a
single selected key returns its value row, a zero softmax scale gives the
plain mean with lse = log(n), the result ignores index order and -1 padding,
and the FP8 path equals the bf16 path on exactly representable values."""
import math

import numpy as np
import torch

from indexer_top_sparse_gb300.inputs import bf16_bits, bf16_to_f32, make_page_table


def _setup(seed, n, H=4, ps=16, D=576):
    rng = np.random.default_rng(seed)
    pt, P = make_page_table(rng, [n], ps)
    kv = bf16_bits(rng.standard_normal((P, ps, D)).astype(np.float32))
    q = bf16_bits(rng.standard_normal((1, H, D)).astype(np.float32))
    return rng, pt, P, kv, q


def _logical(kv, pt_row, ps, idx):
    rows = np.array([pt_row[s // ps] * ps + s % ps for s in idx])
    return kv.reshape(-1, kv.shape[-1])[rows]


def test_all_positions_equals_dense_attention(orc):
    n, ps, H = 90, 16, 4
    rng, pt, P, kv, q = _setup(20, n, H, ps)
    idx = np.arange(n, dtype=np.int32)[None, :]
    scale = 1 / math.sqrt(192)
    out, lse = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), idx, scale, ps)
    Kt = torch.from_numpy(bf16_to_f32(_logical(kv, pt[0], ps, range(n))).astype(np.float64))
    Qt = torch.from_numpy(bf16_to_f32(q[0]).astype(np.float64))
    logits = scale * (Qt @ Kt.T)
    ref = torch.softmax(logits, dim=-1) @ Kt[:, :512]
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(lse[0], torch.logsumexp(logits, -1).numpy(), rtol=1e-6)


def test_single_key_returns_value_row(orc):
    n, ps = 40, 16
    rng, pt, P, kv, q = _setup(21, n, 3, ps)
    idx = np.full((1, 8), -1, np.int32)
    idx[0, 5] = 17
    out, lse = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), idx, 0.3, ps)
    v = bf16_to_f32(_logical(kv, pt[0], ps, [17]))[0, :512]
    for h in range(3):
        np.testing.assert_allclose(out[0, h], v, rtol=1e-6, atol=0)


def test_zero_scale_is_mean_and_lse_log_n(orc):
    n, ps = 64, 16
    rng, pt, P, kv, q = _setup(22, n, 2, ps)
    sel = np.array([3, 9, 10, 33, 63], np.int32)
    out, lse = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), sel[None, :], 0.0, ps)
    v = bf16_to_f32(_logical(kv, pt[0], ps, sel))[:, :512].astype(np.float64)
    np.testing.assert_allclose(out[0, 0], v.mean(0), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(lse[0], np.log(5.0), rtol=1e-7)


def test_order_and_padding_invariance(orc):
    n, ps = 100, 16
    rng, pt, P, kv, q = _setup(23, n, 4, ps)
    sel = rng.choice(n, 30, replace=False).astype(np.int32)
    a, la = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), sel[None, :], 0.07, ps)
    perm = rng.permutation(sel)
    padded = np.concatenate([perm[:10], [-1, -1], perm[10:], [-1]]).astype(np.int32)
    b, lb = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), padded[None, :], 0.07, ps)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-7)
    np.testing.assert_allclose(la, lb, rtol=1e-7)
    # no valid entry: zero output, lse = -inf
    c, lc = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), np.full((1, 4), -1, np.int32), 0.07, ps)
    assert np.all(c == 0) and np.all(np.isneginf(lc))


def test_fp8_path_equals_bf16_path_on_representable_values(orc):
    n, ps, H = 48, 16, 3
    rng = np.random.default_rng(24)
    pt, P = make_page_table(rng, [n], ps)
    codes = rng.integers(0, 256, size=(P, ps, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x31
    codes[(codes & 0x78) >= 0x60] &= 0x9F                 # keep magnitudes moderate
    rope = bf16_bits(rng.standard_normal((P, ps, 64)).astype(np.float32))
    scale = (2.0 ** rng.integers(-3, 2, size=(P, ps))).astype(np.float32)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    deq = table[codes] * scale[..., None].astype(np.float64)
    full = np.concatenate([bf16_bits(deq.astype(np.float32)), rope], axis=-1)
    assert np.array_equal(bf16_to_f32(full[..., :512]), deq.astype(np.float32))
    q = bf16_bits(rng.standard_normal((1, H, 576)).astype(np.float32) * np.float32(0.05))
    sel = rng.choice(n, 20, replace=False).astype(np.int32)[None, :]
    a, la = orc.sparse_mla(q, codes, pt, np.array([0, 1], np.int32), sel, 0.1, ps, dtype=orc.KV_FP8_ROWSCALE,
                           kv_rope=rope, kv_scale=scale, D=576, Dv=512, num_pages=P)
    b, lb = orc.sparse_mla(q, full, pt, np.array([0, 1], np.int32), sel, 0.1, ps)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-9)
    np.testing.assert_allclose(la, lb, rtol=1e-12)


def test_fp8_quantised_cache_close_to_bf16_attention(orc):
    n, ps, H = 128, 64, 8
    rng = np.random.default_rng(25)
    pt, P = make_page_table(rng, [n], ps)
    kv = bf16_bits(rng.standard_normal((P, ps, 576)).astype(np.float32))
    nope, rope, sc = orc.quant_fp8_rows(kv)
    q = bf16_bits(rng.standard_normal((1, H, 576)).astype(np.float32))
    sel = rng.choice(n, 64, replace=False).astype(np.int32)[None, :]
    a, _ = orc.sparse_mla(q, nope, pt, np.array([0, 1], np.int32), sel, 1 / math.sqrt(192), ps,
                          dtype=orc.KV_FP8_ROWSCALE, kv_rope=rope, kv_scale=sc, D=576, Dv=512, num_pages=P)
    b, _ = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), sel, 1 / math.sqrt(192), ps)
    np.testing.assert_allclose(a, b, atol=6e-2, rtol=3e-2)


def test_fp8_tile_path_equals_bf16_path_on_representable_values(orc):
    # power-of-two scales that differ per 128-dim tile: the dequantised values
    # are exact in bf16, so the tile path must equal the bf16 path; a wrong
    # tile index (or the row scale) changes the result
    n, ps, H = 40, 16, 3
    rng = np.random.default_rng(26)
    pt, P = make_page_table(rng, [n], ps)
    codes = rng.integers(0, 256, size=(P, ps, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x31
    codes[(codes & 0x78) >= 0x60] &= 0x9F
    rope = bf16_bits(rng.standard_normal((P, ps, 64)).astype(np.float32))
    scale = (2.0 ** rng.integers(-4, 3, size=(P, ps, 4))).astype(np.float32)
    scale[..., 2] *= np.float32(8.0)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    deq = table[codes] * np.repeat(scale, 128, axis=-1).astype(np.float64)
    full = np.concatenate([bf16_bits(deq.astype(np.float32)), rope], axis=-1)
    assert np.array_equal(bf16_to_f32(full[..., :512]), deq.astype(np.float32))
    q = bf16_bits(rng.standard_normal((1, H, 576)).astype(np.float32) * np.float32(0.05))
    sel = rng.choice(n, 24, replace=False).astype(np.int32)[None, :]
    a, la = orc.sparse_mla(q, codes, pt, np.array([0, 1], np.int32), sel, 0.1, ps, dtype=orc.KV_FP8_TILE128,
                           kv_rope=rope, kv_scale=scale, D=576, Dv=512, num_pages=P)
    b, lb = orc.sparse_mla(q, full, pt, np.array([0, 1], np.int32), sel, 0.1, ps)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-9)
    np.testing.assert_allclose(la, lb, rtol=1e-12)


def test_fp8_tile_quantised_cache_close_to_bf16_attention(orc):
    n, ps, H = 128, 64, 8
    rng = np.random.default_rng(27)
    pt, P = make_page_table(rng, [n], ps)
    kv = rng.standard_normal((P, ps, 576)).astype(np.float32)
    kv[..., 256:384] *= np.float32(0.01)                    # a quiet tile: finer scale than the row's
    kv = bf16_bits(kv)
    nope, rope, sc = orc.quant_fp8_tiles(kv)
    q = bf16_bits(rng.standard_normal((1, H, 576)).astype(np.float32))
    sel = rng.choice(n, 64, replace=False).astype(np.int32)[None, :]
    a, _ = orc.sparse_mla(q, nope, pt, np.array([0, 1], np.int32), sel, 1 / math.sqrt(192), ps,
                          dtype=orc.KV_FP8_TILE128, kv_rope=rope, kv_scale=sc, D=576, Dv=512, num_pages=P)
    b, _ = orc.sparse_mla(q, kv, pt, np.array([0, 1], np.int32), sel, 1 / math.sqrt(192), ps)
    np.testing.assert_allclose(a, b, atol=6e-2, rtol=3e-2)
