"""Pins for the oracle's indexer scores and fused indexer + Top-K: special
cases that reduce to a library dot product, exact integer arithmetic,
linearity in the head weights, invariance under page permutation, the MXFP8
path against the bf16 path on exactly representable values, and the causal
query layout of prefill and chunked prefill."""
import numpy as np
import torch

from indexer_top_sparse_gb300.inputs import bf16_bits, bf16_to_f32, make_page_table, make_workload


def _cache(rng, P, ps, d, ints=False):
    if ints:
        return bf16_bits(rng.integers(-3, 4, size=(P, ps, d)).astype(np.float32))
    return bf16_bits(rng.standard_normal((P, ps, d)).astype(np.float32))


def _logical_keys(k_cache, pt_row, ps, n):
    rows = np.array([pt_row[s // ps] * ps + s % ps for s in range(n)])
    return k_cache.reshape(-1, k_cache.shape[-1])[rows]


def test_single_head_unit_weight_is_relu_dot(orc):
    rng = np.random.default_rng(10)
    ps, d, n = 16, 128, 150
    pt, P = make_page_table(rng, [n], ps)
    kc = _cache(rng, P, ps, d)
    q = bf16_bits(rng.standard_normal((1, d)).astype(np.float32))
    w = np.ones(1, np.float32)
    got = orc.index_scores_row(q, w, kc, pt[0], ps, n)
    K = bf16_to_f32(_logical_keys(kc, pt[0], ps, n)).astype(np.float64)
    dots = torch.from_numpy(K) @ torch.from_numpy(bf16_to_f32(q)[0].astype(np.float64))
    want = np.maximum(dots.numpy(), 0).astype(np.float32)
    np.testing.assert_allclose(got, want, rtol=2e-7, atol=0)
    # negative weight flips the sign of the ReLU'd dot
    got2 = orc.index_scores_row(q, np.array([-2.0], np.float32), kc, pt[0], ps, n)
    np.testing.assert_allclose(got2, -2 * want, rtol=2e-7, atol=0)


def test_integer_inputs_exact(orc):
    rng = np.random.default_rng(11)
    ps, d, n, H = 8, 64, 40, 5
    pt, P = make_page_table(rng, [n], ps)
    kc = _cache(rng, P, ps, d, ints=True)
    q = bf16_bits(rng.integers(-3, 4, size=(H, d)).astype(np.float32))
    w = rng.integers(-4, 5, size=H).astype(np.float32)
    got = orc.index_scores_row(q, w, kc, pt[0], ps, n)
    K = bf16_to_f32(_logical_keys(kc, pt[0], ps, n)).astype(np.int64)
    Q = bf16_to_f32(q).astype(np.int64)
    for s in range(n):
        acc = 0
        for j in range(H):
            dot = int(np.dot(Q[j], K[s]))
            acc += int(w[j]) * max(dot, 0)
        assert got[s] == float(acc)


def test_head_additivity(orc):
    rng = np.random.default_rng(12)
    ps, d, n = 32, 128, 100
    pt, P = make_page_table(rng, [n], ps)
    kc = _cache(rng, P, ps, d)
    q = bf16_bits(rng.standard_normal((6, d)).astype(np.float32))
    w = rng.standard_normal(6).astype(np.float32)
    full = orc.index_scores_row(q, w, kc, pt[0], ps, n).astype(np.float64)
    a = orc.index_scores_row(q[:2], w[:2], kc, pt[0], ps, n).astype(np.float64)
    b = orc.index_scores_row(q[2:], w[2:], kc, pt[0], ps, n).astype(np.float64)
    mag = np.abs(a) + np.abs(b) + 1e-30
    assert np.all(np.abs(full - (a + b)) <= 2e-7 * mag * 2)
    # zero weights give zero scores
    z = orc.index_scores_row(q, np.zeros(6, np.float32), kc, pt[0], ps, n)
    assert np.all(z == 0)


def test_page_permutation_invariance(orc):
    rng = np.random.default_rng(13)
    ps, d, n = 16, 128, 200
    pt_a, P = make_page_table(np.random.default_rng(1), [n], ps, permute=False)
    pt_b, _ = make_page_table(np.random.default_rng(2), [n], ps, permute=True)
    kc_a = _cache(rng, P, ps, d)
    # place logical page i of layout a at physical page pt_b[0, i] in layout b
    kc_b = np.empty_like(kc_a)
    for i in range(P):
        kc_b[pt_b[0, i]] = kc_a[pt_a[0, i]]
    q = bf16_bits(rng.standard_normal((4, d)).astype(np.float32))
    w = rng.standard_normal(4).astype(np.float32)
    sa = orc.index_scores_row(q, w, kc_a, pt_a[0], ps, n)
    sb = orc.index_scores_row(q, w, kc_b, pt_b[0], ps, n)
    assert np.array_equal(sa, sb)


def test_mxfp8_path_equals_bf16_path_on_decoded_values(orc):
    rng = np.random.default_rng(14)
    ps, d, n, H = 16, 128, 64, 3
    pt, P = make_page_table(rng, [n], ps)
    codes_k = rng.integers(0, 256, size=(P, ps, d)).astype(np.uint8)
    codes_k[(codes_k & 0x7F) == 0x7F] = 0x10          # no NaN codes
    codes_q = rng.integers(0, 256, size=(H, d)).astype(np.uint8)
    codes_q[(codes_q & 0x7F) == 0x7F] = 0x22
    sk = rng.integers(120, 134, size=(P, ps, d // 32)).astype(np.uint8)
    sq = rng.integers(120, 134, size=(H, d // 32)).astype(np.uint8)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    deq_k = table[codes_k] * np.repeat(2.0 ** (sk.astype(np.float64) - 127), 32, axis=-1)
    deq_q = table[codes_q] * np.repeat(2.0 ** (sq.astype(np.float64) - 127), 32, axis=-1)
    # every decoded value has <= 4 significant bits: exact in bf16
    kb = bf16_bits(deq_k.astype(np.float32))
    qb = bf16_bits(deq_q.astype(np.float32))
    assert np.array_equal(bf16_to_f32(kb), deq_k.astype(np.float32))
    w = rng.standard_normal(H).astype(np.float32)
    s_mx = orc.index_scores_row(codes_q, w, codes_k, pt[0], ps, n, dtype=orc.IDX_MXFP8, q_scale=sq, k_scale=sk)
    s_bf = orc.index_scores_row(qb, w, kb, pt[0], ps, n)
    assert np.array_equal(s_mx, s_bf)


def test_prefill_causal_layout(orc):
    wl = make_workload("t", [70, 33], [70, 5], H=4, K=16, page_size=16, seed=3, with_kv=False)
    idx, sc = orc.index_topk(wl.q_idx, wl.head_w, wl.k_idx, wl.page_table, wl.seq_lens, wl.cu_q, wl.K,
                             wl.page_size, want_scores=True, ld_scores=80)
    pos = wl.query_pos()
    assert list(pos[:3]) == [0, 1, 2] and pos[69] == 69 and list(pos[70:]) == [28, 29, 30, 31, 32]
    for t in range(wl.T):
        n_valid = min(wl.K, pos[t] + 1)
        row = idx[t]
        assert np.all(row[:n_valid] >= 0) and np.all(row[:n_valid] <= pos[t]) and np.all(row[n_valid:] == -1)
        assert np.all(np.isnan(sc[t, pos[t] + 1:]))
        # selection of the row equals Top-K of its own scores
        want = orc.topk_rows(sc[t:t + 1, :pos[t] + 1], np.array([pos[t] + 1], np.int32), wl.K)[0]
        assert np.array_equal(row, want)
    # row subsets give the same answer as the full batch
    rows = np.array([0, 69, 72], np.int32)
    sub = orc.index_topk(wl.q_idx, wl.head_w, wl.k_idx, wl.page_table, wl.seq_lens, wl.cu_q, wl.K,
                         wl.page_size, rows=rows)
    assert np.array_equal(sub, idx[rows])
