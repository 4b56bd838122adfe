"""Shared helpers for the tests: moving seeded host inputs to the device and
the parity comparisons.  No method arithmetic lives here."""
from __future__ import annotations

import numpy as np
import pytest
import torch


def gpu_available() -> bool:
    return torch.cuda.is_available()


requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_device(wl):
    """Device tensors of a Workload (only the arrays it has)."""
    d = {"page_table": dev(wl.page_table), "seq_lens": dev(wl.seq_lens), "cu_q": dev(wl.cu_q)}
    if wl.q_idx is not None:
        d["q_idx"] = dev_bf16(wl.q_idx)
        d["head_w"] = dev(wl.head_w)
        d["k_idx"] = dev_bf16(wl.k_idx)
    if wl.q is not None:
        d["q"] = dev_bf16(wl.q)
        d["kv"] = dev_bf16(wl.kv)
    return d


class tuning:
    """Set library tuning knobs for the duration of a with-block (0 = automatic
    afterwards)."""

    def __init__(self, **knobs):
        self.knobs = knobs

    def __enter__(self):
        import indexer_top_sparse_gb300 as d
        for k, v in self.knobs.items():
            d.set_tuning(k, v)
        return self

    def __exit__(self, *exc):
        import indexer_top_sparse_gb300 as d
        for k in self.knobs:
            d.set_tuning(k, 0)
        return False


def score_magnitude(q_bits, w, k_rows_bits):
    """sum_j |w_j| * max(q_j . k, 0) per key row (fp64), the natural scale of a
    score when the signed head weights let terms cancel."""
    from indexer_top_sparse_gb300.inputs import bf16_to_f32
    q = bf16_to_f32(q_bits).astype(np.float64)          # [64, 128]
    k = bf16_to_f32(k_rows_bits).astype(np.float64)     # [n, 128]
    dots = k @ q.T                                      # [n, 64]
    return (np.maximum(dots, 0) * np.abs(w.astype(np.float64))[None, :]).sum(1)


def logical_rows(cache, pt_row, ps, n):
    rows = np.array([pt_row[s // ps] * ps + s % ps for s in range(n)], np.int64)
    return cache.reshape(-1, cache.shape[-1])[rows]


def check_index_sets(gpu_idx, ref_idx, ref_scores, n_valid, K, rel=1e-3):
    """Top-K sets must agree except at positions whose oracle score lies within
    `rel` (relative) of the oracle's K-th score."""
    m = min(K, n_valid)
    g = gpu_idx[:m]
    assert np.all(gpu_idx[m:] == -1), "padding must be -1"
    assert np.all(np.diff(g) > 0), "indices must be ascending and distinct"
    assert g.min() >= 0 and g.max() < n_valid
    if n_valid <= K:
        assert np.array_equal(g, np.arange(n_valid))
        return 0
    r = ref_idx[:m]
    diff = np.setxor1d(g, r)
    if diff.size == 0:
        return 0
    kth = np.sort(ref_scores[:n_valid])[::-1][K - 1]
    tol = rel * max(abs(kth), 1e-30)
    bad = diff[np.abs(ref_scores[diff] - kth) > tol]
    assert bad.size == 0, f"positions {bad[:10]} differ beyond the near-threshold band (kth={kth})"
    return int(diff.size)
