"""Seeded synthetic inputs for the DSA path, shared by the CUDA path's tests
and benchmark and by the CPU oracle.

This module holds none of the method's arithmetic: it draws N(0,1) values,
rounds them to bf16 bit patterns, builds paged-cache page tables (a seeded
Fisher-Yates permutation of physical pages) and the per-sequence query
layout.  Quantisation, scoring, selection and attention are not here: the
CUDA path and the oracle each do their own.

Workload shapes follow the decode and prefill cases the pages describe: an
index-key cache of 128-dim keys read through a page table, 64 index heads with
learned per-head weights, and a 576-wide latent KV row (512 latent + 64 rope)
read by index ("Day0 Inference Support and Performance Optimization for
New-Architecture LLMs", §2 item 2 and §4; "Optimizing Inference for Hybrid
Attention LLMs: A Practical Guide to Day-0 Adaptation", §3.1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

H_I = 64       # index heads
D_I = 128      # index head dim
D_QK = 576     # latent (512) + rope (64)
D_V = 512      # value dim = latent part


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) and return the
    16-bit patterns as uint16.  Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) draws rounded to bf16 bits, generated in chunks to bound the
    float32 temporary."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclass
class Workload:
    """One batch of the DSA path.  Arrays are host numpy arrays:

    q_idx     [T, 64, 128]  bf16 bits  index queries
    head_w    [T, 64]       fp32       per-head weights
    k_idx     [P, ps, 128]  bf16 bits  paged index-key cache
    q         [T, H, 576]   bf16 bits  attention queries
    kv        [P, ps, 576]  bf16 bits  paged latent KV cache
    page_table[B, maxp]     int32      logical page -> physical page
    seq_lens  [B]           int32      cached length per sequence
    cu_q      [B+1]         int32      query rows of sequence b: cu_q[b]..cu_q[b+1]-1,
                                       the last positions of that sequence
    """
    name: str
    B: int
    T: int
    H: int
    K: int
    page_size: int
    seq_lens: np.ndarray
    cu_q: np.ndarray
    page_table: np.ndarray
    num_pages: int
    q_idx: np.ndarray
    head_w: np.ndarray
    k_idx: np.ndarray
    q: np.ndarray
    kv: np.ndarray
    scale: float
    seed: int
    extra: dict = field(default_factory=dict)

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    def query_pos(self) -> np.ndarray:
        """Absolute position of every query row."""
        pos = np.empty(self.T, np.int64)
        for b in range(self.B):
            a, e = int(self.cu_q[b]), int(self.cu_q[b + 1])
            pos[a:e] = int(self.seq_lens[b]) - (e - a) + np.arange(e - a)
        return pos


def make_page_table(rng: np.random.Generator, seq_lens, page_size: int, permute: bool = True):
    """Pages for each sequence: ceil(len/ps) logical pages mapped onto a
    seeded permutation of all physical pages.  Unused table slots hold -1."""
    seq_lens = np.asarray(seq_lens, np.int64)
    npg = (seq_lens + page_size - 1) // page_size
    total = int(npg.sum())
    phys = rng.permutation(total).astype(np.int32) if permute else np.arange(total, dtype=np.int32)
    maxp = int(npg.max()) if len(npg) else 0
    pt = np.full((len(seq_lens), max(maxp, 1)), -1, np.int32)
    o = 0
    for b, n in enumerate(npg):
        pt[b, :n] = phys[o:o + n]
        o += int(n)
    return pt, total


def make_workload(name: str, seq_lens, n_queries, *, H: int, K: int, page_size: int = 64, permute: bool = True,
                  seed: int = 0, with_kv: bool = True, with_idx: bool = True) -> Workload:
    """Build a workload.  seq_lens[b] is the cached length of sequence b
    (including its queries); n_queries[b] how many of its last positions are
    queries in this batch."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    n_queries = np.asarray(n_queries, np.int32)
    if np.any(n_queries > seq_lens) or np.any(n_queries < 0):
        raise ValueError("each sequence needs 0 <= queries <= length")
    B = len(seq_lens)
    cu_q = np.zeros(B + 1, np.int32)
    cu_q[1:] = np.cumsum(n_queries)
    T = int(cu_q[-1])
    pt, P = make_page_table(rng, seq_lens, page_size, permute)
    q_idx = normal_bf16(rng, (T, H_I, D_I)) if with_idx else None
    head_w = (rng.standard_normal((T, H_I), dtype=np.float32) / np.float32(8.0)).astype(np.float32) \
        if with_idx else None
    k_idx = normal_bf16(rng, (P, page_size, D_I)) if with_idx else None
    q = normal_bf16(rng, (T, H, D_QK)) if with_kv else None
    kv = normal_bf16(rng, (P, page_size, D_QK)) if with_kv else None
    return Workload(name=name, B=B, T=T, H=H, K=K, page_size=page_size, seq_lens=seq_lens, cu_q=cu_q,
                    page_table=pt, num_pages=P, q_idx=q_idx, head_w=head_w, k_idx=k_idx, q=q, kv=kv,
                    scale=float(1.0 / np.sqrt(192.0)), seed=seed)


# Named workloads: the decode and prefill shapes the benchmark and the
# full-size parity tests use.

def decode_small(seed: int = 0) -> Workload:
    """Decode, 1 sequence of 2048 cached positions, 1 query, K=256, 16 MLA
    heads, contiguous cache (one 2048-row page)."""
    return make_workload("decode_b1_n2048_k256_h16_contiguous", [2048], [1], H=16, K=256, page_size=2048,
                         permute=False, seed=seed)


def decode_b32_n32k(seed: int = 0) -> Workload:
    """Decode, 32 sequences at 32768 cached positions, 1 query each, K=2048,
    128 MLA heads, paged (64 rows per page, permuted)."""
    return make_workload("decode_b32_n32768_k2048_h128_paged64", [32768] * 32, [1] * 32, H=128, K=2048,
                         page_size=64, permute=True, seed=seed)


def decode_b64_mixed(seed: int = 0) -> Workload:
    """Decode, 64 sequences with lengths uniform in [4096, 131072], K=2048,
    128 MLA heads, paged (64).  Values are drawn in bf16 before FP8/MXFP8
    quantisation, which each side performs itself."""
    rng = np.random.default_rng(seed + 7919)
    lens = rng.integers(4096, 131072, size=64, endpoint=True).astype(np.int32)
    return make_workload("decode_b64_n4k-128k_k2048_h128_paged64_fp8", lens, [1] * 64, H=128, K=2048,
                         page_size=64, permute=True, seed=seed)


def prefill(T: int = 16384, seed: int = 0, H: int = 128, K: int = 2048) -> Workload:
    """Prefill of one sequence of T tokens, causal: query t sees 0..t and
    keeps the top min(K, t+1).  Identity page table with 64-row pages."""
    return make_workload(f"prefill_t{T}_k{K}_h{H}", [T], [T], H=H, K=K, page_size=64, permute=False, seed=seed)
