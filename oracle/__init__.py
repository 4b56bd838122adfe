"""CPU oracle for the DSA "score, select, sparse read" path.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the benchmark's CPU-baseline leg, never by the library.  It shares no
code with the CUDA path.  The arithmetic lives in ``dsa_oracle.c`` (plain C,
single-threaded, fp64 accumulation); this module only compiles it with gcc and
marshals numpy arrays through ctypes.

What each function computes and which passage of the pages it follows is
stated in ``dsa_oracle.c``.  Every function is pinned by a CPU test
(tests/test_oracle_*.py) against brute force, closed forms, library routines
on special cases or invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None

IDX_BF16, IDX_MXFP8 = 0, 1
KV_BF16, KV_FP8_ROWSCALE, KV_FP8_TILE128 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into a shared library (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = f64
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f64.restype = f64
            lib.orc_f64_to_e4m3_sat.argtypes = [f64]
            lib.orc_f64_to_e4m3_sat.restype = ctypes.c_uint8
            lib.orc_e8m0_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e8m0_to_f64.restype = f64
            lib.orc_quant_mxfp8.argtypes = [P, i64, P, P]
            lib.orc_quant_mxfp8.restype = None
            lib.orc_quant_fp8_rows.argtypes = [P, i64, P, P, P]
            lib.orc_quant_fp8_rows.restype = None
            lib.orc_quant_fp8_tiles.argtypes = [P, i64, P, P, P]
            lib.orc_quant_fp8_tiles.restype = None
            lib.orc_cache_append.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i64, ctypes.c_int, P, P,
                                             ctypes.c_int, P, P, P]
            lib.orc_cache_append.restype = ctypes.c_int
            lib.orc_index_scores_row.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, i64, P,
                                                 i32, i64, P]
            lib.orc_index_scores_row.restype = ctypes.c_int
            lib.orc_topk_row.argtypes = [P, i64, i32, P]
            lib.orc_topk_row.restype = ctypes.c_int
            lib.orc_topk_rows.argtypes = [P, i64, P, i32, i32, P]
            lib.orc_topk_rows.restype = ctypes.c_int
            lib.orc_index_topk.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, i64, P, i32, P,
                                           P, i32, i32, i32, i32, P, i32, P, P, i64]
            lib.orc_index_topk.restype = ctypes.c_int
            lib.orc_sparse_mla_row.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P,
                                               i64, P, i32, P, i32, f64, P, P]
            lib.orc_sparse_mla_row.restype = ctypes.c_int
            lib.orc_sparse_mla.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, i64,
                                           P, i32, P, i32, i32, P, i32, f64, i32, P, i32, P, P]
            lib.orc_sparse_mla.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codecs

def bf16_to_f64(bits: int) -> float:
    return _load().orc_bf16_to_f64(int(bits))


def e4m3_to_f64(code: int) -> float:
    return _load().orc_e4m3_to_f64(int(code))


def f64_to_e4m3(x: float) -> int:
    return int(_load().orc_f64_to_e4m3_sat(float(x)))


def e8m0_to_f64(code: int) -> float:
    return _load().orc_e8m0_to_f64(int(code))


def quant_mxfp8(x_bf16_bits: np.ndarray):
    """MXFP8 quantisation of a bf16 array (bits as uint16), blocks of 32 along
    the flattened order.  Returns (e4m3 codes uint8, e8m0 scale bytes uint8)."""
    x = _c(x_bf16_bits, np.uint16)
    n = x.size
    if n % 32:
        raise ValueError("size must be a multiple of 32")
    q = np.empty(x.shape, np.uint8)
    e = np.empty(x.shape[:-1] + (x.shape[-1] // 32,), np.uint8)
    _load().orc_quant_mxfp8(_p(x), n, _p(q), _p(e))
    return q, e


def quant_fp8_rows(kv_bf16_bits: np.ndarray):
    """FP8 row quantisation of [..., 576] bf16 latent rows.  Returns
    (nope e4m3 [..., 512] uint8, rope bf16 bits [..., 64] uint16, scale fp32 [...])."""
    kv = _c(kv_bf16_bits, np.uint16)
    if kv.shape[-1] != 576:
        raise ValueError("last dim must be 576")
    rows = kv.size // 576
    nope = np.empty(kv.shape[:-1] + (512,), np.uint8)
    rope = np.empty(kv.shape[:-1] + (64,), np.uint16)
    scale = np.empty(kv.shape[:-1], np.float32)
    _load().orc_quant_fp8_rows(_p(kv), rows, _p(nope), _p(rope), _p(scale))
    return nope, rope, scale


def quant_fp8_tiles(kv_bf16_bits: np.ndarray):
    """FP8 tile quantisation of [..., 576] bf16 latent rows, one scale per
    128 latent dims.  Returns (nope e4m3 [..., 512] uint8, rope bf16 bits
    [..., 64] uint16, scale fp32 [..., 4])."""
    kv = _c(kv_bf16_bits, np.uint16)
    if kv.shape[-1] != 576:
        raise ValueError("last dim must be 576")
    rows = kv.size // 576
    nope = np.empty(kv.shape[:-1] + (512,), np.uint8)
    rope = np.empty(kv.shape[:-1] + (64,), np.uint16)
    scale = np.empty(kv.shape[:-1] + (4,), np.float32)
    _load().orc_quant_fp8_tiles(_p(kv), rows, _p(nope), _p(rope), _p(scale))
    return nope, rope, scale


def _writable(a, dtype, name):
    if a is None:
        return None
    if a.dtype != dtype or not a.flags.c_contiguous or not a.flags.writeable:
        raise ValueError(f"{name} must be a writable C-contiguous {np.dtype(dtype).name} array")
    return a


def cache_append(page_table, seq_lens, cu_q, page_size, *, k_new=None, kv_new=None, idx_dtype=IDX_BF16,
                 k_cache=None, k_scale=None, kv_dtype=KV_BF16, kv_cache=None, kv_rope=None, kv_scale=None,
                 num_pages=None):
    """Write new tokens' index keys (k_new [T, 128] bf16 bits) and latent rows
    (kv_new [T, 576] bf16 bits) into the paged caches, in place, quantising to
    the caches' formats.  Token t of sequence b is at position
    seq_lens[b] - (cu_q[b+1] - cu_q[b]) + (t - cu_q[b]).  Cache arrays:
    k_cache [pages, page_size, 128] (uint16 bf16 bits, or uint8 e4m3 with
    k_scale [..., 4] uint8); kv_cache [pages, page_size, 576] uint16, or
    [..., 512] uint8 with kv_rope [..., 64] uint16 and kv_scale [...] or
    [..., 4] float32.  Returns the C status (0, or -1 if a token's page id was
    out of range)."""
    pt = _c(page_table, np.int32)
    B, maxp = pt.shape
    cq = _c(cu_q, np.int32)
    T = int(cq[-1])
    kn = None if k_new is None else _c(k_new, np.uint16)
    vn = None if kv_new is None else _c(kv_new, np.uint16)
    kc = _writable(k_cache, np.uint16 if idx_dtype == IDX_BF16 else np.uint8, "k_cache")
    ks = _writable(k_scale, np.uint8, "k_scale")
    vc = _writable(kv_cache, np.uint16 if kv_dtype == KV_BF16 else np.uint8, "kv_cache")
    vr = _writable(kv_rope, np.uint16, "kv_rope")
    vs = _writable(kv_scale, np.float32, "kv_scale")
    if num_pages is None:
        num_pages = (kc if kc is not None else vc).shape[0]
    rc = _load().orc_cache_append(_p(kn), _p(vn), _p(pt), maxp, _p(_c(seq_lens, np.int32)), _p(cq), B, T,
                                  page_size, num_pages, idx_dtype, _p(kc), _p(ks), kv_dtype, _p(vc), _p(vr), _p(vs))
    if rc == -3:
        raise RuntimeError("orc_cache_append: token outside cu_q")
    return rc


# ---------------------------------------------------------------- indexer / top-K

def topk_rows(scores: np.ndarray, lens: np.ndarray, K: int) -> np.ndarray:
    """Top-K of each score row (higher first, ties by lower position), valid
    entries 0..lens[r]-1.  Returns int32 [R, K], ascending, -1 padded."""
    s = _c(scores, np.float32)
    R, ld = s.shape
    ln = _c(lens, np.int32)
    out = np.empty((R, K), np.int32)
    rc = _load().orc_topk_rows(_p(s), ld, _p(ln), R, K, _p(out))
    if rc != 0:
        raise RuntimeError(f"orc_topk_rows failed: {rc}")
    return out


def index_scores_row(q, w, k_cache, page_row, page_size, n_pos, *, dtype=IDX_BF16, q_scale=None, k_scale=None,
                     num_pages=None):
    """Scores of one query ([H_I, d_I] q, [H_I] w) against positions 0..n_pos-1."""
    q = _c(q, np.uint16 if dtype == IDX_BF16 else np.uint8)
    H_I, d_I = q.shape
    w = _c(w, np.float32)
    kc = _c(k_cache, np.uint16 if dtype == IDX_BF16 else np.uint8)
    ks = _c(k_scale, np.uint8)
    qs = _c(q_scale, np.uint8)
    pr = _c(page_row, np.int32)
    if num_pages is None:
        num_pages = kc.size // (page_size * d_I)
    out = np.empty(n_pos, np.float32)
    rc = _load().orc_index_scores_row(dtype, H_I, d_I, _p(q), _p(qs), _p(w), _p(kc), _p(ks), num_pages, _p(pr),
                                      page_size, n_pos, _p(out))
    if rc != 0:
        raise RuntimeError(f"orc_index_scores_row failed: {rc}")
    return out


def index_topk(q_idx, head_w, k_cache, page_table, seq_lens, cu_q, K, page_size, *, dtype=IDX_BF16,
               q_scale=None, k_scale=None, rows=None, want_scores=False, ld_scores=None):
    """Fused indexer + Top-K for query rows `rows` (None: all T).
    q_idx [T, H_I, d_I]; head_w [T, H_I]; k_cache [pages, page_size, d_I];
    page_table [B, max_pages]; seq_lens [B]; cu_q [B+1].
    Returns indices [n_rows, K] (and scores [n_rows, ld_scores] if asked)."""
    q = _c(q_idx, np.uint16 if dtype == IDX_BF16 else np.uint8)
    T, H_I, d_I = q.shape
    w = _c(head_w, np.float32)
    kc = _c(k_cache, np.uint16 if dtype == IDX_BF16 else np.uint8)
    num_pages = kc.size // (page_size * d_I)
    pt = _c(page_table, np.int32)
    B, maxp = pt.shape
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    rw = _c(rows, np.int32)
    n_rows = T if rw is None else rw.size
    idx = np.empty((n_rows, K), np.int32)
    sc = None
    if want_scores:
        ld_scores = int(ld_scores if ld_scores is not None else int(sl.max()))
        sc = np.full((n_rows, ld_scores), np.nan, np.float32)
    rc = _load().orc_index_topk(dtype, H_I, d_I, _p(q), _p(_c(q_scale, np.uint8)), _p(w), _p(kc),
                                _p(_c(k_scale, np.uint8)), num_pages, _p(pt), maxp, _p(sl), _p(cq), B, T, K,
                                page_size, _p(rw), n_rows, _p(idx), _p(sc), ld_scores or 0)
    if rc != 0:
        raise RuntimeError(f"orc_index_topk failed: {rc}")
    return (idx, sc) if want_scores else idx


# ---------------------------------------------------------------- sparse MLA

def sparse_mla(q, kv_cache, page_table, cu_q, indices, scale, page_size, *, dtype=KV_BF16, kv_rope=None,
               kv_scale=None, rows=None, D=None, Dv=None, num_pages=None):
    """Sparse MLA attention for query rows `rows` (None: all T).
    q [T, H, D] bf16 bits; kv_cache [pages, page_size, D] bf16 bits (or
    [pages, page_size, 512] e4m3 with kv_rope [..., 64] bf16 and kv_scale
    [pages, page_size] fp32, or [pages, page_size, 4] fp32 for KV_FP8_TILE128);
    indices [T, K] logical positions, -1 skipped.
    Returns (out [n_rows, H, Dv] fp32, lse [n_rows, H] fp32)."""
    q = _c(q, np.uint16)
    T, H, Dq = q.shape
    D = Dq if D is None else D
    if Dv is None:
        Dv = 512 if D == 576 else D
    kv = _c(kv_cache, np.uint16 if dtype == KV_BF16 else np.uint8)
    if num_pages is None:
        num_pages = kv.shape[0]
    pt = _c(page_table, np.int32)
    B, maxp = pt.shape
    cq = _c(cu_q, np.int32)
    ix = _c(indices, np.int32)
    K = ix.shape[1]
    rw = _c(rows, np.int32)
    n_rows = T if rw is None else rw.size
    out = np.empty((n_rows, H, Dv), np.float32)
    lse = np.empty((n_rows, H), np.float32)
    rc = _load().orc_sparse_mla(dtype, H, D, Dv, _p(q), _p(kv), _p(_c(kv_rope, np.uint16)),
                                _p(_c(kv_scale, np.float32)), num_pages, _p(pt), maxp, _p(cq), B, T, _p(ix), K,
                                float(scale), page_size, _p(rw), n_rows, _p(out), _p(lse))
    if rc != 0:
        raise RuntimeError(f"orc_sparse_mla failed: {rc}")
    return out, lse
