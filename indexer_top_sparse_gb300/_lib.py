"""ctypes binding of libdsa.so (the C ABI in include/dsa.h).

Argument marshalling only: torch supplies device memory and the current
stream; every step of the path runs in the library's CUDA kernels.  There is
no CPU fallback: if the library is missing or CUDA is unavailable, the calls
raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

_lock = threading.Lock()
_lib = None

DSA_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "page id out of range",
          5: "selected index out of range", 6: "device wait timed out"}
IDX_DTYPES = {"bf16": 0, "mxfp8": 1, "mxfp8_qbf16": 2}
KV_DTYPES = {"bf16": 0, "fp8_rowscale": 1, "fp8_tile128": 2}

# Every symbol include/dsa.h declares.
EXPORTS = ("dsa_status_string", "dsa_set_tuning", "dsa_index_topk_workspace_size", "dsa_sparse_mla_workspace_size",
           "dsa_workspace_init", "dsa_get_error", "dsa_workspace_set_wait_limit", "dsa_index_topk", "dsa_index_scores", "dsa_topk_from_scores",
           "dsa_sparse_mla", "dsa_sparse_mla_static", "dsa_sparse_mla_static_get_error", "dsa_quant_mxfp8",
           "dsa_quant_fp8_rows",
           "dsa_quant_fp8_tiles", "dsa_cache_append")


class DSAError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libdsa.so (building it first if it is missing and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise FileNotFoundError(f"{path} is not built; run __graft_entry__.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        c_int = ctypes.c_int
        lib.dsa_status_string.argtypes = [c_int]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_set_tuning.argtypes = [ctypes.c_char_p, c_int]
        lib.dsa_set_tuning.restype = c_int
        lib.dsa_index_topk_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.dsa_index_topk_workspace_size.restype = sz
        lib.dsa_sparse_mla_workspace_size.argtypes = [i32, i32, i32]
        lib.dsa_sparse_mla_workspace_size.restype = sz
        lib.dsa_workspace_init.argtypes = [P, sz, P]
        lib.dsa_workspace_init.restype = c_int
        lib.dsa_get_error.argtypes = [P, P]
        lib.dsa_get_error.restype = c_int
        lib.dsa_workspace_set_wait_limit.argtypes = [P, ctypes.c_uint32, P]
        lib.dsa_workspace_set_wait_limit.restype = c_int
        idx_args = [P, P, P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, c_int, P]
        lib.dsa_index_topk.argtypes = idx_args + [P, sz, P]
        lib.dsa_index_topk.restype = c_int
        lib.dsa_index_scores.argtypes = idx_args + [P, i64, P, sz, P]
        lib.dsa_index_scores.restype = c_int
        lib.dsa_topk_from_scores.argtypes = [P, i64, P, i32, i32, P, P, sz, P]
        lib.dsa_topk_from_scores.restype = c_int
        lib.dsa_sparse_mla.argtypes = [P, P, P, P, i64, P, i32, P, P, P, i32, i32, i32, i32, ctypes.c_float, i32,
                                       c_int, P, P, P, sz, P]
        lib.dsa_sparse_mla.restype = c_int
        lib.dsa_sparse_mla_static.argtypes = [P, P, P, P, i64, P, i32, P, P, P, i32, i32, i32, i32, ctypes.c_float,
                                              i32, c_int, P, P, P]
        lib.dsa_sparse_mla_static.restype = c_int
        lib.dsa_sparse_mla_static_get_error.argtypes = [P]
        lib.dsa_sparse_mla_static_get_error.restype = c_int
        lib.dsa_quant_mxfp8.argtypes = [P, i64, P, P, P]
        lib.dsa_quant_mxfp8.restype = c_int
        lib.dsa_quant_fp8_rows.argtypes = [P, i64, P, P, P, P]
        lib.dsa_quant_fp8_rows.restype = c_int
        lib.dsa_quant_fp8_tiles.argtypes = [P, i64, P, P, P, P]
        lib.dsa_quant_fp8_tiles.restype = c_int
        lib.dsa_cache_append.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i64, c_int, P, P, c_int, P, P, P, P, sz, P]
        lib.dsa_cache_append.restype = c_int
        _lib = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, code):
    if code != DSA_OK:
        raise DSAError(fn, code)


def _need(t, name, dtype, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def set_tuning(name: str, value: int) -> None:
    if load().dsa_set_tuning(name.encode(), int(value)) != 0:
        raise KeyError(name)


class Workspace:
    """Device workspace with its error word initialised."""

    def __init__(self, nbytes: int, device=None, stream=None):
        self.nbytes = int(max(nbytes, 256))
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _check("dsa_workspace_init", load().dsa_workspace_init(_ptr(self.buf), self.nbytes, _stream(stream)))

    def ensure(self, nbytes: int, stream=None):
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.buf.device, stream)
        return self

    def set_wait_limit(self, microseconds: int, stream=None) -> None:
        """Test hook: kernels using this workspace give up a pipeline wait
        after `microseconds` (0: the 200 ms default) and report a timeout."""
        _check("dsa_workspace_set_wait_limit",
               load().dsa_workspace_set_wait_limit(_ptr(self.buf), int(microseconds), _stream(stream)))

    def check(self, stream=None) -> None:
        """Synchronise and raise if a kernel recorded a device-side error."""
        _check("device", load().dsa_get_error(_ptr(self.buf), _stream(stream)))


def index_topk_workspace_size(B, T, K, max_pages, page_size) -> int:
    return int(load().dsa_index_topk_workspace_size(B, T, K, max_pages, page_size))


def sparse_mla_workspace_size(T, H, K) -> int:
    return int(load().dsa_sparse_mla_workspace_size(T, H, K))


def _index_call(scores_ld, q_idx, head_w, k_idx_cache, page_table, seq_lens, cu_q, K, indices, scores,
                workspace, q_idx_scale, k_idx_scale, dtype, stream):
    lib = load()
    dt = IDX_DTYPES[dtype]
    elt = torch.uint8 if dt == 1 else torch.bfloat16
    _need(q_idx, "q_idx", elt, 3)
    dev = q_idx.device
    T = q_idx.shape[0]
    if tuple(q_idx.shape[1:]) != (64, 128):
        raise ValueError("q_idx must be [T, 64, 128]")
    _need(head_w, "head_w", torch.float32, 2, dev)
    _need(k_idx_cache, "k_idx_cache", torch.bfloat16 if dt == 0 else torch.uint8, 3, dev)
    if k_idx_cache.shape[2] != 128:
        raise ValueError("k_idx_cache must be [pages, page_size, 128]")
    _need(page_table, "page_table", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    _need(cu_q, "cu_q", torch.int32, 1, dev)
    B = seq_lens.shape[0]
    if cu_q.shape[0] != B + 1 or page_table.shape[0] != B:
        raise ValueError("seq_lens [B], cu_q [B+1], page_table [B, max_pages] must agree")
    P, ps = k_idx_cache.shape[0], k_idx_cache.shape[1]
    maxp = page_table.shape[1]
    if dt == 1:
        _need(q_idx_scale, "q_idx_scale", torch.uint8, 3, dev)
        _need(k_idx_scale, "k_idx_scale", torch.uint8, 3, dev)
        if tuple(q_idx_scale.shape) != (T, 64, 4) or tuple(k_idx_scale.shape) != (P, ps, 4):
            raise ValueError("MXFP8 scales must be q_idx_scale [T, 64, 4] and k_idx_scale [pages, page_size, 4]")
    elif dt == 2:
        if q_idx_scale is not None:
            raise ValueError("dtype='mxfp8_qbf16' takes q_idx in bf16 and no q_idx_scale")
        _need(k_idx_scale, "k_idx_scale", torch.uint8, 3, dev)
        if tuple(k_idx_scale.shape) != (P, ps, 4):
            raise ValueError("k_idx_scale must be [pages, page_size, 4]")
    elif q_idx_scale is not None or k_idx_scale is not None:
        raise ValueError("q_idx_scale / k_idx_scale are for the MXFP8 dtypes only")
    if indices is None:
        indices = torch.empty((T, K), dtype=torch.int32, device=dev)
    _need(indices, "indices", torch.int32, 2, dev)
    if workspace is None:
        workspace = Workspace(index_topk_workspace_size(B, T, K, maxp, ps), dev, stream)
    common = [_ptr(q_idx), _ptr(q_idx_scale), _ptr(head_w), _ptr(k_idx_cache), _ptr(k_idx_scale), P,
              _ptr(page_table), maxp, _ptr(seq_lens), _ptr(cu_q), B, T, K, ps, dt, _ptr(indices)]
    if scores is None:
        _check("dsa_index_topk", lib.dsa_index_topk(*common, _ptr(workspace.buf), workspace.nbytes, _stream(stream)))
        return indices
    _need(scores, "scores", torch.float32, 2, dev)
    _check("dsa_index_scores", lib.dsa_index_scores(*common, _ptr(scores), scores.shape[1], _ptr(workspace.buf),
                                                    workspace.nbytes, _stream(stream)))
    return indices, scores


def dsa_index_topk(q_idx, head_w, k_idx_cache, page_table, seq_lens, cu_q, K, *, indices=None, workspace=None,
                   q_idx_scale=None, k_idx_scale=None, dtype="bf16", stream=None):
    """Fused indexer + Top-K (see include/dsa.h).  Returns indices [T, K] int32."""
    return _index_call(None, q_idx, head_w, k_idx_cache, page_table, seq_lens, cu_q, K, indices, None, workspace,
                       q_idx_scale, k_idx_scale, dtype, stream)


def dsa_index_scores(q_idx, head_w, k_idx_cache, page_table, seq_lens, cu_q, K, scores, *, indices=None,
                     workspace=None, q_idx_scale=None, k_idx_scale=None, dtype="bf16", stream=None):
    """Test hook: dsa_index_topk that also writes fp32 scores into `scores` [T, ld]."""
    return _index_call(scores.shape[1], q_idx, head_w, k_idx_cache, page_table, seq_lens, cu_q, K, indices, scores,
                       workspace, q_idx_scale, k_idx_scale, dtype, stream)


def dsa_topk_from_scores(scores, lens, K, *, out=None, workspace=None, stream=None):
    """Top-K of fp32 score rows [R, ld] valid on 0..lens[r]-1.  Returns [R, K] int32."""
    lib = load()
    _need(scores, "scores", torch.float32, 2)
    dev = scores.device
    _need(lens, "lens", torch.int32, 1, dev)
    R, ld = scores.shape
    if out is None:
        out = torch.empty((R, K), dtype=torch.int32, device=dev)
    _need(out, "out", torch.int32, 2, dev)
    if workspace is None:
        workspace = Workspace(256, dev, stream)
    _check("dsa_topk_from_scores", lib.dsa_topk_from_scores(_ptr(scores), ld, _ptr(lens), R, K, _ptr(out),
                                                            _ptr(workspace.buf), workspace.nbytes, _stream(stream)))
    return out


def dsa_sparse_mla(q, kv_cache, page_table, seq_lens, cu_q, indices, scale, *, out=None, lse=None, workspace=None,
                   kv_rope=None, kv_scale=None, dtype="bf16", stream=None):
    """Sparse MLA attention over the selected rows (see include/dsa.h).
    Returns out [T, H, 512] bf16 (and fills lse [T, H] fp32 if given)."""
    lib = load()
    dt = KV_DTYPES[dtype]
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    T, H, D = q.shape
    if D != 576:
        raise ValueError("q must be [T, H, 576]")
    _need(kv_cache, "kv_cache", torch.bfloat16 if dt == 0 else torch.uint8, 3, dev)
    if dt in (1, 2):
        _need(kv_rope, "kv_rope", torch.bfloat16, 3, dev)
        _need(kv_scale, "kv_scale", torch.float32, 2 if dt == 1 else 3, dev)
        pp, pps = kv_cache.shape[0], kv_cache.shape[1]
        sshape = (pp, pps) if dt == 1 else (pp, pps, 4)
        if kv_cache.shape[2] != 512 or tuple(kv_rope.shape) != (pp, pps, 64) or tuple(kv_scale.shape) != sshape:
            raise ValueError("FP8 cache: kv_cache [pages, page_size, 512] e4m3, kv_rope [.., 64] bf16, kv_scale "
                             "[pages, page_size] (fp8_rowscale) or [pages, page_size, 4] (fp8_tile128) fp32")
    elif kv_rope is not None or kv_scale is not None:
        raise ValueError("kv_rope / kv_scale are for the FP8 dtypes only")
    elif kv_cache.shape[2] != 576:
        raise ValueError("kv_cache must be [pages, page_size, 576] bf16")
    _need(page_table, "page_table", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    _need(cu_q, "cu_q", torch.int32, 1, dev)
    _need(indices, "indices", torch.int32, 2, dev)
    B = seq_lens.shape[0]
    K = indices.shape[1]
    P, ps = kv_cache.shape[0], kv_cache.shape[1]
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, dev)
    if workspace is None:
        workspace = Workspace(sparse_mla_workspace_size(T, H, K), dev, stream)
    _check("dsa_sparse_mla", lib.dsa_sparse_mla(_ptr(q), _ptr(kv_cache), _ptr(kv_rope), _ptr(kv_scale), P,
                                                _ptr(page_table), page_table.shape[1], _ptr(seq_lens), _ptr(cu_q),
                                                _ptr(indices), B, T, H, K, float(scale), ps, dt, _ptr(out),
                                                _ptr(lse), _ptr(workspace.buf), workspace.nbytes, _stream(stream)))
    return out


def dsa_cache_append(page_table, seq_lens, cu_q, *, k_new=None, kv_new=None, k_cache=None, k_scale=None,
                     kv_cache=None, kv_rope=None, kv_scale=None, idx_dtype="bf16", kv_dtype="bf16", workspace=None,
                     stream=None):
    """Write new tokens' index keys (k_new [T, 128] bf16) and latent rows
    (kv_new [T, 576] bf16) into their page slots, quantised to the caches'
    formats (see include/dsa.h).  The caches are updated in place."""
    lib = load()
    it, kt = IDX_DTYPES[idx_dtype], KV_DTYPES[kv_dtype]
    _need(page_table, "page_table", torch.int32, 2)
    dev = page_table.device
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    _need(cu_q, "cu_q", torch.int32, 1, dev)
    B = seq_lens.shape[0]
    if cu_q.shape[0] != B + 1:
        raise ValueError("cu_q must have B + 1 entries")
    T, ps, P = None, None, None
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16, 2, dev)
        _need(k_cache, "k_cache", torch.bfloat16 if it == 0 else torch.uint8, 3, dev)
        if k_new.shape[1] != 128 or k_cache.shape[2] != 128:
            raise ValueError("k_new [T, 128] and k_cache [pages, page_size, 128]")
        if it == 1:
            _need(k_scale, "k_scale", torch.uint8, 3, dev)
            if tuple(k_scale.shape) != tuple(k_cache.shape[:2]) + (4,):
                raise ValueError("k_scale must be [pages, page_size, 4] uint8")
        T, P, ps = k_new.shape[0], k_cache.shape[0], k_cache.shape[1]
    if kv_new is not None:
        _need(kv_new, "kv_new", torch.bfloat16, 2, dev)
        _need(kv_cache, "kv_cache", torch.bfloat16 if kt == 0 else torch.uint8, 3, dev)
        if kv_new.shape[1] != 576 or kv_cache.shape[2] != (576 if kt == 0 else 512):
            raise ValueError("kv_new [T, 576]; kv_cache [pages, page_size, 576] bf16 or [.., 512] e4m3")
        if kt != 0:
            _need(kv_rope, "kv_rope", torch.bfloat16, 3, dev)
            _need(kv_scale, "kv_scale", torch.float32, 2 if kt == 1 else 3, dev)
            sshape = tuple(kv_cache.shape[:2]) + (() if kt == 1 else (4,))
            if tuple(kv_rope.shape) != tuple(kv_cache.shape[:2]) + (64,) or tuple(kv_scale.shape) != sshape:
                raise ValueError("kv_rope [pages, page_size, 64] bf16 and kv_scale [pages, page_size(, 4)] fp32")
        if T is not None and (kv_new.shape[0] != T or kv_cache.shape[0] != P or kv_cache.shape[1] != ps):
            raise ValueError("k_new / kv_new and the two caches must agree on T, pages and page size")
        T, P, ps = kv_new.shape[0], kv_cache.shape[0], kv_cache.shape[1]
    if T is None:
        return
    if workspace is None:
        workspace = Workspace(256, dev, stream)
    _check("dsa_cache_append", lib.dsa_cache_append(_ptr(k_new), _ptr(kv_new), _ptr(page_table), page_table.shape[1],
                                                    _ptr(seq_lens), _ptr(cu_q), B, T, ps, P, it, _ptr(k_cache),
                                                    _ptr(k_scale), kt, _ptr(kv_cache), _ptr(kv_rope), _ptr(kv_scale),
                                                    _ptr(workspace.buf), workspace.nbytes, _stream(stream)))


def dsa_quant_mxfp8(x, *, q=None, scales=None, stream=None):
    """MXFP8 quantisation of a bf16 tensor (last dim a multiple of 32).
    Returns (e4m3 codes uint8, same shape; e8m0 scale bytes uint8, last dim / 32)."""
    lib = load()
    _need(x, "x", torch.bfloat16)
    if x.shape[-1] % 32:
        raise ValueError("last dim must be a multiple of 32")
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (x.shape[-1] // 32,), dtype=torch.uint8, device=x.device)
    _need(q, "q", torch.uint8, None, x.device)
    _need(scales, "scales", torch.uint8, None, x.device)
    if q.numel() != x.numel() or scales.numel() != x.numel() // 32:
        raise ValueError("q must hold one byte per element of x and scales one byte per 32 elements")
    _check("dsa_quant_mxfp8", lib.dsa_quant_mxfp8(_ptr(x), x.numel(), _ptr(q), _ptr(scales), _stream(stream)))
    return q, scales


def dsa_quant_fp8_rows(kv, *, nope=None, rope=None, scale=None, stream=None):
    """FP8 row quantisation of [..., 576] bf16 latent rows.  Returns
    (nope e4m3 [..., 512] uint8, rope [..., 64] bf16, scale [...] fp32)."""
    return _quant_fp8(kv, 1, nope, rope, scale, stream)


def dsa_quant_fp8_tiles(kv, *, nope=None, rope=None, scale=None, stream=None):
    """FP8 quantisation of [..., 576] bf16 latent rows with one scale per 128
    latent dims.  Returns (nope e4m3 [..., 512] uint8, rope [..., 64] bf16,
    scale [..., 4] fp32)."""
    return _quant_fp8(kv, 4, nope, rope, scale, stream)


def _quant_fp8(kv, tiles, nope, rope, scale, stream):
    lib = load()
    _need(kv, "kv", torch.bfloat16)
    if kv.shape[-1] != 576:
        raise ValueError("last dim must be 576")
    lead = kv.shape[:-1]
    rows = kv.numel() // 576
    nope = torch.empty(lead + (512,), dtype=torch.uint8, device=kv.device) if nope is None else nope
    rope = torch.empty(lead + (64,), dtype=torch.bfloat16, device=kv.device) if rope is None else rope
    if scale is None:
        scale = torch.empty(lead if tiles == 1 else lead + (tiles,), dtype=torch.float32, device=kv.device)
    _need(nope, "nope", torch.uint8, None, kv.device)
    _need(rope, "rope", torch.bfloat16, None, kv.device)
    _need(scale, "scale", torch.float32, None, kv.device)
    if nope.numel() != rows * 512 or rope.numel() != rows * 64 or scale.numel() != rows * tiles:
        raise ValueError(f"nope, rope and scale must hold rows x 512, rows x 64 and rows x {tiles} elements")
    fn = "dsa_quant_fp8_rows" if tiles == 1 else "dsa_quant_fp8_tiles"
    _check(fn, getattr(lib, fn)(_ptr(kv), rows, _ptr(nope), _ptr(rope), _ptr(scale), _stream(stream)))
    return nope, rope, scale
