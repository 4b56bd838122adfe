"""GB300-native (sm_103a) DSA "score, select, sparse read" path.

    dsa_index_topk   fused lightweight indexer + Top-K over a paged index-key cache
    dsa_sparse_mla   sparse MLA attention over the selected latent KV rows

Both run in hand-written CUDA kernels of libdsa.so (C ABI: include/dsa.h);
this package only marshals torch tensors into that ABI.  There is no CPU
fallback.
"""
from ._lib import (DSAError, Workspace, dsa_cache_append, dsa_index_scores, dsa_index_topk, dsa_quant_fp8_rows,
                   dsa_quant_fp8_tiles,
                   dsa_quant_mxfp8,
                   dsa_sparse_mla, dsa_topk_from_scores, index_topk_workspace_size, library_path, load, set_tuning,
                   sparse_mla_workspace_size)

__all__ = ["DSAError", "Workspace", "dsa_index_topk", "dsa_index_scores", "dsa_topk_from_scores", "dsa_sparse_mla",
           "index_topk_workspace_size", "sparse_mla_workspace_size", "load", "library_path", "set_tuning",
           "dsa_quant_mxfp8", "dsa_quant_fp8_rows", "dsa_quant_fp8_tiles", "dsa_cache_append"]
