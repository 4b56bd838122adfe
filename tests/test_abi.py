"""CPU checks of the boundary: the library builds for sm_103a, loads without a
GPU, and exports every function include/dsa.h declares; host-side argument
validation rejects bad calls before any launch."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    import indexer_top_sparse_gb300 as d
    from indexer_top_sparse_gb300 import _build
    _build.build()
    return d.load()


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("dsa_index_topk", "dsa_sparse_mla", "dsa_topk_from_scores", "dsa_index_scores", "dsa_get_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from indexer_top_sparse_gb300 import _build, _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dsa_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    assert set(_lib.EXPORTS) == set(declared_functions())
    for n in declared_functions():
        assert hasattr(lib, n)


def test_library_is_built_for_sm103a_only():
    from indexer_top_sparse_gb300 import _build
    flags = " ".join(_build.ARCH)
    assert "compute_103a" in flags and "sm_103a" in flags


def test_status_strings_and_tuning(lib):
    assert lib.dsa_status_string(0) == b"ok"
    assert lib.dsa_status_string(6) == b"device wait timed out"
    assert lib.dsa_set_tuning(b"indexer_cluster", 0) == 0
    assert lib.dsa_set_tuning(b"no_such_knob", 1) == -1


def test_host_validation_rejects_bad_arguments(lib):
    # null pointers and bad sizes fail on the host, before any CUDA call
    import ctypes
    rc = lib.dsa_index_topk(None, None, None, None, None, 1, None, 1, None, None, 1, 1, 1, 64, 0, None, None, 0, None)
    assert rc == 1
    rc = lib.dsa_sparse_mla(None, None, None, None, 1, None, 1, None, None, None, 1, 1, 17, 1, ctypes.c_float(1.0),
                            64, 0, None, None, None, 0, None)
    assert rc == 1
    rc = lib.dsa_topk_from_scores(None, 1, None, 1, 0, None, None, 0, None)
    assert rc == 1
    assert lib.dsa_workspace_init(None, 0, None) == 1
    assert lib.dsa_index_topk_workspace_size(1, 1, 1, 1, 64) >= 16
    assert lib.dsa_sparse_mla_workspace_size(1, 128, 2048) >= 16


def test_flat_indexer_is_chosen_for_large_decode_batches(lib):
    # the workspace size reports whether the flat bf16 indexer applies: one
    # query row per sequence and at least 3 * 2^20 positions in all, rows of
    # at most 49152 positions
    assert lib.dsa_index_topk_workspace_size(96, 96, 2048, 512, 64) > 256       # 96 x 32768
    assert lib.dsa_index_topk_workspace_size(32, 32, 2048, 512, 64) == 256      # 32 x 32768
    assert lib.dsa_index_topk_workspace_size(1, 4096, 2048, 512, 64) == 256     # a prefill: rows share a sequence
    assert lib.dsa_index_topk_workspace_size(96, 96, 2048, 1024, 64) == 256     # rows past the staging limit
