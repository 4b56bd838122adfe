"""The allocation-free sparse MLA entry point (dsa_sparse_mla_static).

Some callers cannot allocate device memory around the attention call -- a
serving step that must not take the synchronisation an allocation can imply,
or a plug-in whose host framework owns every device buffer.  For them the
library offers a variant whose split-K scratch lives in a fixed array inside
the library.  This test calls that variant through the C ABI and checks it
against the workspace-taking dsa_sparse_mla on the same inputs, twice in a row
(the second call finds the first call's leftovers in the shared array).  The
file sorts last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

from _util import dev, to_device
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu


def _indices(rng, wl):
    pos = wl.query_pos()
    idx = np.full((wl.T, wl.K), -1, np.int32)
    for t in range(wl.T):
        n = int(pos[t]) + 1
        m = min(wl.K, n)
        idx[t, :m] = np.sort(rng.choice(n, m, replace=False))
    return idx


def _call_static(lib, t, idx_d, wl, out, lse, kv=None, rope=None, scale=None, dtype=0):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = ctypes.c_void_p
    kv = t["kv"] if kv is None else kv
    rc = lib.dsa_sparse_mla_static(P(t["q"].data_ptr()), P(kv.data_ptr()),
                                   None if rope is None else P(rope.data_ptr()),
                                   None if scale is None else P(scale.data_ptr()), kv.shape[0],
                                   P(t["page_table"].data_ptr()), t["page_table"].shape[1],
                                   P(t["seq_lens"].data_ptr()), P(t["cu_q"].data_ptr()), P(idx_d.data_ptr()), wl.B,
                                   wl.T, wl.H, wl.K, ctypes.c_float(wl.scale), wl.page_size, dtype,
                                   P(out.data_ptr()), P(lse.data_ptr()), stream)
    assert rc == 0, f"dsa_sparse_mla_static returned {rc}"


def test_static_scratch_matches_workspace_version_twice():
    import indexer_top_sparse_gb300 as d
    lib = d.load()
    for call, seed in enumerate([1, 2]):
        rng = np.random.default_rng(seed)
        # few query rows and many keys: the split-K path (and its scratch) is used
        wl = make_workload(f"static{seed}", [3000 + seed, 900, 1500], [1, 1, 1], H=64, K=1000, page_size=64,
                           seed=seed, with_idx=False)
        assert d.sparse_mla_workspace_size(wl.T, wl.H, wl.K) > 256, "the case must use split partials"
        t = to_device(wl)
        idx_d = dev(_indices(rng, wl))
        ref_out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
        ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, wl.K))
        d.dsa_sparse_mla(t["q"], t["kv"], t["page_table"], t["seq_lens"], t["cu_q"], idx_d, wl.scale, out=ref_out,
                         lse=ref_lse, workspace=ws)
        ws.check()
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        _call_static(lib, t, idx_d, wl, out, lse)
        torch.cuda.synchronize()
        np.testing.assert_allclose(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), atol=2e-2, rtol=1e-2,
                                   err_msg=f"call {call}")
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=1e-3, rtol=1e-3)


@pytest.mark.parametrize("case", ["fp8_rowscale_h64", "bf16_h128_dims_split"])
def test_static_other_kernels_match_workspace_version(orc, case):
    # The FP8 latent cache (E4M3 rows with a row scale) and the 128-head
    # dims-split CTA pair also run through the static scratch: each call is
    # compared with dsa_sparse_mla on the same inputs and with the oracle.
    import indexer_top_sparse_gb300 as d
    from _util import tuning
    lib = d.load()
    H = 64 if case.startswith("fp8") else 128
    rng = np.random.default_rng(5 + H)
    wl = make_workload(f"static_{case}", [2500, 1300], [1, 1], H=H, K=1200, page_size=64, seed=5 + H,
                       with_idx=False)
    t = to_device(wl)
    idx = _indices(rng, wl)
    idx_d = dev(idx)
    knobs = dict(mla_dsplit=1) if case.startswith("bf16") else dict(mla_dsplit=-1)
    fp8 = case.startswith("fp8")
    if fp8:
        nope, rope, rsc = d.dsa_quant_fp8_rows(t["kv"])
        kw = dict(kv_rope=rope, kv_scale=rsc, dtype="fp8_rowscale")
    else:
        nope, rope, rsc, kw = None, None, None, {}
    with tuning(**knobs):
        assert d.sparse_mla_workspace_size(wl.T, wl.H, wl.K) > 256, "the case must use split partials"
        ref_out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
        ws = d.Workspace(d.sparse_mla_workspace_size(wl.T, wl.H, wl.K))
        d.dsa_sparse_mla(t["q"], t["kv"] if not fp8 else nope, t["page_table"], t["seq_lens"], t["cu_q"], idx_d,
                         wl.scale, out=ref_out, lse=ref_lse, workspace=ws, **kw)
        ws.check()
        for call in range(2):
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            _call_static(lib, t, idx_d, wl, out, lse, kv=nope, rope=rope, scale=rsc, dtype=1 if fp8 else 0)
            torch.cuda.synchronize()
            np.testing.assert_allclose(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), atol=2e-2,
                                       rtol=1e-2, err_msg=f"{case} call {call}")
            np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=1e-3, rtol=1e-3)
    if fp8:
        rn, rr, rs = orc.quant_fp8_rows(wl.kv)
        want, _ = orc.sparse_mla(wl.q, rn, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size,
                                 dtype=orc.KV_FP8_ROWSCALE, kv_rope=rr, kv_scale=rs)
    else:
        want, _ = orc.sparse_mla(wl.q, wl.kv, wl.page_table, wl.cu_q, idx, wl.scale, wl.page_size)
    np.testing.assert_allclose(out.float().cpu().numpy(), want, atol=2e-2, rtol=1e-2, err_msg=f"{case} vs oracle")


def test_static_rejects_requests_beyond_its_scratch():
    import indexer_top_sparse_gb300 as d
    lib = d.load()
    # 100 rows x 128 heads x 8192 keys need at least 4 splits: ~105 MB of partials
    need = d.sparse_mla_workspace_size(100, 128, 8192)
    if need <= (32 << 20):
        pytest.skip("this device's split choice fits the static scratch")
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    rc = lib.dsa_sparse_mla_static(P(dummy.data_ptr()), P(dummy.data_ptr()), None, None, 1, P(dummy.data_ptr()), 1,
                                   P(dummy.data_ptr()), P(dummy.data_ptr()), P(dummy.data_ptr()), 1, 100, 128, 8192,
                                   ctypes.c_float(1.0), 64, 0, P(dummy.data_ptr()), None, None)
    assert rc == 2


def test_static_errors_are_read_back():
    # An index past its row's position is reported and its key skipped (the
    # same rule as dsa_sparse_mla); the allocation-free call keeps the error
    # bit in its static array, and dsa_sparse_mla_static_get_error reads it
    # back and clears it, so the next clean call reads DSA_OK.
    import indexer_top_sparse_gb300 as d
    lib = d.load()
    rng = np.random.default_rng(7)
    wl = make_workload("static_err", [2000, 700], [1, 1], H=64, K=512, page_size=64, seed=7, with_idx=False)
    t = to_device(wl)
    idx = _indices(rng, wl)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
    _call_static(lib, t, dev(idx), wl, out, lse)
    assert lib.dsa_sparse_mla_static_get_error(stream) == 0
    bad = idx.copy()
    bad[1, 3] = int(wl.query_pos()[1]) + 5  # a position row 1 cannot see
    _call_static(lib, t, dev(bad), wl, out, lse)
    assert lib.dsa_sparse_mla_static_get_error(stream) == 5  # DSA_ERR_BAD_INDEX
    assert np.isfinite(out.float().cpu().numpy()).all()
    _call_static(lib, t, dev(idx), wl, out, lse)
    assert lib.dsa_sparse_mla_static_get_error(stream) == 0
