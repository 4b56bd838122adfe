"""The library's calls are safe to capture in a CUDA graph (no allocation,
no host synchronisation, no pageable copy when the caller passes the outputs
and the workspace): a decode step captured once and replayed on new inputs
gives bit for bit what the same calls give eagerly, for the bf16 path and
for the FP8 path with its Q quantisation (index-Q quantise -> indexer + Top-K
-> sparse MLA -> split combine, chained by programmatic dependent launch), and
for the FP8 path with the index query quantised inside the indexer (one
launch fewer).
The replayed step is also checked against the oracle on the new inputs:
index sets within the near-threshold band, attention (fed the replay's
indices) within 2e-2 / 1e-2."""
import numpy as np
import pytest
import torch

from _util import check_index_sets, dev, dev_bf16
from indexer_top_sparse_gb300.inputs import make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fp8", [False, True, "fused_q"])
def test_decode_step_replays_in_a_cuda_graph(orc, fp8):
    import indexer_top_sparse_gb300 as d
    wl = make_workload("graph", [3000, 700, 64, 2049], [1, 1, 1, 1], H=128, K=512, page_size=64, seed=77)
    pt, sl, cq = dev(wl.page_table), dev(wl.seq_lens), dev(wl.cu_q)
    q_idx, head_w, q = dev_bf16(wl.q_idx), dev(wl.head_w), dev_bf16(wl.q)
    idx = torch.empty((wl.T, wl.K), dtype=torch.int32, device="cuda")
    out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    ws = d.Workspace(max(d.index_topk_workspace_size(wl.B, wl.T, wl.K, wl.max_pages, wl.page_size),
                         d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)))
    if fp8:
        k8, ks = d.dsa_quant_mxfp8(dev_bf16(wl.k_idx))
        nope, rope, vsc = d.dsa_quant_fp8_tiles(dev_bf16(wl.kv))
        q8 = torch.empty((wl.T, 64, 128), dtype=torch.uint8, device="cuda")
        qs = torch.empty((wl.T, 64, 4), dtype=torch.uint8, device="cuda")
    else:
        k_idx, kv = dev_bf16(wl.k_idx), dev_bf16(wl.kv)

    def step():
        if fp8 == "fused_q":
            d.dsa_index_topk(q_idx, head_w, k8, pt, sl, cq, wl.K, indices=idx, workspace=ws, k_idx_scale=ks,
                             dtype="mxfp8_qbf16")
            d.dsa_sparse_mla(q, nope, pt, sl, cq, idx, wl.scale, out=out, workspace=ws, kv_rope=rope,
                             kv_scale=vsc, dtype="fp8_tile128")
        elif fp8:
            d.dsa_quant_mxfp8(q_idx, q=q8, scales=qs)
            d.dsa_index_topk(q8, head_w, k8, pt, sl, cq, wl.K, indices=idx, workspace=ws, q_idx_scale=qs,
                             k_idx_scale=ks, dtype="mxfp8")
            d.dsa_sparse_mla(q, nope, pt, sl, cq, idx, wl.scale, out=out, workspace=ws, kv_rope=rope,
                             kv_scale=vsc, dtype="fp8_tile128")
        else:
            d.dsa_index_topk(q_idx, head_w, k_idx, pt, sl, cq, wl.K, indices=idx, workspace=ws)
            d.dsa_sparse_mla(q, kv, pt, sl, cq, idx, wl.scale, out=out, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            step()                       # warm up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    rng = np.random.default_rng(3)
    for trial in range(2):
        # new step inputs, written in place into the captured buffers
        q_idx.copy_(torch.from_numpy(rng.standard_normal(tuple(q_idx.shape)).astype(np.float32)).to(q_idx))
        q.copy_(torch.from_numpy(rng.standard_normal(tuple(q.shape)).astype(np.float32)).to(q))
        step()
        torch.cuda.synchronize()
        want_idx, want_out = idx.clone(), out.clone()
        idx.fill_(-7)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ws.check()
        assert torch.equal(idx, want_idx), trial
        assert torch.equal(out.view(torch.int16), want_out.view(torch.int16)), trial
        _check_against_oracle(orc, wl, fp8, q_idx, q, idx, out)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _check_against_oracle(orc, wl, fp8, q_idx, q, idx, out):
    qi, qb = _bits(q_idx), _bits(q)
    g_idx = idx.cpu().numpy()
    if fp8:
        q8, qs = orc.quant_mxfp8(qi)
        k8, ks = orc.quant_mxfp8(wl.k_idx)
        ref_idx, ref_sc = orc.index_topk(q8, wl.head_w, k8, wl.page_table, wl.seq_lens, wl.cu_q, wl.K, wl.page_size,
                                         dtype=orc.IDX_MXFP8, q_scale=qs, k_scale=ks, want_scores=True)
        nope, rope, vsc = orc.quant_fp8_tiles(wl.kv)
        ref_out, _ = orc.sparse_mla(qb, nope, wl.page_table, wl.cu_q, g_idx, wl.scale, wl.page_size,
                                    dtype=orc.KV_FP8_TILE128, kv_rope=rope, kv_scale=vsc)
    else:
        ref_idx, ref_sc = orc.index_topk(qi, wl.head_w, wl.k_idx, wl.page_table, wl.seq_lens, wl.cu_q, wl.K,
                                         wl.page_size, want_scores=True)
        ref_out, _ = orc.sparse_mla(qb, wl.kv, wl.page_table, wl.cu_q, g_idx, wl.scale, wl.page_size)
    pos = wl.query_pos()
    for t in range(wl.T):
        check_index_sets(g_idx[t], ref_idx[t], ref_sc[t], int(pos[t]) + 1, wl.K)
    np.testing.assert_allclose(out.float().cpu().numpy(), ref_out, atol=2e-2, rtol=1e-2)
