"""Benchmark of the DSA "score, select, sparse read" path on GB300.

One step = the whole hot path over one batch: dsa_index_topk (fused indexer +
Top-K) then dsa_sparse_mla, on the decode workload of 32 sequences at 32768
cached positions (K=2048, 64x128 index heads, 128 MLA heads, 576-wide bf16
latent rows, 64-row pages in a seeded random permutation).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N>1) every rank runs its own
batch (independent replicas, no collective on the data path): value is the
sum of all ranks' tokens over the slowest rank's time.

--impl reference times the CPU oracle (plain single-threaded C, fp64) on this
machine's host cores, on a bounded sample of the same workload.

The default run also measures the other workloads, one after the other, and
nests their results under "workloads" (skip with --no-workloads):
decode_b1_n2048 (one sequence of 2048 positions, K=256, 16 MLA heads, one
contiguous 2048-row page), decode_b64_mixed_fp8 (64 sequences, lengths
uniform in [4096, 131072], MXFP8 index keys, FP8 latent rows), prefill_16k
(one 16384-token sequence, causal, bf16) and prefill_131k_chunked_fp8 (one
131072-token sequence in 32 chunks of 4096 queries against the paged cache,
MXFP8 / FP8).  --workload NAME measures one of them alone (same JSON line,
config.workload naming it).  Their caches are drawn on the device (seeded
torch generator) and quantised by the library's own quantisers.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s + prefill tokens/s (index+TopK+sparse MLA), % HBM/tensor roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0


def peaks():
    try:
        p = json.load(open(PEAKS_FILE))
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


NOMINAL_HBM_GBS = 8000.0


def bf16_peaks():
    try:
        return float(json.load(open(PEAKS_FILE))["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def kernel_source_hash(name: str) -> str:
    """Hash of a kernel's source file and the headers every kernel includes."""
    csrc = os.path.join(ROOT, "indexer_top_sparse_gb300", "csrc")
    h = hashlib.sha256()
    for f in (name, "ptx.cuh", "kernels.h", "mxfp8.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, source: str):
    """DRAM bytes per launch from a committed ncu summary, only if the kernel
    source is unchanged since the capture."""
    try:
        t = json.load(open(TRAFFIC_FILE))[kernel]
        if t["source_sha"] == kernel_source_hash(source):
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------- algorithmic bytes

def indexer_bytes(wl) -> float:
    """Bytes the indexer must move for the batch: every causal history key once
    (128 bf16 = 256 B), the query's 64x128 bf16 index query and 64 fp32 head
    weights, its page-table row and its K int32 indices."""
    pos = wl.query_pos()
    n = (pos + 1).astype(np.float64)
    return float(np.sum(n * 256 + 64 * 128 * 2 + 64 * 4 + 4 * wl.K + 4 * np.ceil(n / wl.page_size)))


def mla_bytes(wl) -> float:
    """Bytes sparse MLA must move: min(K, n) selected 576-wide bf16 rows, the
    H x 576 bf16 query, the H x 512 bf16 output, the K int32 indices and the
    page-table row."""
    pos = wl.query_pos()
    n = (pos + 1).astype(np.float64)
    sel = np.minimum(n, wl.K)
    return float(np.sum(sel * 1152 + wl.H * 1152 + wl.H * 1024 + 4 * wl.K + 4 * np.ceil(n / wl.page_size)))


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle timing

def oracle_rate(wl, budget_s, max_queries: int, frac: int = 1):
    """Time the CPU oracle on whole decode queries (frac = 1) until budget_s
    seconds of work (None: no time bound) or max_queries units; with frac > 1 each unit is 1/frac of a query
    (the indexer over the first N/frac positions and Top-K of those, attention
    for H/frac heads).  Returns (queries per second, units, seconds)."""
    import oracle
    oracle.build()
    H = wl.H
    hq = max(1, H // frac)
    units, spent = 0, 0.0
    t = 0
    while units < max_queries and (budget_s is None or spent < budget_s or units == 0):
        b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
        n = int(wl.query_pos()[t]) + 1
        n_part = max(1, n // frac)
        t0 = time.perf_counter()
        sc = oracle.index_scores_row(wl.q_idx[t], wl.head_w[t], wl.k_idx, wl.page_table[b], wl.page_size, n_part)
        idx = oracle.topk_rows(sc[None, :], np.array([n_part], np.int32), wl.K)
        q_part = np.ascontiguousarray(wl.q[t:t + 1, :hq])
        cu = np.array([0, 1], np.int32)
        oracle.sparse_mla(q_part, wl.kv, wl.page_table[b:b + 1], cu, idx, wl.scale, wl.page_size)
        spent += time.perf_counter() - t0
        units += 1
        t = (t + 1) % wl.T
    return (units / frac) / spent, units, spent


# ---------------------------------------------------------------- multi-rank

def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats across all ranks of the
    default process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def aggregate_rate(tokens_per_rank: int, world: int, seconds_max: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * max(world, 1) / seconds_max


# ---------------------------------------------------------------- other workloads

def attention_flops(rows_sel: np.ndarray, H: int) -> float:
    """QK over 576 dims and PV over 512 dims for every (query, selected key, head)."""
    return float(np.sum(rows_sel.astype(np.float64))) * H * 2.0 * (576 + 512)


WORKLOADS = ("decode_b1_n2048", "decode_b64_mixed_fp8", "prefill_16k", "prefill_131k_chunked_fp8")


def measure_workload(name, args, dev, world, rank, steps, warmup, seed):
    """Timed steps of one of the other workloads on this rank's GPU: the
    one-sequence 2048-position decode (K = 256, 16 heads, one contiguous
    2048-row page), the mixed-length FP8 decode, the 16k prefill or the 131k
    chunked FP8 prefill.  Returns the JSON object of the run (the caller
    prints it or nests it)."""
    import torch
    import indexer_top_sparse_gb300 as d
    from indexer_top_sparse_gb300.inputs import make_page_table

    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 1000 * rank)

    def normal_bf16(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)

    H, K, ps, scale = 128, 2048, 64, float(1.0 / np.sqrt(192.0))
    fp8 = name.endswith("fp8")
    kv_fmt = "fp8_tile128" if args.kv_scales == "tile128" else "fp8_rowscale"
    row_b = 512 + 128 + (16 if kv_fmt == "fp8_tile128" else 4)   # e4m3 latent + bf16 rope + fp32 scales
    use_graph = name == "decode_b1_n2048"
    if name == "decode_b1_n2048":
        H, K, ps = 16, 256, 2048
        chunks = [(np.array([2048], np.int32), np.array([1], np.int32))]
        permute, copies = False, 0   # copies: enough to cycle through more than L2 (set below)
    elif name == "decode_b64_mixed_fp8":
        lens = np.random.default_rng(seed + rank + 7919).integers(4096, 131072, size=64, endpoint=True)
        lens = lens.astype(np.int32)
        chunks = [(lens, np.ones(64, np.int32))]
        permute, copies = True, 2
    elif name == "prefill_16k":
        n = args.prefill_tokens
        chunks = [(np.array([n], np.int32), np.array([n], np.int32))]
        permute, copies = False, 1
    else:
        chunks = [(np.array([4096 * (c + 1)], np.int32), np.array([4096], np.int32)) for c in range(32)]
        permute, copies = True, 1
    cache_lens = chunks[-1][0]
    pt_np, P = make_page_table(np.random.default_rng(seed + rank), cache_lens, ps, permute)
    T_all = int(sum(int(n.sum()) for _, n in chunks))
    pt = torch.from_numpy(pt_np).to(dev)
    if copies == 0:
        # the small decode's whole input is about 1 MB: cycle through enough
        # separate copies that every step reads inputs last touched more than
        # L2's capacity ago
        one = P * ps * (128 + 576) * 2 + T_all * (64 * 128 * 2 + 64 * 4 + H * 576 * 2)
        copies = int(np.ceil(384 * 2**20 / one))

    sets = []
    for _ in range(copies):
        k_bf, kv_bf = normal_bf16(P, ps, 128), normal_bf16(P, ps, 576)
        st = {"q_idx": normal_bf16(T_all, 64, 128), "q": normal_bf16(T_all, H, 576),
              "head_w": torch.randn(T_all, 64, generator=gen, device=dev) / 8.0}
        if fp8:
            st["k_idx"], st["k_sc"] = d.dsa_quant_mxfp8(k_bf)
            quant = d.dsa_quant_fp8_tiles if kv_fmt == "fp8_tile128" else d.dsa_quant_fp8_rows
            st["kv"], st["rope"], st["rsc"] = quant(kv_bf)
        else:
            st["k_idx"], st["kv"] = k_bf, kv_bf
        del k_bf, kv_bf
        sets.append(st)
    torch.cuda.synchronize(dev)
    in_bytes = sum(v.numel() * v.element_size() for v in sets[0].values())

    # per-chunk views and small tensors
    plan = []
    q0 = 0
    for sl_np, nq_np in chunks:
        B = len(sl_np)
        cq_np = np.zeros(B + 1, np.int32)
        cq_np[1:] = np.cumsum(nq_np)
        T = int(cq_np[-1])
        plan.append({"r0": q0, "T": T, "B": B, "sl": torch.from_numpy(sl_np).to(dev),
                     "cq": torch.from_numpy(cq_np).to(dev), "pt": pt[:B], "sl_np": sl_np, "cq_np": cq_np})
        q0 += T
    idx = torch.empty((max(c["T"] for c in plan), K), dtype=torch.int32, device=dev)
    out = torch.empty((T_all, H, 512), dtype=torch.bfloat16, device=dev)
    if fp8 and args.q_quant == "separate":
        qi8 = torch.empty((T_all, 64, 128), dtype=torch.uint8, device=dev)
        qi_sc = torch.empty((T_all, 64, 4), dtype=torch.uint8, device=dev)
    ws = d.Workspace(max(max(d.index_topk_workspace_size(c["B"], c["T"], K, pt.shape[1], ps) for c in plan),
                         max(d.sparse_mla_workspace_size(c["T"], H, K) for c in plan)), dev)
    stream = torch.cuda.current_stream(dev)
    launches = 0

    def step(st, ev=None, part="both"):
        nonlocal launches
        n = 0
        for c in plan:
            r0, T = c["r0"], c["T"]
            if ev is not None:
                ev[0].append(torch.cuda.Event(enable_timing=True))
                ev[0][-1].record(stream)
            if part == "mla":
                pass
            elif fp8 and args.q_quant == "separate":
                d.dsa_quant_mxfp8(st["q_idx"][r0:r0 + T], q=qi8[r0:r0 + T], scales=qi_sc[r0:r0 + T])
                d.dsa_index_topk(qi8[r0:r0 + T], st["head_w"][r0:r0 + T], st["k_idx"], c["pt"], c["sl"], c["cq"], K,
                                 indices=idx[:T], workspace=ws, q_idx_scale=qi_sc[r0:r0 + T], k_idx_scale=st["k_sc"],
                                 dtype="mxfp8")
                n += 2
            elif fp8:
                # MXFP8 keys; the bf16 index query is quantised inside the indexer
                d.dsa_index_topk(st["q_idx"][r0:r0 + T], st["head_w"][r0:r0 + T], st["k_idx"], c["pt"], c["sl"],
                                 c["cq"], K, indices=idx[:T], workspace=ws, k_idx_scale=st["k_sc"],
                                 dtype="mxfp8_qbf16")
                n += 1
            else:
                d.dsa_index_topk(st["q_idx"][r0:r0 + T], st["head_w"][r0:r0 + T], st["k_idx"], c["pt"], c["sl"],
                                 c["cq"], K, indices=idx[:T], workspace=ws)
                # (the flat bf16 indexer also zeroes its counters with a cudaMemsetAsync: not a kernel
                # of this library, not counted)
                n += 1
            if ev is not None:
                ev[1].append(torch.cuda.Event(enable_timing=True))
                ev[1][-1].record(stream)
            if part == "index":
                pass
            elif fp8:
                d.dsa_sparse_mla(st["q"][r0:r0 + T], st["kv"], c["pt"], c["sl"], c["cq"], idx[:T], scale,
                                 out=out[r0:r0 + T], workspace=ws, kv_rope=st["rope"], kv_scale=st["rsc"],
                                 dtype=kv_fmt)
                n += 1 + (1 if d.sparse_mla_workspace_size(T, H, K) > 256 else 0)
            else:
                d.dsa_sparse_mla(st["q"][r0:r0 + T], st["kv"], c["pt"], c["sl"], c["cq"], idx[:T], scale,
                                 out=out[r0:r0 + T], workspace=ws)
                n += 1 + (1 if d.sparse_mla_workspace_size(T, H, K) > 256 else 0)
            if ev is not None:
                ev[2].append(torch.cuda.Event(enable_timing=True))
                ev[2][-1].record(stream)
        launches = n

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    for i in range(warmup):
        step(sets[i % copies])
    ws.check()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    timing = "CUDA events on the launching stream around each step; per-kernel times from a second pass with an " \
             "event between the calls"
    if use_graph:
        # A step of about 1 MB takes microseconds on the GPU, less than the
        # host needs to issue its calls: eagerly issued steps would time the
        # host.  The steps (each on its own input copy) are captured once in
        # a CUDA graph -- whole steps, the indexer calls alone, the attention
        # calls alone -- and each graph is replayed and timed as a whole.
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graphs = {}
        for part in ("both", "index", "mla"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(steps):
                    step(sets[(warmup + i) % copies], part=part)
            graphs[part] = g
        stream.wait_stream(side)
        for g in graphs.values():
            g.replay()
        torch.cuda.synchronize(dev)

        def replay_time(g):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) * 1e-3 / steps

        t_step = max_over_ranks([replay_time(graphs["both"])], dev)[0]
        t_idx, t_mla = replay_time(graphs["index"]), replay_time(graphs["mla"])
        step(sets[0])  # the launch count of one whole step
        torch.cuda.synchronize(dev)
        timing = (f"one CUDA graph of {steps} steps (each on its own input copy) replayed and timed with CUDA events; "
                  f"per-kernel times from graphs of the indexer calls alone and of the attention calls alone")
        if world > 1:
            torch.distributed.barrier()
    else:
        # whole steps, events only around each step (the kernels of a step
        # overlap through programmatic dependent launch as in use) ...
        s_ev = []
        for i in range(steps):
            e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            e[0].record(stream)
            step(sets[(warmup + i) % copies])
            e[1].record(stream)
            s_ev.append(e)
        torch.cuda.synchronize(dev)
        # ... then the same steps with an event between the calls, for the
        # per-kernel times (that event stops the overlap)
        evs = []
        for i in range(steps):
            ev = ([], [], [])
            step(sets[(warmup + i) % copies], ev)
            evs.append(ev)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        t_step = max_over_ranks([sum(a.elapsed_time(b) for a, b in s_ev) * 1e-3 / steps], dev)[0]
        t_idx = sum(a.elapsed_time(b) for ev in evs for a, b in zip(ev[0], ev[1])) * 1e-3 / steps
        t_mla = sum(a.elapsed_time(b) for ev in evs for a, b in zip(ev[1], ev[2])) * 1e-3 / steps
    clk = clocks.stop()
    ws.check()

    # algorithmic bytes and flops
    sel_all, idx_bytes, mla_b, n_hist = [], 0.0, 0.0, 0.0
    for c in plan:
        for b in range(c["B"]):
            nq = int(c["cq_np"][b + 1] - c["cq_np"][b])
            p = int(c["sl_np"][b]) - nq + np.arange(nq)
            n = (p + 1).astype(np.float64)
            sel = np.minimum(n, K)
            sel_all.append(sel)
            n_hist += float(n.sum())
            key_b = 132 if fp8 else 256
            idx_bytes += float(np.sum(n * key_b + 64 * 128 * 2 + 256 + 4 * K + 4 * np.ceil(n / ps)))
            mla_b += float(np.sum(sel * (row_b if fp8 else 1152) + H * 1152 + H * 1024 + 4 * K + 4 * np.ceil(n / ps)))
    sel_all = np.concatenate(sel_all)
    f_mla = attention_flops(sel_all, H)
    f_idx = n_hist * 64 * 128 * 2.0
    hbm, peak_kind = peaks()
    bf16_peak, bf16_kind = bf16_peaks()
    tokens = T_all * max(world, 1)
    line = {"metric": METRIC, "value": tokens / t_step, "unit": "tokens/s", "n_gpus": max(world, 1),
            "steps": steps, "warmup": warmup, "ms_per_step": 1e3 * t_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/bf16" if fp8 else "bf16",
            "data": "synthetic (seeded N(0,1) drawn on the device; FP8 caches made by the library's quantisers)",
            "config": {"workload": name, "H": H, "K": K, "H_I": 64, "d_I": 128, "page_size": ps,
                       "query_rows": T_all, "cached_positions": int(np.sum(cache_lens)), "chunks": len(plan),
                       "kv_cache": kv_fmt if fp8 else "bf16",
                       "tuning": getattr(args, "tuned", None) or "automatic",
                       "index_query": ("bf16, quantised inside the indexer" if args.q_quant == "fused" else
                                       "quantised to MXFP8 in its own launch") if fp8 else "bf16",
                       "parallelism": f"replicas{max(world, 1)}",
                       "l2": (f"inputs larger than L2: {copies} alternating cop{'ies' if copies > 1 else 'y'} of "
                              f"every step input ({in_bytes / 2**30:.3f} GiB each), no flush"),
                       "timing": timing},
            "kernels": {"indexer_topk": {"seconds_per_step": t_idx, "algorithmic_bytes": idx_bytes,
                                         "achieved_gbs": idx_bytes / t_idx / 1e9, "flops": f_idx,
                                         "achieved_tflops": f_idx / t_idx / 1e12},
                        "sparse_mla": {"seconds_per_step": t_mla, "algorithmic_bytes": mla_b,
                                       "achieved_gbs": mla_b / t_mla / 1e9, "flops": f_mla,
                                       "achieved_tflops": f_mla / t_mla / 1e12}},
            "gpu_launches": launches * steps, "clocks": clk}
    if name.startswith("prefill"):
        # the sparse MLA kernel against the bf16 tensor peak (FP8 caches are
        # dequantised to bf16 on the way into shared memory, so its MMAs are
        # bf16 too); the MXFP8 indexer of the chunked prefill against the
        # bf16 peak times the nominal FP8 / bf16 ratio of 2
        line["roofline"] = {"bound": "tensor", "kernel": "sparse_mla", "achieved": f_mla / t_mla / 1e12,
                            "peak": bf16_peak, "peak_kind": bf16_kind, "unit": "TFLOP/s",
                            "frac": f_mla / t_mla / 1e12 / bf16_peak, "traffic": None}
        if fp8:
            fp8_peak = 2.0 * bf16_peak
            line["kernels"]["indexer_topk"]["tensor_frac"] = {
                "achieved": f_idx / t_idx / 1e12, "peak": fp8_peak, "unit": "TFLOP/s",
                "peak_kind": f"{bf16_kind} bf16 x 2 (nominal FP8/bf16 dense ratio)",
                "frac": f_idx / t_idx / 1e12 / fp8_peak}
    else:
        dom = "indexer_topk" if t_idx >= t_mla else "sparse_mla"
        ach = (idx_bytes / t_idx if dom == "indexer_topk" else mla_b / t_mla) / 1e9
        line["roofline"] = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "peak_kind": peak_kind,
                            "unit": "GB/s", "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                            "traffic": None}
        line["step_roofline"] = {"bytes": idx_bytes + mla_b, "achieved_gbs": (idx_bytes + mla_b) / t_step / 1e9,
                                 "frac": (idx_bytes + mla_b) / t_step / 1e9 / hbm,
                                 "frac_of_nominal_8tbs": (idx_bytes + mla_b) / t_step / 1e9 / NOMINAL_HBM_GBS}
        if name == "decode_b1_n2048":
            line["roofline"]["note"] = ("a single 2048-position query moves about 1 MB: launch and latency "
                                        "bound, so the HBM fraction is reported but not meaningful")
    del sets, out, idx, ws
    torch.cuda.empty_cache()
    return line


def run_other_workload(args, world, rank, local_rank):
    """One of the other workloads as the whole run (its own JSON line)."""
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    line = measure_workload(args.workload, args, dev, world, rank, args.steps, args.warmup, args.seed)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_append_workload(args, world, rank, local_rank):
    """Cache append of one 131072-token sequence (a long prefill's keys): the
    new index keys go into an MXFP8 cache and the new latent rows into an FP8
    cache with tile-128 scales, written straight into permuted pages.
    HBM-bound: bf16 rows in, quantised rows out."""
    import torch
    import indexer_top_sparse_gb300 as d
    from indexer_top_sparse_gb300.inputs import make_page_table

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 1000 * rank)
    T, ps = 131072, 64
    pt_np, P = make_page_table(np.random.default_rng(args.seed + rank), [T], ps, True)
    pt = torch.from_numpy(pt_np).to(dev)
    sl = torch.tensor([T], dtype=torch.int32, device=dev)
    cq = torch.tensor([0, T], dtype=torch.int32, device=dev)
    copies = 2   # alternating inputs, each far larger than L2
    src = [(torch.randn(T, 128, generator=gen, device=dev).to(torch.bfloat16),
            torch.randn(T, 576, generator=gen, device=dev).to(torch.bfloat16)) for _ in range(copies)]
    kc = torch.empty((P, ps, 128), dtype=torch.uint8, device=dev)
    ksc = torch.empty((P, ps, 4), dtype=torch.uint8, device=dev)
    kv = torch.empty((P, ps, 512), dtype=torch.uint8, device=dev)
    rope = torch.empty((P, ps, 64), dtype=torch.bfloat16, device=dev)
    vsc = torch.empty((P, ps, 4), dtype=torch.float32, device=dev)
    ws = d.Workspace(256, dev)

    def step(i):
        k_new, kv_new = src[i % copies]
        d.dsa_cache_append(pt, sl, cq, k_new=k_new, kv_new=kv_new, k_cache=kc, k_scale=ksc, kv_cache=kv,
                           kv_rope=rope, kv_scale=vsc, idx_dtype="mxfp8", kv_dtype="fp8_tile128", workspace=ws)

    clocks = ClockSampler(local_rank)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    ws.check()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ws.check()
    t_step = max_over_ranks([e0.elapsed_time(e1) * 1e-3 / args.steps], dev)[0]
    # bytes: bf16 key and latent row in; e4m3 key + 4 e8m0, e4m3 latent + bf16 rope + 4 fp32 out; the
    # page table row and the two small per-sequence arrays
    row_bytes = (128 * 2 + 576 * 2) + (128 + 4) + (512 + 128 + 16)
    nbytes = float(T) * row_bytes + 4 * pt.shape[1] + 12
    hbm, peak_kind = peaks()
    ach = nbytes / t_step / 1e9
    line = {"metric": "cache append tokens/s (index key MXFP8 + latent FP8 tile-128 into pages)",
            "value": T * max(world, 1) / t_step, "unit": "tokens/s", "n_gpus": max(world, 1), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16->e4m3", "data": "synthetic (seeded N(0,1) drawn on the device)",
            "config": {"workload": args.workload, "tokens": T, "page_size": ps, "pages": P,
                       "parallelism": f"replicas{max(world, 1)}",
                       "l2": f"inputs larger than L2: {copies} alternating copies of the new rows "
                             f"({T * 1408 / 2**20:.0f} MiB each), no flush"},
            "roofline": {"bound": "hbm", "kernel": "cache_append", "achieved": ach, "peak": hbm,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": ach / hbm, "traffic": None},
            "gpu_launches": args.steps, "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# steps and warm-up steps of each other workload in the default run (the
# chunked 131k prefill takes about half a second per step)
WORKLOAD_STEPS = {"decode_b1_n2048": (200, 20), "decode_b64_mixed_fp8": (50, 5), "prefill_16k": (10, 3),
                  "prefill_131k_chunked_fp8": (3, 3)}
NESTED_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "kernels", "roofline",
               "step_roofline", "gpu_launches", "clocks")


def other_workloads(args, dev):
    """The other workloads, one after the other (the headline decode's few GB
    stay allocated; HBM holds both): each entry is that workload's own
    measurement."""
    import torch
    torch.cuda.synchronize(dev)
    res = {}
    for name in WORKLOADS:
        steps, warmup = WORKLOAD_STEPS[name]
        line = measure_workload(name, args, dev, 1, 0, steps, warmup, args.seed)
        res[name] = {k: line[k] for k in NESTED_KEYS if k in line}
    return res


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2", default="rotate", choices=["rotate", "flush"],
                    help="between timed steps: alternate two copies of every step input (default) or write a "
                         "512 MiB buffer")
    ap.add_argument("--workload", default="decode_b32_n32768",
                    choices=["decode_b32_n32768", "decode_b1_n2048", "decode_b64_mixed_fp8", "prefill_16k",
                             "prefill_131k_chunked_fp8", "append_131k_fp8"])
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads the default run measures after the headline decode")
    ap.add_argument("--tune", action="append", default=[], metavar="NAME=VALUE",
                    help="set a library tuning knob (dsa_set_tuning) for the run, e.g. mla_dsplit=1")
    ap.add_argument("--q-quant", default="fused", choices=["fused", "separate"],
                    help="FP8 workloads: quantise the index query inside the indexer (default) or in its own launch")
    ap.add_argument("--kv-scales", default="row", choices=["row", "tile128"],
                    help="FP8 workloads: one fp32 scale per latent row (default) or per 128 latent dims")
    ap.add_argument("--graph", action="store_true",
                    help="also time the decode step captured once in a CUDA graph and replayed")
    ap.add_argument("--batch", type=int, default=32,
                    help="sequences per rank (default 32, the benchmark workload; smaller only for profiling)")
    ap.add_argument("--prefill-tokens", type=int, default=16384,
                    help="prefill_16k: tokens of the sequence (default 16384, the benchmark workload; smaller only "
                         "for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    tuned = {}
    for kv in args.tune:
        name, _, val = kv.partition("=")
        tuned[name] = int(val)
    args.tuned = tuned
    if tuned and args.impl == "ours":
        import indexer_top_sparse_gb300 as d
        for name, val in tuned.items():
            d.set_tuning(name, val)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload != "decode_b32_n32768":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the oracle baseline is timed on the "
                                  "decode_b32_n32768 workload only"}), flush=True)
            return
        if args.workload == "append_131k_fp8":
            run_append_workload(args, world, rank, local_rank)
        else:
            run_other_workload(args, world, rank, local_rank)
        return

    from indexer_top_sparse_gb300.inputs import decode_b32_n32k, make_workload
    if args.batch == 32:
        wl = decode_b32_n32k(args.seed + rank)
    else:
        wl = make_workload(f"decode_b{args.batch}_n32768_k2048_h128_paged64", [32768] * args.batch,
                           [1] * args.batch, H=128, K=2048, page_size=64, permute=True, seed=args.seed + rank)
    cfg = {"workload": wl.name, "B": wl.B, "N": int(wl.seq_lens[0]), "K": wl.K, "H": wl.H, "H_I": 64, "d_I": 128,
           "D": 576, "D_v": 512, "page_size": wl.page_size, "global_batch": wl.B * max(world, 1),
           "parallelism": f"replicas{max(world, 1)}", "tuning": tuned or "automatic"}

    if args.impl == "reference":
        if rank != 0:
            return
        # bounded sample: each step is 1/frac of one decode query, frac chosen
        # so that the whole run takes about two minutes
        probe, _, tprobe = oracle_rate(wl, None, 1)
        per_query = 1.0 / probe
        frac = 1
        while frac < 256 and (args.steps + args.warmup) * per_query / frac > 120.0:
            frac *= 2
        oracle_rate(wl, None, args.warmup, frac)
        rate, units, spent = oracle_rate(wl, None, args.steps, frac)
        sample = (f"{units} steps, each 1/{frac} of a decode query (indexer over N/{frac} positions + Top-K, "
                  f"attention for H/{frac} heads) of the same workload; tokens/s = queries / time")
        line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / max(units, 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import indexer_top_sparse_gb300 as d

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    # Step inputs.  With --l2 rotate, two separate copies of every input (the
    # caches included) alternate between steps: a step reads buffers last
    # touched two steps earlier, with far more than the L2 capacity read in
    # between, so no step finds its data in L2.
    copies = 2 if args.l2 == "rotate" else 1
    sets = []
    for _ in range(copies):
        sets.append({"k_idx": bf16(wl.k_idx), "kv": bf16(wl.kv), "q_idx": bf16(wl.q_idx), "q": bf16(wl.q),
                     "head_w": torch.from_numpy(wl.head_w).to(dev), "pt": torch.from_numpy(wl.page_table).to(dev),
                     "sl": torch.from_numpy(wl.seq_lens).to(dev), "cq": torch.from_numpy(wl.cu_q).to(dev)})
    in_bytes = sum(v.numel() * v.element_size() for v in sets[0].values())
    cfg["l2"] = (f"inputs larger than L2: {copies} alternating copies of every step input "
                 f"({in_bytes / 2**30:.2f} GiB each), no flush" if copies > 1 else
                 "flushed between steps (512 MiB device write)")
    k_idx, kv = sets[0]["k_idx"], sets[0]["kv"]
    q_idx, q, head_w = sets[0]["q_idx"], sets[0]["q"], sets[0]["head_w"]
    pt, sl, cq = sets[0]["pt"], sets[0]["sl"], sets[0]["cq"]
    idx = torch.empty((wl.T, wl.K), dtype=torch.int32, device=dev)
    out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, device=dev)
    ws = d.Workspace(max(d.index_topk_workspace_size(wl.B, wl.T, wl.K, wl.max_pages, wl.page_size),
                         d.sparse_mla_workspace_size(wl.T, wl.H, wl.K)), dev)
    # indexer, sparse MLA, and the split combine when there are splits (the
    # flat indexer's counter zeroing is a cudaMemsetAsync, not a kernel of
    # this library, and is not counted)
    launches_per_step = 2 + (1 if d.sparse_mla_workspace_size(wl.T, wl.H, wl.K) > 256 else 0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if copies == 1 else None
    stream = torch.cuda.current_stream(dev)

    def between_steps():
        if flush is not None:
            flush.zero_()

    def run_step(qi, hw, qq, ptab, slen, cuq, c=0, out_buf=None):
        d.dsa_index_topk(qi, hw, sets[c]["k_idx"], ptab, slen, cuq, wl.K, indices=idx, workspace=ws)
        d.dsa_sparse_mla(qq, sets[c]["kv"], ptab, slen, cuq, idx, wl.scale, out=out if out_buf is None else out_buf,
                         workspace=ws)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local_rank)
    clocks.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.0:           # bring clocks to their loaded state
        run_step(q_idx, head_w, q, pt, sl, cq)
        torch.cuda.synchronize(dev)
    for i in range(args.warmup):
        between_steps()
        c = i % copies
        st_ = sets[c]
        run_step(st_["q_idx"], st_["head_w"], st_["q"], st_["pt"], st_["sl"], st_["cq"], c)
    ws.check()

    # ---- device-resident timing of whole steps (no L2 reuse between steps):
    # events only around each step, so the kernels of a step overlap as they
    # do in use (programmatic dependent launch)
    barrier()
    s_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        between_steps()
        st_ = sets[(args.warmup + i) % copies]
        s_ev[i][0].record(stream)
        run_step(st_["q_idx"], st_["head_w"], st_["q"], st_["pt"], st_["sl"], st_["cq"], (args.warmup + i) % copies)
        s_ev[i][1].record(stream)
    barrier()
    total = sum(e[0].elapsed_time(e[1]) * 1e-3 for e in s_ev)
    ws.check()

    # ---- the same steps with an event between the kernels: per-kernel times
    # for the roofline (the event stops the overlap, so these sum to a little
    # more than the step)
    barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        between_steps()
        st_ = sets[(args.warmup + i) % copies]
        ev[i][0].record(stream)
        d.dsa_index_topk(st_["q_idx"], st_["head_w"], st_["k_idx"], st_["pt"], st_["sl"], st_["cq"], wl.K,
                         indices=idx, workspace=ws)
        ev[i][1].record(stream)
        d.dsa_sparse_mla(st_["q"], st_["kv"], st_["pt"], st_["sl"], st_["cq"], idx, wl.scale, out=out, workspace=ws)
        ev[i][2].record(stream)
    barrier()
    t_idx = [e[0].elapsed_time(e[1]) * 1e-3 for e in ev]
    t_mla = [e[1].elapsed_time(e[2]) * 1e-3 for e in ev]
    ws.check()

    # ---- optional: the same step captured in a CUDA graph (one per input
    # copy) and replayed, timed with events around each replay
    t_graph = None
    if args.graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graphs = []
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            st_ = sets[c]
            with torch.cuda.graph(g, stream=side):
                run_step(st_["q_idx"], st_["head_w"], st_["q"], st_["pt"], st_["sl"], st_["cq"], c)
            graphs.append(g)
        stream.wait_stream(side)
        for i in range(args.warmup):
            graphs[i % copies].replay()
        barrier()
        g_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            g_ev[i][0].record(stream)
            graphs[(args.warmup + i) % copies].replay()
            g_ev[i][1].record(stream)
        barrier()
        t_graph = sum(e[0].elapsed_time(e[1]) * 1e-3 for e in g_ev)
        ws.check()

    # ---- end to end through the public API: every step copies its inputs
    # from pinned host memory to the device, runs the calls and copies its
    # output back to pinned host memory.  The steps are pipelined as a serving
    # loop runs them: one copy stream brings step i+1's inputs in and another
    # takes step i-1's output out while step i computes (two buffers of each).
    h_in = {k: v.pin_memory() for k, v in {"q_idx": q_idx.cpu(), "head_w": head_w.cpu(), "q": q.cpu(),
                                           "pt": pt.cpu(), "sl": sl.cpu(), "cq": cq.cpu()}.items()}
    d_in = [{k: torch.empty_like(v, device=dev) for k, v in h_in.items()} for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = h_out[0].numel() * h_out[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_steps(n, first_cache):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]

        def copy_in(i):
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[i - 2])  # step i-2 has finished reading this buffer
                for k in h_in:
                    d_in[i % 2][k].copy_(h_in[k], non_blocking=True)
                ev_in[i].record(s_in)

        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            between_steps()
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # step i-2's output has left this buffer
            b = d_in[i % 2]
            run_step(b["q_idx"], b["head_w"], b["q"], b["pt"], b["sl"], b["cq"], (first_cache + i) % copies,
                     out_buf=outs[i % 2])
            ev_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i])
                h_out[i % 2].copy_(outs[i % 2], non_blocking=True)
                ev_out[i].record(s_out)
        return ev_out[n - 1]

    e2e_steps(3, 0)
    barrier()
    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_start.record(s_in)
    last = e2e_steps(args.steps, 1)
    s_out.wait_event(last)
    e2e_end.record(s_out)
    barrier()
    clk = clocks.stop()
    e2e_total = e2e_start.elapsed_time(e2e_end) * 1e-3
    ws.check()

    # ---- max over ranks
    t_max, e2e_max = max_over_ranks([total, e2e_total], dev)
    if t_graph is not None:
        t_graph = max_over_ranks([t_graph], dev)[0]
    tokens = wl.T * args.steps

    if rank == 0:
        hbm, peak_kind = peaks()
        ib, mb = indexer_bytes(wl), mla_bytes(wl)
        ti, tm = statistics.mean(t_idx), statistics.mean(t_mla)
        kernels = {
            "indexer_topk": {"seconds_per_launch": ti, "algorithmic_bytes": ib, "achieved_gbs": ib / ti / 1e9,
                             "traffic": recorded_traffic("indexer_topk", "indexer_topk.cu")},
            "sparse_mla": {"seconds_per_launch": tm, "algorithmic_bytes": mb, "achieved_gbs": mb / tm / 1e9,
                           "traffic": recorded_traffic("sparse_mla", "sparse_mla.cu")},
        }
        dom = max(kernels, key=lambda k: kernels[k]["seconds_per_launch"])
        k = kernels[dom]
        line = {
            "metric": METRIC, "value": aggregate_rate(tokens, world, t_max), "unit": "tokens/s",
            "n_gpus": max(world, 1),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, random page permutation)", "config": cfg,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": k["achieved_gbs"], "peak": hbm,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": k["achieved_gbs"] / hbm,
                         "frac_of_nominal_8tbs": k["achieved_gbs"] / NOMINAL_HBM_GBS, "traffic": k["traffic"]},
            # the whole step (both kernels, overlapping as in use) against HBM:
            # the figure the 60 % target is stated for
            "step_roofline": {"bytes": ib + mb, "achieved_gbs": (ib + mb) / (t_max / args.steps) / 1e9,
                              "frac": (ib + mb) / (t_max / args.steps) / 1e9 / hbm,
                              "frac_of_nominal_8tbs": (ib + mb) / (t_max / args.steps) / 1e9 / NOMINAL_HBM_GBS},
            "kernels": kernels,
            "e2e": {"value": aggregate_rate(tokens, world, e2e_max), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "pipelining": "each step's copies on two copy streams, overlapping the neighbouring steps' kernels"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        if t_graph is not None:
            line["graph"] = {"value": aggregate_rate(tokens, world, t_graph), "unit": "tokens/s",
                             "ms_per_step": 1e3 * t_graph / args.steps,
                             "note": "the step captured once per input copy in a CUDA graph, replayed"}
        if world <= 1 and not args.no_workloads:
            line["workloads"] = other_workloads(args, dev)
        if world <= 1 and not args.no_cpu_baseline:
            rate, units, spent = oracle_rate(wl, 10.0, 16)
            line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                    "sample": f"{units} whole decode queries of this workload ({spent:.1f} s, "
                                              f"single-threaded C oracle, fp64)"}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
