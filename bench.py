#!/usr/bin/env python
"""Benchmark of the block-wise Sparse GQA prefill (merge + index + top-k +
union + attention) on GB300.

One step = one sgqa_prefill call over the whole workload (by default the
Step-5-shaped 128K prefill: 131072 queries, 64 query / 8 KV heads, d = 128,
B = 8, k = 4096, union tile 64).  Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle, timed on the host)

Timing: W untimed steps, then exactly K steps between CUDA events on the
launch stream, bracketed by a barrier and a device synchronise; the maximum
over ranks is reported.  The inputs (several GB) are larger than the 129 MB
L2, so no flush is needed between steps.  Multi-GPU runs are independent
replicas (each rank prefills its own copy of the workload; the path has no
exchange step), so scaling is weak and the value is the total over ranks.

End to end (`e2e`): the same K steps through the C ABI with every step's
inputs (Q, K, V) copied from pinned host memory and its outputs (O, lse)
copied back, pipelined as a serving loop would run them: two slots of device
buffers, the copies on their own streams, so step i's uploads overlap step
i-1's prefill and step i-2's downloads; events order each slot's reuse.  The
time runs from the first upload to the last download.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Sparse-GQA prefill tokens/s at 128K (merge+index+topk+attn) and % of roofline"
UNIT = "tokens/s"


# ----------------------------------------------------------------------------- setup
def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="step5_128k")
    ap.add_argument("--rho-q", type=float, default=None,
                    help="AR(1) correlation of the query noise (0 = i.i.d. stress case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-quality", action="store_true",
                    help="skip the union / recall / coverage report (computed after timing)")
    ap.add_argument("--index-mode", choices=["split", "bf16"], default="split",
                    help="indexer precision: fp32 scores from a bf16 split (exact selection) "
                         "or bf16 scores (one product; recall against split reported)")
    ap.add_argument("--decode", action="store_true",
                    help="time decode steps (one query at the end of the 1M paged cache) "
                         "through sgqa_decode with a persistent block-key cache, beside "
                         "sgqa_prefill on the same query; prints its own line")
    ap.add_argument("--no-bwd", action="store_true",
                    help="skip timing the attention backward on the workload's selection")
    ap.add_argument("--no-stress", action="store_true",
                    help="skip the i.i.d. query-noise run reported beside the headline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--seq", type=int, default=None,
                    help="shrink the workload to this many queries (profiling small cases)")
    ap.add_argument("--tile-q", type=int, default=None,
                    help="union tile size (queries) instead of the workload's")
    ap.add_argument("--union-mode", choices=["masked", "full"], default="masked",
                    help="masked: each query attends its own selection; full: the tile's union")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29531")
        dist.init_process_group(backend)


def reduce_max(x: float, device=None) -> float:
    """Maximum of a float over all ranks (the identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained", m["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(1.0)  # let nvidia-smi attach before the timed region starts
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9 or not parts[0].isdigit():
                    continue
                if int(parts[0]) != self.gpu_index:
                    continue
                rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if _isnum(r[3])), default=None)}


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


# ----------------------------------------------------------------------------- algorithmic work
def algorithmic(wl, chunk: int):
    """Closed-form algorithmic work of one prefill (mode A):
      indexer FLOPs  = Hkv * sum_t nh(t) * 2d          (each scored pair once)
      attention FLOPs = H * sum_t (min(Ks, nh(t)) * B + pos(t) mod B + 1) * 4d
                        (QK^T and PV over each query's own keys, not the union)
      compulsory bytes = Q + O + lse + K read by the merge + Kbar write + read
                        + K and V read once.
    Also per-chunk attention and indexer FLOPs (one attention / indexer
    launch per chunk of `chunk` queries)."""
    T, off, B, d = wl.seq_q, wl.q_offset, wl.block_size, wl.head_dim
    H, Hkv, Ks = wl.n_q_heads, wl.n_kv_heads, wl.k_blocks
    t = np.arange(T, dtype=np.int64)
    pos = off + t
    nh = np.minimum(pos // B, wl.n_blocks)
    keys = np.minimum(Ks, nh) * B + pos % B + 1
    attn = H * keys * 4.0 * d
    idx = Hkv * nh * 2.0 * d
    e = 2 if wl.dtype == "bf16" else 4
    new_blocks = wl.n_blocks - off // B  # the prefix's block keys are cached (chunked prefill)
    byts = (2 * T * H * d * e + H * T * 4 + new_blocks * B * Hkv * d * e
            + 2 * wl.n_blocks * Hkv * d * 4 + 2 * wl.seq_kv * Hkv * d * e)
    nch = (T + chunk - 1) // chunk
    per_chunk = lambda a: [float(a[i * chunk:(i + 1) * chunk].sum()) for i in range(nch)]
    return {"attn_flops": float(attn.sum()), "index_flops": float(idx.sum()),
            "bytes": float(byts), "attn_flops_chunks": per_chunk(attn),
            "index_flops_chunks": per_chunk(idx)}


def traffic_from_profiles(kernel_file: str, workload: str):
    """dram bytes per launch recorded by a committed ncu summary, if the kernel
    source has not changed since (the summary carries the source's sha256)."""
    prof = os.path.join(ROOT, "profiles", f"{os.path.splitext(kernel_file)[0]}_{workload}.md")
    src = os.path.join(ROOT, "block_sparse_long_sgqa_gb300", "csrc", kernel_file)
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    text = open(prof).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not (m and h):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != h.group(1):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(wl, inp, budget_s: float):
    """Time the CPU oracle on a bounded sample of the workload: the full block
    merge, plus the per-query pipeline (index query, scores, top-k, attention)
    for a few spread contiguous query ranges.  Returns (tokens/s extrapolated
    to the whole workload, sample description, seconds spent)."""
    import oracle
    from block_sparse_long_sgqa_gb300 import synth

    Q = synth.widen(inp["Q"])
    K = synth.widen(inp["K"])
    V = synth.widen(inp["V"])
    t0 = time.perf_counter()
    Kbar = oracle.merge_f64(K, wl.block_size)
    t_merge = time.perf_counter() - t0

    def run_rows(n_ranges, per):
        T = wl.seq_q
        starts = np.linspace(0, T - per, n_ranges).astype(np.int64) if T > per else [0]
        t1 = time.perf_counter()
        n = 0
        for s0 in starts:
            s0 = int(s0)
            rows = np.arange(s0, min(T, s0 + per), dtype=np.int32)
            qt = oracle.index_query(Q, wl.n_kv_heads, rows)
            S = oracle.scores(qt, Kbar, wl.block_size, wl.q_offset, rows)
            sel = oracle.select(S, wl.block_size, wl.q_offset, rows, wl.k_blocks)
            # attention for these rows: a sub-problem with the same positions
            sub_off = wl.q_offset + s0
            oracle.sparse_attn(Q[s0:s0 + len(rows)], K, V, sub_off, wl.block_size, sel, 0,
                               W=wl.tile_q)
            n += len(rows)
        return n, time.perf_counter() - t1

    # two probes fit a cost per range (the sub-problem's set-up) and per row,
    # so the sample fills the budget
    n1, dt1 = run_rows(4, 1)
    n2, dt2 = run_rows(4, 8)
    per_row = max((dt2 - dt1) / max(n2 - n1, 1), 1e-6)
    per_range = max((dt1 - per_row * n1) / 4, 0.0)
    per = max(1, int((budget_s - 8 * per_range) / per_row / 8))
    n, dt = run_rows(8, per)
    total = t_merge + wl.seq_q * dt / n
    desc = (f"full block merge ({t_merge:.2f} s) + {n} queries in 8 spread ranges "
            f"({dt:.2f} s), extrapolated to {wl.seq_q} queries")
    return wl.seq_q / total, desc, t_merge + dt


# ----------------------------------------------------------------------------- main
def run_reference(args, wl, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    from block_sparse_long_sgqa_gb300 import synth

    if rank != 0:
        return None
    if args.union_mode != "masked":
        return {"impl": "reference",
                "unavailable": "the oracle sample times the masked union mode only"}
    inp = synth.make_inputs(wl, rho_q=args.rho_q)
    cores = len(os.sched_getaffinity(0))
    vals, desc = [], ""
    per_step = max(2.0, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        v, desc, _ = oracle_sample(wl, inp, per_step)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wl.seq_q / value * 1000.0, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc, "extrapolated": True},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


def quality(wl, inp, Q, K, V, pt, Kbar, lse, dev, nq_max=1024, index_mode=0):
    """Selection quality on the last nq_max queries (a whole number of tiles),
    through the C ABI and outside the timed region:
      union inflation |U| / min(k/B, nh) per (tile, group) of the standalone
      selection; needle recall (planted blocks found in each query's own
      selection); attention-mass coverage exp(lse_sparse - lse_dense) per
      (query, head), lse_sparse from the timed prefill and lse_dense from the
      same prefill with k covering every historical block."""
    import torch

    from block_sparse_long_sgqa_gb300 import sgqa

    W, B = wl.tile_q, wl.block_size
    nq = min(nq_max, wl.seq_q) // W * W
    if nq == 0:
        return None
    q0 = wl.seq_q - nq
    sub = wl.replace(seq_q=nq, q_offset=wl.q_offset + q0)
    ps = sgqa.params_for(sub, index_mode=index_mode)
    Qs = Q[q0:].contiguous()
    nblk = wl.seq_kv // B
    Ks = wl.topk_tokens // B
    st = sgqa.new_status(dev)

    def select_sub(p_):
        sc = torch.empty(wl.n_kv_heads, nq, nblk, device=dev)
        sgqa.sgqa_index_scores(p_, Qs, Kbar, 0, nq, sc,
                               sgqa.alloc_workspace(p_, sgqa.WS_INDEX_SCORES, dev))
        sl = torch.empty(wl.n_kv_heads, nq, Ks, dtype=torch.int32, device=dev)
        u_ = sgqa.alloc_union(p_, dev)
        sgqa.sgqa_topk_union(p_, sc, 0, nq, sl, *u_, status=st)
        return sl, u_

    sel, (uo, ul, ub, um) = select_sub(ps)
    t = np.arange(q0, wl.seq_q)
    nh = np.minimum((wl.q_offset + t) // B, nblk)
    tiles = np.arange(nq // W)
    kcap = np.minimum(Ks, nh[tiles * W + W - 1])  # the tile's last query has the most blocks
    infl = (ul.cpu().numpy().reshape(wl.n_kv_heads, -1)[:, :len(tiles)] / np.maximum(kcap, 1))
    out = {"queries": f"last {nq}", "union_inflation_mean": float(infl.mean()),
           "union_inflation_p99": float(np.percentile(infl, 99))}
    if index_mode == sgqa.INDEX_BF16:  # recall of the exact (split) selection
        ref_sel, _ = select_sub(sgqa.params_for(sub))
        a, b = ref_sel.cpu().numpy(), sel.cpu().numpy()
        hit = sum(len(np.intersect1d(a[g, r][a[g, r] >= 0], b[g, r]))
                  for g in range(a.shape[0]) for r in range(a.shape[1]))
        out["recall_vs_split_index"] = hit / max(1, int((a >= 0).sum()))
    if "needles" in inp:
        seln = sel.cpu().numpy()
        nd = inp["needles"]
        found = total = 0
        for i in range(nq):
            tau = (q0 + i) // W
            for g in range(wl.n_kv_heads):
                js = nd[tau, g][nd[tau, g] >= 0]
                js = js[js < nh[i]]
                total += len(js)
                found += int(np.isin(js, seln[g, i]).sum())
        out["needle_recall"] = found / total if total else None
    del sel
    # dense reference: every historical block selected
    dense = sub.replace(topk_tokens=nblk * B)
    pd = sgqa.params_for(dense, index_mode=index_mode)
    Od, lsed = sgqa.alloc_outputs(pd, dev)
    Kb = sgqa.kbar_empty(pd, dev)
    sgqa.sgqa_prefill(pd, Qs, K, V, Kb, Od, lsed, sgqa.alloc_workspace(pd, sgqa.WS_PREFILL, dev),
                      page_table=pt, status=st)
    code, det = sgqa.read_status(st)
    if code != 0:
        raise RuntimeError(f"device status in the quality report: {sgqa.status_string(code)} ({det})")
    cov = torch.exp(lse[:, q0:].double() - lsed.double()).cpu().numpy()
    out["coverage_mean"] = float(cov.mean())
    out["coverage_p1"] = float(np.percentile(cov, 1))
    return out


def time_backward(wl, p, Q, K, V, pt, Kbar, alg, tensor_peak, dev, steps=3):
    """The attention's forward alone and its backward (sgqa_sparse_attn_bwd)
    on the union lists of the whole workload (built by the step entry points
    on ranges of 4096 queries), with a seeded upstream gradient dO; CUDA
    events on the launch stream.  Algorithmic FLOPs: the forward's two
    products over each query's own keys, the backward's five (S, dP, dV, dK,
    dQ: 2.5 times the forward)."""
    import torch

    from block_sparse_long_sgqa_gb300 import sgqa

    u = sgqa.alloc_union(p, dev)
    nblk = wl.seq_kv // wl.block_size
    st = sgqa.new_status(dev)
    ws_t = sgqa.alloc_workspace(p, sgqa.WS_TOPK_UNION, dev)
    ws_i = sgqa.alloc_workspace(p, sgqa.WS_INDEX_SCORES, dev)
    for q0 in range(0, wl.seq_q, 4096):
        q1 = min(wl.seq_q, q0 + 4096)
        sc = torch.empty(wl.n_kv_heads, q1 - q0, nblk, device=dev)
        sgqa.sgqa_index_scores(p, Q, Kbar, q0, q1, sc, ws_i)
        sgqa.sgqa_topk_union(p, sc, q0, q1, None, *u, ws=ws_t, status=st)
        del sc
    del ws_t, ws_i
    O2, lse2 = sgqa.alloc_outputs(p, dev)
    ws_f = sgqa.alloc_workspace(p, sgqa.WS_SPARSE_ATTN, dev)
    ws_b = sgqa.alloc_workspace(p, sgqa.WS_ATTN_BWD, dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(20261299)
    dO = torch.randn(O2.shape, generator=gen, device=dev).to(torch.bfloat16)
    dQ = torch.empty(O2.shape, dtype=torch.float32, device=dev)
    dK = torch.empty(wl.seq_kv, wl.n_kv_heads, wl.head_dim, dtype=torch.float32, device=dev)
    dV = torch.empty_like(dK)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        sgqa.sgqa_sparse_attn_fwd(p, Q, K, V, *u, O2, lse2, page_table=pt, ws=ws_f, status=st)

    def bwd():
        sgqa.sgqa_sparse_attn_bwd(p, Q, K, V, *u, O2, lse2, dO, dQ, dK, dV, ws_b, page_table=pt,
                                  status=st)

    out = {}
    for name, fn in (("forward", fwd), ("backward", bwd)):
        fn()
        torch.cuda.synchronize(dev)
        log = sgqa.launch_log(steps * 16)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with log:
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
        out[name] = {"ms": e0.elapsed_time(e1) / steps, "launches": log.entries()}
    code, det = sgqa.read_status(st)
    if code != 0:
        raise RuntimeError(f"device status in the backward timing: {sgqa.status_string(code)} ({det})")
    f_fwd = alg["attn_flops"]
    bl = [t for k, t in out["backward"]["launches"] if k == sgqa.K_ATTN_BWD]
    res = {"workload": "the prefill's own selection (whole-call union lists), seeded dO",
           "fwd_attn_ms": out["forward"]["ms"], "bwd_ms": out["backward"]["ms"],
           "bwd_flops_alg": 2.5 * f_fwd,
           "bwd_tflops_alg": 2.5 * f_fwd / (out["backward"]["ms"] * 1e-3) / 1e12,
           "fwd_tflops_alg": f_fwd / (out["forward"]["ms"] * 1e-3) / 1e12,
           "peak_tflops": tensor_peak}
    res["bwd_frac"] = res["bwd_tflops_alg"] / tensor_peak
    res["fwd_frac"] = res["fwd_tflops_alg"] / tensor_peak
    if len(bl) >= 2 * steps:  # per call: the dQ kernel, then the dK/dV kernel
        res["dq_ms"] = sum(bl[0::2]) / steps
        res["dkv_ms"] = sum(bl[1::2]) / steps
    return res


def run_decode(args, dev):
    """Decode steps over the 1M paged cache: the block-key cache is built by
    the first call, then each timed step is one query at the last position
    (the cache already holds every complete block)."""
    import torch

    from block_sparse_long_sgqa_gb300 import sgqa, synth

    base = synth.WORKLOADS["chunk_1m"]
    pos = base.seq_kv - 1
    wl = base.replace(name="decode_1m", seq_q=1, q_offset=pos)
    inp = synth.make_inputs(wl)
    p = sgqa.params_for(wl)
    Kh = synth.to_paged(inp["K"], inp["page_table"], wl.page_size)
    Vh = synth.to_paged(inp["V"], inp["page_table"], wl.page_size)
    tod = lambda x: torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    Q, K, V = tod(inp["Q"]), tod(Kh), tod(Vh)
    pt = torch.from_numpy(inp["page_table"]).to(dev)
    O, lse = sgqa.alloc_outputs(p, dev)
    st = sgqa.new_status(dev)
    cache = sgqa.KeyCache(p, cap_blocks=wl.n_blocks, device=dev)
    ws = sgqa.alloc_workspace(p, sgqa.WS_DECODE, dev)
    sgqa.sgqa_decode(p, Q, K, V, cache, O, lse, ws, page_table=pt, status=st)  # builds the cache
    Kbar = cache.Kbar.clone()
    wsp = sgqa.alloc_workspace(p, sgqa.WS_PREFILL, dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, fn in (("decode", lambda: sgqa.sgqa_decode(p, Q, K, V, cache, O, lse, ws,
                                                         page_table=pt, status=st)),
                     ("prefill_one_query", lambda: sgqa.sgqa_prefill(
                         p, Q, K, V, Kbar, O, lse, wsp, page_table=pt,
                         kbar_valid_blocks=wl.n_blocks, status=st))):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize(dev)
        log = sgqa.launch_log(args.steps * 64)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with log:
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
        per = {}
        for kind, t_ms in log.entries():
            nm = sgqa.KERNEL_NAMES.get(kind, str(kind))
            per[nm] = per.get(nm, 0.0) + t_ms / args.steps
        out[name] = {"ms_per_step": e0.elapsed_time(e1) / args.steps, "kernels_ms": per}
    code, det = sgqa.read_status(st)
    if code != 0:
        raise RuntimeError(f"device status in the decode timing: {sgqa.status_string(code)} ({det})")
    return {"metric": "decode step latency, one query over a 1M-token paged cache",
            "unit": "ms", "higher_is_better": False, "steps": args.steps,
            "config": {"workload": wl.name, "seq_kv": wl.seq_kv, "n_q_heads": wl.n_q_heads,
                       "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
                       "block_size": wl.block_size, "topk_tokens": wl.topk_tokens,
                       "page_size": wl.page_size},
            **out}


def config_of(wl, args):
    return {"workload": wl.name, "seq_q": wl.seq_q, "seq_kv": wl.seq_kv, "q_offset": wl.q_offset,
            "n_q_heads": wl.n_q_heads, "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size, "topk_tokens": wl.topk_tokens, "tile_q": wl.tile_q,
            "page_size": wl.page_size, "union_mode": args.union_mode,
            "index_mode": args.index_mode,
            "inputs": f"seeded {wl.dist}" + (f", AR(1) query noise rho={wl.rho_q if args.rho_q is None else args.rho_q}"
                                              if wl.dist == "clustered" else "")
                      + (f", {wl.needles} needle blocks per tile" if wl.needles else ""),
            "l2": "inputs larger than L2 (no flush between steps)",
            "parallelism": f"replicas x{args.gpus}"}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    from block_sparse_long_sgqa_gb300 import synth

    wl = synth.WORKLOADS[args.workload]
    if args.seq:
        wl = wl.replace(seq_q=args.seq, seq_kv=wl.q_offset + args.seq)
    if args.tile_q:
        wl = wl.replace(tile_q=args.tile_q)
    if args.impl == "reference":
        line = run_reference(args, wl, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    import torch

    from block_sparse_long_sgqa_gb300 import sgqa

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    if args.decode:
        if rank == 0:
            print(json.dumps(run_decode(args, dev)), flush=True)
        return 0
    index_mode = sgqa.INDEX_BF16 if args.index_mode == "bf16" else sgqa.INDEX_SPLIT
    p = sgqa.params_for(wl, union_mode=1 if args.union_mode == "full" else 0,
                        index_mode=index_mode)
    chunk, launches = sgqa.sgqa_prefill_plan(p)

    t_gen = time.perf_counter()
    inp = synth.make_inputs(wl, rho_q=args.rho_q)
    t_gen = time.perf_counter() - t_gen

    def to_dev(x):
        t = torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x)
        t = t.to(dev)
        return t.view(torch.bfloat16) if x.dtype == np.uint16 else t

    Kh, Vh = inp["K"], inp["V"]
    if wl.page_size:
        Kh = synth.to_paged(Kh, inp["page_table"], wl.page_size)
        Vh = synth.to_paged(Vh, inp["page_table"], wl.page_size)
    Q, K, V = to_dev(inp["Q"]), to_dev(Kh), to_dev(Vh)
    pt = torch.from_numpy(inp["page_table"]).to(dev) if wl.page_size else None
    O, lse = sgqa.alloc_outputs(p, dev)
    ws = sgqa.alloc_workspace(p, sgqa.WS_PREFILL, dev)
    st = sgqa.new_status(dev)
    stream = torch.cuda.current_stream(dev)

    # a chunked prefill at 1M: the block keys of the cached prefix exist already
    kvalid = 0
    Kbar = sgqa.kbar_empty(p, dev)
    if wl.q_offset > 0:
        kvalid = wl.q_offset // wl.block_size
        sgqa.sgqa_block_merge(p, K, Kbar, 0, kvalid, page_table=pt)

    def step():
        sgqa.sgqa_prefill(p, Q, K, V, Kbar, O, lse, ws, page_table=pt, kbar_valid_blocks=kvalid,
                          status=st)

    for _ in range(max(args.warmup, 0)):
        step()
    code, detail = sgqa.read_status(st)
    if code != 0:
        raise RuntimeError(f"device status after warm-up: {sgqa.status_string(code)} ({detail})")

    # ---------------- timed region (device-resident inputs)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip().isdigit()]
    gpu_index = int(ids[local]) if local < len(ids) else local
    log = sgqa.launch_log(args.steps * (launches + 4))
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_index) as clk, log:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    code, detail = sgqa.read_status(st)
    if code != 0:
        raise RuntimeError(f"device status after timing: {sgqa.status_string(code)} ({detail})")
    ms_max = reduce_max(ms, dev)
    n_launch = int(reduce_sum(log.count, dev))
    clocks = clk.summary()

    # ---------------- per-kernel durations from the launch log
    alg = algorithmic(wl, chunk)
    peaks = measured_peaks()
    per_kind = {}
    for kind, t_ms in log.entries():
        per_kind.setdefault(kind, []).append(t_ms)
    total_logged = sum(sum(v) for v in per_kind.values())
    kernels = {}
    for kind, ts in per_kind.items():
        name = sgqa.KERNEL_NAMES.get(kind, str(kind))
        kernels[name] = {"launches_per_step": len(ts) / args.steps,
                         "ms_per_step": sum(ts) / args.steps,
                         "share": sum(ts) / total_logged if total_logged else None}
    tensor_peak = peaks["bf16_tflops_sustained"]
    if sgqa.K_ATTN in per_kind:
        k = kernels["sparse_attn"]
        k["achieved_tflops"] = alg["attn_flops"] / (k["ms_per_step"] * 1e-3) / 1e12
        k["frac"] = k["achieved_tflops"] / tensor_peak
    if sgqa.K_INDEX_SCORES in per_kind:
        k = kernels["index_scores"]
        k["achieved_tflops"] = alg["index_flops"] / (k["ms_per_step"] * 1e-3) / 1e12
        k["frac"] = k["achieved_tflops"] / tensor_peak
    if sgqa.K_TOPK_UNION in per_kind:
        # long rows select from the indexer's threshold candidates, not from
        # score rows, so this kernel class is reported in rows per second
        k = kernels["topk_union"]
        k["rows_per_s"] = wl.n_kv_heads * wl.seq_q / (k["ms_per_step"] * 1e-3)
    dominant = max(kernels, key=lambda n: kernels[n]["ms_per_step"])
    dk = kernels[dominant]
    src_of = {"sparse_attn": "attn.cu", "index_scores": "index_gemm.cu",
              "topk_union": "topk_union.cu", "tile_union": "topk_union.cu", "merge": "merge.cu"}
    traffic = traffic_from_profiles(src_of.get(dominant, ""), wl.name)
    if dominant in ("sparse_attn", "index_scores"):
        roofline = {"kernel": dominant, "bound": "tensor", "achieved": dk["achieved_tflops"],
                    "peak": tensor_peak, "unit": "TFLOP/s", "frac": dk["frac"],
                    "traffic": traffic,
                    "peak_source": f"bf16_tflops_sustained of {peaks['source']}"}
    else:
        ach = dk.get("achieved_gbs")
        roofline = {"kernel": dominant, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": (ach / peaks["hbm_gbs"]) if ach else None,
                    "traffic": traffic, "peak_source": f"hbm_gbs of {peaks['source']}"}
    f_alg = alg["attn_flops"] + alg["index_flops"]
    t_roof = max(f_alg / (tensor_peak * 1e12), alg["bytes"] / (peaks["hbm_gbs"] * 1e9))
    step_roof = {"flops_alg": f_alg, "bytes_alg": alg["bytes"], "t_roof_ms": t_roof * 1e3,
                 "frac": t_roof * 1e3 / ms, "peak_tflops": tensor_peak,
                 "peak_gbs": peaks["hbm_gbs"], "of": peaks["source"]}

    # ---------------- end to end through the C ABI from pinned host memory
    e2e = None
    if not args.no_e2e:
        hQ = torch.from_numpy(inp["Q"].view(np.int16) if inp["Q"].dtype == np.uint16
                              else inp["Q"]).pin_memory()
        hK = torch.from_numpy(Kh.view(np.int16) if Kh.dtype == np.uint16 else Kh).pin_memory()
        hV = torch.from_numpy(Vh.view(np.int16) if Vh.dtype == np.uint16 else Vh).pin_memory()
        hO = torch.empty(O.numel(), dtype=torch.int16 if O.dtype == torch.bfloat16 else torch.float32).pin_memory()
        hl = torch.empty(lse.numel(), dtype=torch.float32).pin_memory()
        as16 = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t
        # A serving loop's pipeline: two slots of device inputs and outputs;
        # step i's host-to-device copies (copy stream) run while step i-1
        # computes (the compute stream) and step i-2's results return (a
        # third stream).  Events order each slot's reuse: its inputs are
        # overwritten only after the step that read them has computed, its
        # outputs only after they have been copied back.
        slots = [(Q, K, V, O, lse),
                 (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V),
                  torch.empty_like(O), torch.empty_like(lse))]
        hOs = [hO, torch.empty_like(hO).pin_memory()]
        hls = [hl, torch.empty_like(hl).pin_memory()]
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        in_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]
        # per-step spans of the three streams' work (each starts once its waits
        # are met): where the end-to-end time goes
        spans = None

        def mark(s):
            if spans is None:
                return None
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(s)
            return ev

        def e2e_step(i):
            b = i & 1
            Qb, Kb, Vb, Ob, lb = slots[b]
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(comp_done[b])
                a0 = mark(s_in)
                as16(Qb).view(-1).copy_(hQ.view(-1), non_blocking=True)
                as16(Kb).view(-1).copy_(hK.view(-1), non_blocking=True)
                as16(Vb).view(-1).copy_(hV.view(-1), non_blocking=True)
                in_done[b].record(s_in)
                a1 = mark(s_in)
            stream.wait_event(in_done[b])
            if used[b]:
                stream.wait_event(out_done[b])
            c0 = mark(stream)
            sgqa.sgqa_prefill(p, Qb, Kb, Vb, Kbar, Ob, lb, ws, page_table=pt,
                              kbar_valid_blocks=kvalid, status=st, stream=stream)
            comp_done[b].record(stream)
            c1 = mark(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                d0 = mark(s_out)
                hOs[b].copy_(as16(Ob).view(-1), non_blocking=True)
                hls[b].copy_(lb.view(-1), non_blocking=True)
                out_done[b].record(s_out)
                d1 = mark(s_out)
            used[b] = True
            if spans is not None:
                spans.append((a0, a1, c0, c1, d0, d1))

        for i in range(max(2, min(args.warmup, 2))):
            e2e_step(i)
        barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(args.steps):
            e2e_step(i)
        s_out.wait_event(comp_done[(args.steps - 1) & 1])
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, dev)
        h2d = (hQ.numel() + hK.numel() + hV.numel()) * hQ.element_size()
        d2h = hO.numel() * hO.element_size() + hl.numel() * 4
        e2e = {"value": world * wl.seq_q / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms}
        # a second, untimed pass with per-stream events: the uploads', the
        # prefill's and the downloads' own durations while the three overlap
        spans = []
        for i in range(min(args.steps, 8)):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        if spans:
            mean = lambda j: statistics.mean(x[j].elapsed_time(x[j + 1]) for x in spans)
            h_ms, c_ms, d_ms = mean(0), mean(2), mean(4)
            e2e["overlap"] = {"steps": len(spans), "h2d_ms": h_ms, "prefill_ms": c_ms, "d2h_ms": d_ms,
                              "h2d_gbs": h2d / (h_ms * 1e-3) / 1e9,
                              "d2h_gbs": d2h / (d_ms * 1e-3) / 1e9}

    # ---------------- a chunked prefill's cached prefix: its merge timed alone
    # (the timed steps merge only the chunk's new blocks)
    full_merge = None
    if rank == 0 and kvalid > 0:
        Kb2 = sgqa.kbar_empty(p, dev)
        sgqa.sgqa_block_merge(p, K, Kb2, 0, wl.n_blocks, page_table=pt)
        torch.cuda.synchronize(dev)
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        m0.record(stream)
        for _ in range(reps):
            sgqa.sgqa_block_merge(p, K, Kb2, 0, wl.n_blocks, page_table=pt)
        m1.record(stream)
        torch.cuda.synchronize(dev)
        mms = m0.elapsed_time(m1) / reps
        nbytes = (wl.n_blocks * wl.block_size * wl.n_kv_heads * wl.head_dim * (2 if wl.dtype == "bf16" else 4)
                  + wl.n_blocks * wl.n_kv_heads * wl.head_dim * 4)
        gbs = nbytes / (mms * 1e-3) / 1e9
        full_merge = {"blocks": wl.n_blocks, "ms": mms, "bytes": nbytes, "achieved_gbs": gbs,
                      "frac": gbs / peaks["hbm_gbs"], "peak_source": f"hbm_gbs of {peaks['source']}"}
        del Kb2

    # ---------------- selection quality (rank 0, after timing)
    qual = None
    if rank == 0 and not args.no_quality:
        qual = quality(wl, inp, Q, K, V, pt, Kbar, lse, dev, index_mode=index_mode)

    # ---------------- attention backward on the workload's own selection
    bwd = None
    if (rank == 0 and not args.no_bwd and wl.dtype == "bf16" and wl.block_size >= 8
            and args.index_mode == "split"):
        bwd = time_backward(wl, p, Q, K, V, pt, Kbar, alg, tensor_peak, dev)

    # ---------------- the literal input reading (rank 0, after the headline)
    # The headline's query noise is AR(1) along the sequence (rho 0.99); the
    # workload text's "N(0,1) noise" read literally is i.i.d. (rho 0), which
    # makes adjacent queries' selections overlap far less, so the unions and
    # the attention's gathered keys grow.  Timed the same way on a few steps.
    stress = None
    if (rank == 0 and not args.no_stress and wl.dist == "clustered"
            and (args.rho_q is None or args.rho_q != 0.0)):
        inp0 = synth.make_inputs(wl, rho_q=0.0)
        Q.copy_(to_dev(inp0["Q"]))
        step()
        n_st = 3
        log0 = sgqa.launch_log(n_st * (launches + 4))
        torch.cuda.synchronize(dev)
        with log0:
            ev0.record(stream)
            for _ in range(n_st):
                step()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
        code, detail = sgqa.read_status(st)
        if code != 0:
            raise RuntimeError(f"device status in the stress run: {sgqa.status_string(code)} ({detail})")
        ms0 = ev0.elapsed_time(ev1) / n_st
        per0 = {}
        for kind, t_ms in log0.entries():
            name = sgqa.KERNEL_NAMES.get(kind, str(kind))
            per0[name] = per0.get(name, 0.0) + t_ms / n_st
        stress = {"rho_q": 0.0, "steps": n_st, "ms_per_step": ms0,
                  "tokens_per_s": wl.seq_q / (ms0 * 1e-3),
                  "kernels_ms_per_step": per0,
                  "step_roofline_frac": t_roof * 1e3 / ms0}
        if not args.no_quality:
            q0 = quality(wl, inp0, Q, K, V, pt, Kbar, lse, dev, index_mode=index_mode)
            if q0:
                stress.update({k: q0[k] for k in ("union_inflation_mean", "union_inflation_p99",
                                                   "needle_recall", "coverage_mean") if k in q0})

    # ---------------- CPU baseline (rank 0, single GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and args.union_mode == "masked":
        v, desc, _ = oracle_sample(wl, inp, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": desc, "extrapolated": True}

    if rank == 0:
        line = {"metric": METRIC, "value": world * wl.seq_q / (ms_max * 1e-3), "unit": UNIT,
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
                "data": "synthetic", "config": config_of(wl, args), "clocks": clocks,
                "e2e": e2e, "gpu_launches": n_launch, "roofline": roofline,
                "full_cache_merge": full_merge,
                "step_roofline": step_roof, "kernels": kernels, "quality": qual,
                "backward": bwd, "stress_iid_query_noise": stress, "cpu_baseline": cpu,
                "input_gen_s": round(t_gen, 2)}
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
