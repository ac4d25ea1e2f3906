"""Benchmark: one shard of round-robin sequence-sharded DSA prefill attention on GB300.

Workload (default): the varlen batch {8000, 800, 5, 3000} tokens, sp = 8, shard rank 3
(1,476 queries); indexer 64 heads x 128, top-k 2048; MLA 128 heads, qk 576 / v 512, bf16.
A step is one pass of the whole shard path through the C ABI:
  split metadata + the shard's row gather -> rerange of the all-gathered k_idx and latent rows
  -> indexer scores + top-k -> sparse MLA.
The other shards' rows are inputs (one GPU, no collective). With --gpus N (torchrun), GPU i
takes shard (3 + i) % 8 of the same batch: independent problems, weak scaling.

value = shard queries processed / device time of the timed steps (CUDA events on the launch
stream, L2 flushed between steps); e2e = the same through host buffers: every step copies its
inputs from pinned host memory and reads o back, inside the timed region, pipelined over two
buffer sets and three streams (upload of step i + 1 and download of step i - 1 overlap step i).
--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "shard prefill query tokens/s (indexer+top-k+sparse MLA); % of BF16 TC roofline"
WORKLOAD_ID = 1
BASE_RANK = 3


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16": float(d["bf16_tflops"]), "bf16_sustained": float(d["bf16_tflops_sustained"]),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def profiled_traffic(kernel_file, summary):
    """DRAM bytes per launch from a committed ncu summary, only while the kernel source is the
    one that was profiled (its sha1 prefix is recorded next to the figure); else None."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "deepseek_v3_sparse_round_gb300", "csrc", kernel_file), "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()[:12]
        fields = {}
        with open(os.path.join(ROOT, "profiles", summary), encoding="utf-8") as f:
            for line in f:
                if ":" in line and line.split(":")[0].strip() in ("traffic_bytes_per_launch", "source_sha1"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha1") == sha:
            return int(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


def shard_for_rank(rank: int, sp: int) -> int:
    """GPU `rank` of the job processes shard (BASE_RANK + rank) % sp of the varlen batch."""
    return (BASE_RANK + rank) % sp


def max_over_ranks(value: float, dist, device) -> float:
    """The job's time is the slowest rank's: all-reduce MAX (no-op without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples every INTERVAL_MS, each stamped with its arrival time
    so that only the samples taken inside the timed window are summarised."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.stamped = []
        self.window = (0.0, float("inf"))

    def _reader(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.stamped.append((time.perf_counter(), ln))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def mark(self, t0, t1):
        self.window = (t0, t1 + self.INTERVAL_MS / 1e3)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
        t0, t1 = self.window
        self.lines = [ln for t, ln in self.stamped if t0 <= t <= t1]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm
class ShardStep:
    """Device buffers and the launches of one step for shard `rank` of the varlen workload."""

    def __init__(self, torch, dsa, W, rank, device):
        self.torch, self.dsa = torch, dsa
        wl = W.WORKLOADS[WORKLOAD_ID]
        self.wl, self.rank, self.dev = wl, rank, device
        cu_np = W.cu_seqlens(wl.lengths)
        self.N = int(cu_np[-1])
        self.n_req = len(wl.lengths)
        self.n_r = dsa.dsa_rr_shard_len(self.N, wl.sp, rank)
        self.max_ctx = int(max(wl.lengths))
        idx = W.indexer_inputs(wl, self.n_r, self.N, rank)
        mi = W.mla_inputs(wl, self.n_r, self.N, rank)
        # host inputs (pinned): the shard's queries, and the all-gathered (rank-major) KV rows
        # that the other shards contribute; built by plain indexing of the logical rows.
        perm = np.concatenate([np.arange(q, self.N, wl.sp) for q in range(wl.sp)])
        self.h = {
            "cu": torch.as_tensor(cu_np).pin_memory(),
            "q_idx": idx.q_idx.pin_memory(), "w": idx.w.pin_memory(), "q": mi.q.pin_memory(),
            "k_gath": idx.k_idx[torch.as_tensor(perm)].contiguous().pin_memory(),
            "c_gath": mi.c[torch.as_tensor(perm)].contiguous().pin_memory(),
            "c_log": mi.c.pin_memory(),
        }
        self.d = {k: v.to(device) for k, v in self.h.items()}
        e = lambda *s, dt=torch.int32: torch.empty(*s, dtype=dt, device=device)
        self.cu_shard, self.pos, self.bid, self.gidx = e(self.n_req + 1), e(self.n_r), e(self.n_r), e(self.n_r)
        self.c_local = e(self.n_r, wl.dqk, dt=torch.bfloat16)
        self.k_idx = e(self.N, wl.Di, dt=torch.bfloat16)
        self.c = e(self.N, wl.dqk, dt=torch.bfloat16)
        self.ws = e(dsa.dsa_indexer_topk_workspace_size(self.n_r, self.max_ctx, wl.topk), dt=torch.uint8)
        self.topk = e(self.n_r, wl.topk)
        self.o = e(self.n_r, wl.H, wl.dv, dt=torch.bfloat16)
        self.lse = e(self.n_r, wl.H, dt=torch.float32)
        self.mla_ws = e(dsa.dsa_sparse_mla_workspace_size(self.n_r), dt=torch.uint8)
        # split (metadata + row gather: one launch), 2 reranges, indexer plan + indexer, top-k,
        # MLA schedule + MLA (as the ncu launch list of a step shows)
        self.launches_per_step = 8
        self.h_o = [torch.empty(self.o.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        # second input / output set for the end-to-end pipeline (step i + 1 uploads while step i runs)
        self.d_sets = [self.d, {k: torch.empty_like(v) for k, v in self.d.items()}]
        self.o_sets = [self.o, torch.empty_like(self.o)]

    def run(self, ev=None, b=0):
        dsa, wl, d = self.dsa, self.wl, self.d_sets[b]
        dsa.dsa_rr_split_metadata(d["cu"], self.N, wl.sp, self.rank, self.cu_shard, self.pos,
                                  self.bid, self.gidx, src_rows=d["c_log"], dst_rows=self.c_local)
        dsa.dsa_rr_rerange(d["k_gath"], self.k_idx, self.N, wl.sp, 0)
        dsa.dsa_rr_rerange(d["c_gath"], self.c, self.N, wl.sp, 0)
        dsa.dsa_indexer_topk(d["q_idx"], d["w"], self.k_idx, d["cu"], self.n_req, self.pos,
                             self.bid, wl.topk, self.max_ctx, self.topk, self.ws)
        if ev is not None:
            ev[0].record()
        dsa.dsa_sparse_mla_balanced(d["q"], self.c, d["cu"], self.n_req, self.bid, self.pos,
                                    self.topk, wl.scale, self.o_sets[b], self.mla_ws,
                                    lse=self.lse)
        if ev is not None:
            ev[1].record()

    def upload(self, b=0):
        for k in ("cu", "q_idx", "w", "q", "k_gath", "c_gath", "c_log"):
            self.d_sets[b][k].copy_(self.h[k], non_blocking=True)

    def h2d_bytes(self):
        return sum(self.h[k].numel() * self.h[k].element_size()
                   for k in ("cu", "q_idx", "w", "q", "k_gath", "c_gath", "c_log"))

    def work(self):
        pos = self.pos.cpu().numpy().astype(np.int64)
        wl = self.wl
        sel = np.minimum(pos + 1, wl.topk)
        idx_flops = 2.0 * wl.Hi * wl.Di * float(np.sum(pos + 1))
        mla_flops = 2.0 * wl.H * (wl.dqk + wl.dv) * float(np.sum(sel))
        return idx_flops, mla_flops


def shard_balance(torch, dsa, W, device, wid=3):
    """Per-shard work of the many-request batch (32 requests, N = 71,014, sp = 4): queries and
    causal (query, key) pairs under the round-robin split, read from the library's split
    metadata on the GPU, and for comparison under the contiguous in-sequence split that cuts
    every request into sp chunks of ceil(L / sp) tokens. spread = (max - min) / mean."""
    wl = W.WORKLOADS[wid]
    cu_np = W.cu_seqlens(wl.lengths)
    n = int(cu_np[-1])
    cu = torch.as_tensor(cu_np, device=device)
    rr_q, rr_p = [], []
    for r in range(wl.sp):
        n_r = dsa.dsa_rr_shard_len(n, wl.sp, r)
        e = lambda m: torch.empty(m, dtype=torch.int32, device=device)
        pos = e(n_r)
        dsa.dsa_rr_split_metadata(cu, n, wl.sp, r, e(len(cu_np)), pos, e(n_r), e(n_r))
        p = pos.cpu().numpy().astype(np.int64)
        rr_q.append(int(n_r))
        rr_p.append(int(np.sum(p + 1)))
    is_q, is_p = [0] * wl.sp, [0] * wl.sp
    for length in wl.lengths:
        c = -(-int(length) // wl.sp)
        for q in range(wl.sp):
            lo, hi = q * c, min((q + 1) * c, int(length))
            if hi > lo:
                is_q[q] += hi - lo
                is_p[q] += (lo + 1 + hi) * (hi - lo) // 2      # sum of (p + 1) over [lo, hi)
    spread = lambda v: round((max(v) - min(v)) / (sum(v) / len(v)), 5)
    return {"workload": "many_req: 32 requests U[128,4096] (N=71,014), sp=4",
            "round_robin": {"queries": rr_q, "causal_pairs": rr_p, "pair_spread": spread(rr_p)},
            "in_seq": {"queries": is_q, "causal_pairs": is_p, "pair_spread": spread(is_p)}}


def gpu_arm(args):
    import torch
    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import __graft_entry__ as ge
    ge.build()
    import deepseek_v3_sparse_round_gb300 as dsa
    import workloads as W

    shard = shard_for_rank(rank, W.WORKLOADS[WORKLOAD_ID].sp)
    st = ShardStep(torch, dsa, W, shard, device)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)   # > L2
    stream = torch.cuda.current_stream()

    clk = ClockSampler(local).__enter__()            # running before the timed window opens
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    idx_flops, mla_flops = st.work()

    # ---- device-timed steps (inputs resident in HBM), L2 flushed between steps ----
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        evs[i][0].record(stream)
        st.run(ev=(evs[i][2], evs[i][3]))
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_end = time.perf_counter()
    wall = t_end - t_wall
    clk.mark(t_wall, t_end)
    clk.__exit__(None, None, None)
    step_ms = [a.elapsed_time(b) for a, b, _, _ in evs]
    mla_ms = [c.elapsed_time(d) for _, _, c, d in evs]
    dev_s = max_over_ranks(sum(step_ms) / 1e3, dist, device)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()

    # ---- end to end through host buffers: every step uploads its inputs from pinned host memory
    # and reads o back. Pipelined over two input/output sets and three streams (upload, compute,
    # download), so step i + 1's upload and step i - 1's download overlap step i.
    e2e_steps = max(2, min(args.steps, 20))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    s_in, s_run, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    mk = lambda: torch.cuda.Event()
    ev_in, ev_run, ev_out = ([mk() for _ in range(e2e_steps)] for _ in range(3))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_run.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(e2e_steps):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_run[i - 2])       # step i - 2 is done reading input set b
            st.upload(b)
            ev_in[i].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[i])
            if i >= 2:
                s_run.wait_event(ev_out[i - 2])      # o of step i - 2 has been read back
            st.run(b=b)
            ev_run[i].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[i])
            st.h_o[b].copy_(st.o_sets[b], non_blocking=True)
            ev_out[i].record(s_out)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, dist, device)

    errors = dsa.dsa_read_device_errors()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    pk = peaks()
    queries = st.n_r * ws
    value = queries * args.steps / dev_s
    mla_avg_s = float(np.mean(mla_ms)) / 1e3
    achieved = mla_flops / mla_avg_s / 1e12
    cpu = cpu_baseline(sample_queries=args.cpu_baseline_queries) if not args.no_cpu_baseline else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dev_s * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded bf16 N(0,1) queries/keys/latents; no weights needed)",
        "config": {"workload": "varlen {8000,800,5,3000} tokens, sp=8, shard rank 3 (+i per GPU): "
                               "1476 queries, indexer 64x128 top-2048, MLA 128 heads 576/512",
                   "queries_per_gpu": st.n_r, "kv_tokens": st.N, "topk": st.wl.topk,
                   "l2": "flushed between timed steps (256 MB write)",
                   "step": "split+gather, 2x rerange, indexer scores, top-k, sparse MLA"},
        "roofline": {"bound": "tensor", "kernel": "sparse_mla_pair_kernel",
                     "achieved": round(achieved, 1), "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": round(achieved / pk["bf16"], 4),
                     "traffic": profiled_traffic("mla.cu", "sparse_mla_pair_varlen_rank3.md"),
                     "peak_source": f"{pk['source']} bf16 burst (MEASURED_PEAKS.json)",
                     "algorithmic_flop_per_launch": mla_flops},
        "indexer_topk": {"algorithmic_flop_per_step": idx_flops},
        "e2e": {"value": round(queries * e2e_steps / e2e_s, 2), "unit": "tokens/s",
                "h2d_bytes_per_step": st.h2d_bytes(),
                "d2h_bytes_per_step": st.o.numel() * st.o.element_size()},
        "gpu_launches": st.launches_per_step * args.steps,
        "clocks": clk.summary(),
        "device_errors": errors,
        "wall_s_timed_region": round(wall, 4),
        "cpu_baseline": cpu,
        "shard_balance": shard_balance(torch, dsa, W, device),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle arm
def _oracle_step(W, wl, sh, sel):
    from oracle import indexer as oidx, mla as omla, topk as otopk
    from oracle.kv import ContiguousKV
    kv = ContiguousKV(sh["cu"])
    rows = oidx.indexer_scores(sh["q_idx"][sel], sh["w"][sel], sh["k_idx"], kv, sh["pos"][sel],
                               sh["bid"][sel])
    topk = otopk.topk_rows(rows, wl.topk)
    return omla.sparse_mla(sh["q"][sel], sh["c"], kv, sh["bid"][sel], topk, wl.scale, wl.dv)


def _oracle_inputs(n_sample):
    import workloads as W
    from oracle import split as osplit
    wl = W.WORKLOADS[WORKLOAD_ID]
    cu = W.cu_seqlens(wl.lengths)
    meta = osplit.round_robin_split(cu, wl.sp, BASE_RANK)
    n_r = len(meta["pos"])
    idx = W.indexer_inputs(wl, n_r, int(cu[-1]), BASE_RANK)
    mi = W.mla_inputs(wl, n_r, int(cu[-1]), BASE_RANK)
    # a bounded sample spread over the shard (every request, short and long histories)
    sel = np.unique(np.linspace(0, n_r - 1, n_sample).round().astype(np.int64))
    sh = {"cu": cu, "pos": meta["pos"], "bid": meta["bid"],
          "q_idx": idx.q_idx.float().numpy().astype(np.float64)[sel],
          "w": idx.w.numpy().astype(np.float64)[sel],
          "k_idx": idx.k_idx.float().numpy().astype(np.float64),
          "q": mi.q[sel].float().numpy().astype(np.float64),
          "c": mi.c.float().numpy().astype(np.float64)}
    sh["pos"], sh["bid"] = sh["pos"][sel], sh["bid"][sel]
    return W, wl, sh, n_r


def cpu_baseline(sample_queries=12, min_seconds=10.0, max_passes=6):
    """Passes of the oracle over the sample until at least `min_seconds` of CPU work (bounded
    by `max_passes`), so the figure rests on 10-30 s of work without stretching the bench."""
    W, wl, sh, n_r = _oracle_inputs(sample_queries)
    sel = np.arange(len(sh["pos"]))
    steps = 0
    t0 = time.perf_counter()
    while steps < max_passes and (steps == 0 or time.perf_counter() - t0 < min_seconds):
        _oracle_step(W, wl, sh, sel)
        steps += 1
    dt = time.perf_counter() - t0
    cores = _blas_threads()
    return {"value": round(len(sel) * steps / dt, 4), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(sel)} of the {n_r} rank-3 queries (evenly spaced, all requests), "
                      f"fp64 NumPy indexer + full-sort top-k + sparse MLA, {steps} pass(es), "
                      f"{dt:.1f} s"}


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    W, wl, sh, n_r = _oracle_inputs(args.cpu_sample)
    sel = np.arange(len(sh["pos"]))
    for _ in range(args.warmup):
        _oracle_step(W, wl, sh, sel[:1])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(W, wl, sh, sel)
    dt = time.perf_counter() - t0
    value = len(sel) * args.steps / dt
    cores = _blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "varlen {8000,800,5,3000} tokens, sp=8, shard rank 3: a bounded "
                               f"sample of {len(sel)} of its {n_r} queries per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{len(sel)} evenly spaced queries of the rank-3 shard per step"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def next_rows(args):
    """Separate measurements of the two widened rows (not part of the step): the rerange fused
    with the paged KV-cache write (HBM roofline, algorithmic bytes = 2 x rows x row bytes) and
    the decode-step split (launch bound). One JSON line per case; `--next-rows large` runs only
    the 1,048,576-row case (the one captured under ncu)."""
    import torch
    import __graft_entry__ as ge
    ge.build()
    import deepseek_v3_sparse_round_gb300 as dsa
    import workloads as W
    hbm = peaks()["hbm"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def timeit(fn, reps, do_flush):
        fn()
        torch.cuda.synchronize()
        ts = []
        for i in range(reps):
            if do_flush:
                flush.fill_(i & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    rng = np.random.default_rng(0)

    def paged_case(lengths, sp, width, page=64):
        cu = W.cu_seqlens(lengths)
        n = int(cu[-1])
        per = [(int(x) + page - 1) // page for x in lengths]
        total = sum(per)
        perm = rng.permutation(total + 8)[:total]          # pages scattered over the pool
        table = np.full((len(lengths), max(per)), -1, np.int32)
        k = 0
        for b, m in enumerate(per):
            table[b, :m] = perm[k:k + m]
            k += m
        gathered = torch.randn(n, width, device="cuda").to(torch.bfloat16)
        pool = torch.zeros((total + 8) * page, width, dtype=torch.bfloat16, device="cuda")
        dcu, dt = torch.as_tensor(cu, device="cuda"), torch.as_tensor(table, device="cuda")
        out = torch.empty_like(gathered)
        return (n, lambda: dsa.dsa_rr_rerange_paged(gathered, pool, n, sp, dcu, dt, 0, page),
                lambda: dsa.dsa_rr_rerange(gathered, out, n, sp, 0), 2 * n * width * 2)

    large = args.next_rows == "large"
    cases = [] if large else [("varlen {8000,800,5,3000}, sp=8", W.WORKLOADS[1].lengths, 8),
                              ("many_req (32 requests), sp=4", W.WORKLOADS[3].lengths, 4)]
    cases.append(("64 requests x 16384 tokens, sp=8", (16384,) * 64, 8))
    for name, lengths, sp in cases:
        for width in ((576,) if large else (576, 128)):
            n, f_paged, f_plain, nbytes = paged_case(lengths, sp, width)
            for kind, fn in (("rerange_paged", f_paged), ("rerange", f_plain))[:1 if large else 2]:
                ms = timeit(fn, 20, True)
                gbs = nbytes / ms / 1e6
                print(json.dumps({"kernel": kind, "workload": name, "row_bytes": width * 2,
                                  "rows": n, "us": round(ms * 1e3, 1), "GB/s": round(gbs),
                                  "frac_of_measured_hbm": round(gbs / hbm, 3),
                                  "l2": "flushed between launches"}), flush=True)
            torch.cuda.empty_cache()
    if not large:
        wl = W.WORKLOADS[4]
        q = wl.decode_queries
        ctx = np.asarray(wl.lengths, dtype=np.int64)
        cu_new = torch.as_tensor((np.arange(len(ctx) + 1) * q).astype(np.int32), device="cuda")
        base = torch.as_tensor((ctx - q).astype(np.int32), device="cuda")
        n = int(len(ctx) * q)
        for sp in (1, 8):
            n_r = dsa.dsa_rr_shard_len(n, sp, 0)
            e = lambda m: torch.empty(m, dtype=torch.int32, device="cuda")
            cs, p, b, g = e(len(ctx) + 1), e(n_r), e(n_r), e(n_r)
            src = torch.randn(n, 576, device="cuda").to(torch.bfloat16)
            dst = torch.empty(n_r, 576, dtype=torch.bfloat16, device="cuda")
            f = lambda: dsa.dsa_rr_split_decode_metadata(cu_new, base, n, sp, 0, cs, p, b, g, src, dst)
            eager = timeit(f, 100, False)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                f()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                f()
            replay = timeit(graph.replay, 100, False)
            print(json.dumps({"kernel": "split_decode (metadata + row gather)",
                              "workload": f"decode batch: {len(ctx)} requests x {q} new tokens, sp={sp}",
                              "rows_gathered": n_r, "us_eager": round(eager * 1e3, 2),
                              "us_graph_replay": round(replay * 1e3, 2)}), flush=True)
    print(json.dumps({"device_errors": dsa.dsa_read_device_errors()}), flush=True)


def config_rows(args):
    """The metric's steps (indexer + top-k + sparse MLA) on every workload config, one JSON line
    each: shard queries / device time (per shard the median of 20 launches after 3 warm-up, L2
    flushed before each; the shards of a config back to back), and the indexer's and the MLA's
    algorithmic TFLOP/s against the measured bf16 peak. For the paged decode batch also their
    algorithmic bytes (k_idx read once per request; the selected latent rows) against the
    measured copy bandwidth. Inputs are generated on the device; positions of prefill shards come
    from the library's own split."""
    import torch
    import __graft_entry__ as ge
    ge.build()
    import deepseek_v3_sparse_round_gb300 as dsa
    import workloads as W
    pk = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(parts, reps=20):
        for _ in range(3):
            for f in parts:
                f()
        t = [[] for _ in parts]
        for i in range(reps):
            flush.fill_(i & 255)
            es = [ev() for _ in range(len(parts) + 1)]
            es[0].record()
            for j, f in enumerate(parts):
                f()
                es[j + 1].record()
            torch.cuda.synchronize()
            for j in range(len(parts)):
                t[j].append(es[j].elapsed_time(es[j + 1]))
        return [float(np.median(x)) for x in t]

    def shard_inputs(wl, rank):
        if wl.decode_queries:
            table, n_pages = W.random_block_table(wl.lengths, wl.page_size,
                                                  W.seed_of(wl, "block_table"))
            bid, pos = W.decode_queries(wl.lengths, wl.decode_queries)
            n_rows = n_pages * wl.page_size
            cu = torch.zeros(len(wl.lengths) + 1, dtype=torch.int32, device="cuda")
            return dict(n_rows=n_rows, cu=cu, bt=torch.as_tensor(table, device="cuda"),
                        bid=torch.as_tensor(np.asarray(bid, np.int32), device="cuda"),
                        pos=torch.as_tensor(np.asarray(pos, np.int32), device="cuda"),
                        max_ctx=int(max(wl.lengths)))
        cu_np = W.cu_seqlens(wl.lengths)
        n_tok = int(cu_np[-1])
        n_r = dsa.dsa_rr_shard_len(n_tok, wl.sp, rank)
        cu = torch.as_tensor(cu_np, device="cuda")
        e = lambda m: torch.empty(m, dtype=torch.int32, device="cuda")
        cs, pos, bid, gidx = e(len(cu_np)), e(n_r), e(n_r), e(n_r)
        dsa.dsa_rr_split_metadata(cu, n_tok, wl.sp, rank, cs, pos, bid, gidx)
        return dict(n_rows=n_tok, cu=cu, bt=None, bid=bid, pos=pos, max_ctx=int(max(wl.lengths)))

    for wid in (1, 2, 3, 4):
        wl = W.WORKLOADS[wid]
        ranks = (0,) if wl.decode_queries else wl.ranks
        tot_q = tot_idx = tot_mla = 0.0
        idx_flop = mla_flop = idx_bytes = mla_bytes = 0.0
        for rank in ranks:
            si = shard_inputs(wl, rank)
            n_q = si["pos"].numel()
            idx = W.indexer_inputs(wl, n_q, si["n_rows"], rank, device="cuda")
            mi = W.mla_inputs(wl, n_q, si["n_rows"], rank, device="cuda")
            ws = torch.empty(dsa.dsa_indexer_topk_workspace_size(n_q, si["max_ctx"], wl.topk),
                             dtype=torch.uint8, device="cuda")
            mws = torch.empty(dsa.dsa_sparse_mla_workspace_size(n_q), dtype=torch.uint8,
                              device="cuda")
            topk = torch.empty((n_q, wl.topk), dtype=torch.int32, device="cuda")
            o = torch.empty((n_q, wl.H, wl.dv), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((n_q, wl.H), device="cuda")
            n_req = len(wl.lengths)
            f_idx = lambda: dsa.dsa_indexer_topk(idx.q_idx, idx.w, idx.k_idx, si["cu"], n_req,
                                                 si["pos"], si["bid"], wl.topk, si["max_ctx"],
                                                 topk, ws, block_table=si["bt"])
            f_mla = lambda: dsa.dsa_sparse_mla_balanced(mi.q, mi.c, si["cu"], n_req, si["bid"],
                                                        si["pos"], topk, wl.scale, o, mws,
                                                        lse=lse, block_table=si["bt"])
            t_idx, t_mla = timed([f_idx, f_mla])
            p = si["pos"].cpu().numpy().astype(np.int64)
            tot_q += n_q
            tot_idx += t_idx
            tot_mla += t_mla
            idx_flop += 2.0 * wl.Hi * wl.Di * float(np.sum(p + 1))
            sel = float(np.sum(np.minimum(p + 1, wl.topk)))
            mla_flop += 2.0 * wl.H * (wl.dqk + wl.dv) * sel
            if wl.decode_queries:
                idx_bytes = float(sum(wl.lengths)) * wl.Di * 2
                mla_bytes += sel * wl.dqk * 2
            if args.with_oracle and rank == ranks[-1]:
                or_q, or_s = _oracle_sample_time(W, wl, si, idx, mi, 16 if wl.decode_queries else 64)
            del idx, mi, ws, mws, topk, o, lse, si
            torch.cuda.empty_cache()
        ms = tot_idx + tot_mla
        line = {"config": wid, "workload": wl.name, "shards": len(ranks), "queries": int(tot_q),
                "ms": round(ms, 4), "tokens_per_s": round(tot_q / (ms * 1e-3), 1),
                "indexer_topk_ms": round(tot_idx, 4), "mla_ms": round(tot_mla, 4),
                "indexer_topk_tflops": round(idx_flop / (tot_idx * 1e-3) / 1e12, 1),
                "indexer_topk_frac_bf16": round(idx_flop / (tot_idx * 1e-3) / 1e12 / pk["bf16"], 3),
                "mla_tflops": round(mla_flop / (tot_mla * 1e-3) / 1e12, 1),
                "mla_frac_bf16": round(mla_flop / (tot_mla * 1e-3) / 1e12 / pk["bf16"], 3),
                "runs": "median of 20 per shard, L2 flushed before each"}
        if args.with_oracle:
            line["oracle"] = {"tokens_per_s": round(or_q / or_s, 3), "kind": "oracle",
                              "cores": _blas_threads(),
                              "sample": f"{or_q} evenly spaced queries of one shard (the longest "
                                        f"included), {or_s:.2f} s, extrapolated per query"}
        if wl.decode_queries:
            line["indexer_topk_gbs"] = round(idx_bytes / (tot_idx * 1e-3) / 1e9, 1)
            line["indexer_topk_frac_hbm"] = round(idx_bytes / (tot_idx * 1e-3) / 1e9 / pk["hbm"], 3)
            line["mla_gbs"] = round(mla_bytes / (tot_mla * 1e-3) / 1e9, 1)
            line["mla_frac_hbm"] = round(mla_bytes / (tot_mla * 1e-3) / 1e9 / pk["hbm"], 3)
        print(json.dumps(line), flush=True)
    print(json.dumps({"device_errors": dsa.dsa_read_device_errors()}), flush=True)


def _oracle_sample_time(W, wl, si, idx, mi, n_sample):
    """fp64 oracle (indexer, full-sort top-k, sparse MLA) on `n_sample` queries of a shard whose
    inputs live on the device; returns (queries, seconds). Only the sampled queries' requests are
    copied to the host, as one compact contiguous KV (a paged cache is read through its table)."""
    from oracle.kv import ContiguousKV
    pos = si["pos"].cpu().numpy().astype(np.int64)
    bid = si["bid"].cpu().numpy().astype(np.int64)
    sel = np.unique(np.concatenate([np.linspace(0, len(pos) - 1, n_sample).round(),
                                    [int(np.argmax(pos))]]).astype(np.int64))
    reqs = sorted(set(int(b) for b in bid[sel]))
    need = {b: int(pos[sel][bid[sel] == b].max()) + 1 for b in reqs}
    if si["bt"] is not None:
        table = si["bt"].cpu().numpy().astype(np.int64)
        rows = np.concatenate([table[b, np.arange(need[b]) // wl.page_size] * wl.page_size
                               + np.arange(need[b]) % wl.page_size for b in reqs])
    else:
        cu = si["cu"].cpu().numpy().astype(np.int64)
        rows = np.concatenate([cu[b] + np.arange(need[b]) for b in reqs])
    import torch
    r_dev = torch.as_tensor(rows, device=idx.k_idx.device)
    k64 = idx.k_idx[r_dev].float().cpu().numpy().astype(np.float64)
    c64 = mi.c[r_dev].float().cpu().numpy().astype(np.float64)
    cu2 = np.concatenate([[0], np.cumsum([need[b] for b in reqs])]).astype(np.int64)
    remap = {b: i for i, b in enumerate(reqs)}
    s_dev = torch.as_tensor(sel, device=idx.k_idx.device)
    sh = {"cu": cu2, "q_idx": idx.q_idx[s_dev].float().cpu().numpy().astype(np.float64),
          "w": idx.w[s_dev].cpu().numpy().astype(np.float64), "k_idx": k64,
          "q": mi.q[s_dev].float().cpu().numpy().astype(np.float64), "c": c64,
          "pos": pos[sel], "bid": np.asarray([remap[int(b)] for b in bid[sel]], dtype=np.int64)}
    loc = np.arange(len(sel))
    t0 = time.perf_counter()
    _oracle_step(W, wl, sh, loc)
    return len(sel), time.perf_counter() - t0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=96, help="queries per reference-arm step")
    ap.add_argument("--cpu-baseline-queries", type=int, default=1476)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--next-rows", nargs="?", const="all", default=None,
                    help="measure the widened rows (paged rerange, decode split) and exit")
    ap.add_argument("--configs", action="store_true",
                    help="indexer + top-k + sparse MLA on every workload config, then exit")
    ap.add_argument("--with-oracle", action="store_true",
                    help="with --configs: also time the fp64 oracle on a sample of each config")
    args = ap.parse_args()
    if args.configs:
        config_rows(args)
        return
    if args.next_rows:
        next_rows(args)
        return
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
