"""Benchmark: round-robin sequence-sharded DSA prefill attention on one GB300.

Workload (default): the many-request batch -- 32 requests with lengths U[128, 4096] (seed 0,
N = 71,014 tokens), sp = 4, all four shards processed back to back on one GPU (17,753-17,754
queries each, 71,014 in total); indexer 64 heads x 128, top-k 2048; MLA 128 heads, qk 576 /
v 512, bf16. A step is the whole shard path of every shard through the C ABI:
  split metadata + the shard's row gather -> rerange of the all-gathered k_idx and latent rows
  -> indexer scores (for the groups of queries whose history exceeds k; the others take every
  key) + top-k -> sparse MLA.
The other shards' rows are inputs (one GPU, no collective). The long single prompt (32,768
tokens, sp = 8, all eight shards) is timed the same way and reported under "config_long".
With --gpus N (torchrun) every GPU runs an independent replica of the same batch: weak scaling,
no collective on the data path.

value = query tokens processed / device time of the timed steps (CUDA events on the launch
stream, L2 flushed between steps); e2e = the same through host buffers: every step copies its
inputs from pinned host memory and reads o back inside the timed region, pipelined shard by
shard over two buffer sets and three streams (the upload of the next shard and the download of
the previous one overlap the current shard's kernels).
--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
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
WORKLOAD_ID = 3          # many-request batch, all shards (the largest single-GPU prefill config)
LONG_ID = 2              # long single prompt, all shards (reported beside it)
NOMINAL = {"bf16": 2250.0, "hbm": 7900.0}   # GB300 dense bf16 TFLOP/s and HBM3e GB/s, nominal


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16": float(d["bf16_tflops"]), "bf16_sustained": float(d["bf16_tflops_sustained"]),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def profiled_traffic(kernel):
    """DRAM bytes per unit of work from profiles/traffic.json (written from an ncu capture),
    only while the kernel's source file still has the hash recorded there; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json"), encoding="utf-8") as f:
            rec = json.load(f)[kernel]
        with open(os.path.join(ROOT, "deepseek_v3_sparse_round_gb300", "csrc", rec["source"]), "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()[:12]
        if rec.get("source_sha1") == sha:
            return rec
    except (OSError, KeyError, ValueError):
        pass
    return None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, dist, device) -> float:
    """The job's time is the slowest rank's: all-reduce MAX (no-op without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shards_for_rank(rank: int, world: int, sp: int) -> list:
    """Every GPU runs an independent replica of the whole batch: all sp shards of it. The job
    processes world x (all queries of the batch); no shard is shared between GPUs."""
    del rank, world
    return list(range(sp))


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
class ConfigStep:
    """Device buffers and the launches of one step of a prefill workload: every shard of the
    batch, back to back. Inputs are drawn on the device (seeded); `host()` makes pinned host
    copies for the end-to-end run."""

    LAUNCHES_PER_SHARD = 7   # split (+gather), rerange (k_idx and latent rows together),
    #                          indexer plan, indexer, top-k, MLA schedule, MLA -- as the ncu
    #                          launch list of a step shows

    def __init__(self, torch, dsa, W, wid, device):
        self.torch, self.dsa, self.W = torch, dsa, W
        wl = W.WORKLOADS[wid]
        self.wl, self.wid, self.dev = wl, wid, device
        cu_np = W.cu_seqlens(wl.lengths)
        self.cu_np = cu_np
        self.N = int(cu_np[-1])
        self.n_req = len(wl.lengths)
        self.max_ctx = int(max(wl.lengths))
        self.ranks = list(wl.ranks)
        e = lambda *sh, dt=torch.int32: torch.empty(*sh, dtype=dt, device=device)
        self.n_r = {r: dsa.dsa_rr_shard_len(self.N, wl.sp, r) for r in self.ranks}
        # shared inputs: request offsets, the logical latent rows (each shard gathers its own
        # rows from them), and the all-gathered (rank-major, packed) k_idx and latent rows that
        # every shard reranges
        idx0 = W.indexer_inputs(wl, 1, self.N, 0, device=device)
        mi0 = W.mla_inputs(wl, 1, self.N, 0, device=device)
        perm = torch.as_tensor(np.concatenate([np.arange(q, self.N, wl.sp) for q in range(wl.sp)]),
                               device=device)
        self.shared = {"cu": torch.as_tensor(cu_np, device=device), "c_log": mi0.c,
                       "k_gath": idx0.k_idx[perm].contiguous(), "c_gath": mi0.c[perm].contiguous()}
        del idx0, mi0
        # per-shard inputs and outputs
        self.inp, self.out = {}, {}
        for r in self.ranks:
            n = self.n_r[r]
            idx = W.indexer_inputs(wl, n, 1, r, device=device)
            mi = W.mla_inputs(wl, n, 1, r, device=device)
            self.inp[r] = {"q_idx": idx.q_idx, "w": idx.w, "q": mi.q}
            self.out[r] = {"cu_shard": e(self.n_req + 1), "pos": e(n), "bid": e(n), "gidx": e(n),
                           "c_local": e(n, wl.dqk, dt=torch.bfloat16),
                           "o": e(n, wl.H, wl.dv, dt=torch.bfloat16),
                           "lse": e(n, wl.H, dt=torch.float32)}
        n_max = max(self.n_r.values())
        # one rank's working buffers, reused shard after shard (the shards run in order)
        self.k_idx = e(self.N, wl.Di, dt=torch.bfloat16)
        self.c = e(self.N, wl.dqk, dt=torch.bfloat16)
        self.ws = e(dsa.dsa_indexer_topk_workspace_size(n_max, self.max_ctx, wl.topk), dt=torch.uint8)
        self.topk = e(n_max, wl.topk)
        self.mla_ws = e(dsa.dsa_sparse_mla_workspace_size(n_max), dt=torch.uint8)
        self.launches_per_step = self.LAUNCHES_PER_SHARD * len(self.ranks)

    def run_shard(self, r, inp=None, shared=None, o=None, ev=None):
        """One shard's path. ev: optional 5 events recorded before the split, after it, after
        the rerange, after indexer+top-k and after the MLA."""
        dsa, wl = self.dsa, self.wl
        inp = self.inp[r] if inp is None else inp
        sh = self.shared if shared is None else shared
        out = self.out[r]
        n = self.n_r[r]
        if ev is not None:
            ev[0].record()
        dsa.dsa_rr_split_metadata(sh["cu"], self.N, wl.sp, r, out["cu_shard"], out["pos"],
                                  out["bid"], out["gidx"], src_rows=sh["c_log"],
                                  dst_rows=out["c_local"])
        if ev is not None:
            ev[1].record()
        dsa.dsa_rr_rerange_multi([sh["k_gath"], sh["c_gath"]], [self.k_idx, self.c], self.N,
                                 wl.sp, 0)
        if ev is not None:
            ev[2].record()
        topk = self.topk[:n]
        dsa.dsa_indexer_topk(inp["q_idx"], inp["w"], self.k_idx, sh["cu"], self.n_req, out["pos"],
                             out["bid"], wl.topk, self.max_ctx, topk, self.ws)
        if ev is not None:
            ev[3].record()
        dsa.dsa_sparse_mla_balanced(inp["q"], self.c, sh["cu"], self.n_req, out["bid"],
                                    out["pos"], topk, wl.scale, out["o"] if o is None else o,
                                    self.mla_ws, lse=out["lse"])
        if ev is not None:
            ev[4].record()

    def run(self):
        for r in self.ranks:
            self.run_shard(r)

    def work(self):
        """Algorithmic work of one step: indexer flop (the causal pairs of the queries whose
        history exceeds k: the others select every key and need no score), MLA flop (selected
        pairs), bytes moved by the split gather and the two reranges."""
        wl = self.wl
        idx = mla = 0.0
        pairs_c = pairs_i = pairs_s = 0
        for r in self.ranks:
            pos = self.out[r]["pos"].cpu().numpy().astype(np.int64)
            pairs_c += int(np.sum(pos + 1))
            pairs_i += int(np.sum((pos + 1)[pos + 1 > wl.topk]))
            pairs_s += int(np.sum(np.minimum(pos + 1, wl.topk)))
        idx = 2.0 * wl.Hi * wl.Di * pairs_i
        mla = 2.0 * wl.H * (wl.dqk + wl.dv) * pairs_s
        rerange_bytes = 2 * self.N * (wl.Di + wl.dqk) * 2 * len(self.ranks)
        nbytes = sum(2 * self.n_r[r] * wl.dqk * 2 for r in self.ranks) + rerange_bytes
        return {"indexer_flop": idx, "mla_flop": mla, "causal_pairs": pairs_c,
                "indexer_pairs": pairs_i,
                "selected_pairs": pairs_s, "copy_bytes": nbytes, "rerange_bytes": rerange_bytes,
                "shard_queries": [self.n_r[r] for r in self.ranks]}

    def queries(self):
        return sum(self.n_r.values())

    def host(self):
        """Pinned host copies of every input, and pinned host outputs (o per shard)."""
        torch = self.torch
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        self.h_shared = {k: pin(v) for k, v in self.shared.items()}
        self.h_inp = {r: {k: pin(v) for k, v in d.items()} for r, d in self.inp.items()}
        self.h_o = {r: torch.empty(self.out[r]["o"].shape, dtype=torch.bfloat16, pin_memory=True)
                    for r in self.ranks}
        n_max = max(self.n_r.values())
        wl = self.wl
        mk = lambda *sh, dt: torch.empty(*sh, dtype=dt, device=self.dev)
        # two device sets for the pipeline: shared inputs, one shard's inputs and its o
        self.d_shared = [{k: torch.empty_like(v) for k, v in self.shared.items()} for _ in range(2)]
        self.d_inp = [{"q_idx": mk(n_max, wl.Hi, wl.Di, dt=torch.bfloat16),
                       "w": mk(n_max, wl.Hi, dt=torch.float32),
                       "q": mk(n_max, wl.H, wl.dqk, dt=torch.bfloat16)} for _ in range(2)]
        self.d_o = [mk(n_max, wl.H, wl.dv, dt=torch.bfloat16) for _ in range(2)]

    def h2d_bytes(self):
        b = sum(v.numel() * v.element_size() for v in self.h_shared.values())
        for d in self.h_inp.values():
            b += sum(v.numel() * v.element_size() for v in d.values())
        return b

    def d2h_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.h_o.values())


def time_steps(torch, st, steps, flush, stream):
    """Device time of `steps` steps, L2 flushed before each; per-shard events split each step
    into split+reranges, indexer+top-k and MLA. Returns (total seconds, per-part seconds)."""
    mk = lambda: torch.cuda.Event(enable_timing=True)
    evs = []
    for i in range(steps):
        flush.fill_(float(i))
        e0 = mk()
        e0.record(stream)
        per = []
        for r in st.ranks:
            ev = (mk(), mk(), mk(), mk(), mk())
            st.run_shard(r, ev=ev)
            per.append(ev)
        e1 = mk()
        e1.record(stream)
        evs.append((e0, e1, per))
    torch.cuda.synchronize()
    total = sum(a.elapsed_time(b) for a, b, _ in evs) / 1e3
    parts = {"split_rerange": 0.0, "rerange": 0.0, "indexer_topk": 0.0, "mla": 0.0}
    for _, _, per in evs:
        for ev in per:
            parts["split_rerange"] += ev[0].elapsed_time(ev[2]) / 1e3
            parts["rerange"] += ev[1].elapsed_time(ev[2]) / 1e3
            parts["indexer_topk"] += ev[2].elapsed_time(ev[3]) / 1e3
            parts["mla"] += ev[3].elapsed_time(ev[4]) / 1e3
    return total, parts


def roofline_obj(kernel, bound, achieved, peak, unit, nominal, traffic, extra):
    d = {"bound": bound, "kernel": kernel, "achieved": round(achieved, 1), "peak": peak,
         "unit": unit, "frac": round(achieved / peak, 4),
         "nominal_peak": nominal, "frac_of_nominal": round(achieved / nominal, 4),
         "traffic": traffic}
    d.update(extra)
    return d


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


def host_link(torch, device, h2d_bytes, d2h_bytes):
    """The host link the e2e line runs over: 1 GiB pinned copies, each direction alone and both
    at once on two streams (CUDA events, best of 3), and the per-step time those rates allow
    for the step's bytes with both directions busy."""
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h2 = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(n, dtype=torch.uint8, device=device)
    d2 = torch.empty(n, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def best(fn):
        ts = []
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
        return min(ts)

    def both():
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)

    h2d = n / best(lambda: d.copy_(h, non_blocking=True)) / 1e9
    d2h = n / best(lambda: h2.copy_(d2, non_blocking=True)) / 1e9
    each = n / best(both) / 1e9
    del h, h2, d, d2
    return {"h2d_gbps": round(h2d, 1), "d2h_gbps": round(d2h, 1),
            "both_directions_gbps_each": round(each, 1),
            "ms_per_step_at_link_rate": round(max(h2d_bytes, d2h_bytes) / each / 1e6, 2),
            "how": "1 GiB pinned copies, best of 3"}


def mla_gather_roofline(torch, dsa, W, device, work, mla_s, clocks):
    """The sparse MLA against the resource that binds it: the rate at which an SM brings
    selected latent rows into shared memory. CTA 0 of each pair gathers 1,152 B per selected
    pair; the ceiling is measured in this run by the library's row-gather probe (16-byte
    cp.async, every SM, a 3-slot ring of 48-row tiles, nothing consuming them), as bytes per SM
    clock. Achieved = CTA 0's bytes per launch / (MLA time x the SM clock sampled during the
    timed steps)."""
    n_ctas = torch.cuda.get_device_properties(device).multi_processor_count
    n_tiles = 400
    n_rows = int(sum(W.WORKLOADS[WORKLOAD_ID].lengths))
    g = torch.Generator(device="cpu").manual_seed(7)
    c = torch.randn(n_rows, 576, generator=g).to(torch.bfloat16).to(device)
    rows = torch.randint(0, n_rows, (n_ctas * n_tiles * 48,), generator=g,
                         dtype=torch.int32).to(device)
    cycles = torch.zeros(n_ctas, dtype=torch.int64, device=device)
    per_tile = []
    for _ in range(3):
        dsa.dsa_probe_row_gather(c, rows, n_ctas, n_tiles, 0, 1, cycles)
        torch.cuda.synchronize()
        per_tile.append(float(cycles.double().mean()) / n_tiles)
    ceiling = 48 * 1152 / sorted(per_tile)[1]        # B per SM clock (median of 3)
    sm_mhz = clocks.get("sm_mhz") if isinstance(clocks, dict) else None
    pairs_per_launch = min(n_ctas // 2, min(work["shard_queries"]))
    launches = len(work["shard_queries"])
    if not sm_mhz:
        return {"bound": "l2_row_gather", "peak": round(ceiling, 2), "achieved": None,
                "note": "no SM clock sample"}
    b_sm = work["selected_pairs"] * 1152 / launches / pairs_per_launch   # CTA 0, one launch
    achieved = b_sm / ((mla_s / launches) * sm_mhz * 1e6)
    return {"bound": "l2_row_gather", "achieved": round(achieved, 2), "peak": round(ceiling, 2),
            "unit": "B per SM clock (CTA 0 of each pair)", "frac": round(achieved / ceiling, 4),
            "peak_source": "dsa_probe_row_gather mode 0 in this run (median of 3)",
            "clock_mhz": sm_mhz,
            "unit_of_work": "selected (query, key) pair: CTA 0 gathers its 576-column row "
                            "(1,152 B); CTA 1 gathers 1,024 B of the same row"}


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

    pk = peaks()
    st = ConfigStep(torch, dsa, W, WORKLOAD_ID, device)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)   # > L2
    stream = torch.cuda.current_stream()

    clk = ClockSampler(local).__enter__()            # running before the timed window opens
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    work = st.work()

    # ---- device-timed steps (inputs resident in HBM), L2 flushed between steps ----
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    dev_s, parts = time_steps(torch, st, args.steps, flush, stream)
    t_end = time.perf_counter()
    clk.mark(t_wall, t_end)
    clk.__exit__(None, None, None)
    dev_s = max_over_ranks(dev_s, dist, device)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()

    # ---- the long single prompt (8 shards of 4,096 queries), timed the same way ----
    long_line = None
    if not args.no_long:
        st2 = ConfigStep(torch, dsa, W, LONG_ID, device)
        for _ in range(args.warmup):
            st2.run()
        torch.cuda.synchronize()
        work2 = st2.work()
        steps2 = max(3, args.steps // 2)
        if dist:
            dist.barrier()
        l_s, l_parts = time_steps(torch, st2, steps2, flush, stream)
        l_s = max_over_ranks(l_s, dist, device)
        q2 = st2.queries() * ws
        mla2 = work2["mla_flop"] / (l_parts["mla"] / steps2) / 1e12
        idx2 = work2["indexer_flop"] / (l_parts["indexer_topk"] / steps2) / 1e12
        long_line = {
            "workload": "long: 1 request of 32,768 tokens, sp=8, all 8 shards back to back "
                        "(4,096 queries each)",
            "value": round(q2 * steps2 / l_s, 2), "unit": "tokens/s", "steps": steps2,
            "ms_per_step": round(l_s * 1e3 / steps2, 4),
            "ms_split_rerange": round(l_parts["split_rerange"] * 1e3 / steps2, 4),
            "ms_indexer_topk": round(l_parts["indexer_topk"] * 1e3 / steps2, 4),
            "ms_mla": round(l_parts["mla"] * 1e3 / steps2, 4),
            "mla_tflops": round(mla2, 1), "mla_frac": round(mla2 / pk["bf16"], 4),
            "mla_frac_of_nominal": round(mla2 / NOMINAL["bf16"], 4),
            "indexer_topk_tflops": round(idx2, 1), "indexer_topk_frac": round(idx2 / pk["bf16"], 4),
            "indexer_topk_frac_of_nominal": round(idx2 / NOMINAL["bf16"], 4)}
        del st2
        torch.cuda.empty_cache()

    # ---- end to end through host buffers, pipelined shard by shard ----
    st.host()
    n_units = len(st.ranks)
    e2e_steps = max(2, min(args.e2e_steps, args.steps))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    s_in, s_run, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    total_units = e2e_steps * n_units
    ev_in, ev_run, ev_out = ([torch.cuda.Event() for _ in range(total_units)] for _ in range(3))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_run.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(total_units):
        step, r = divmod(i, n_units)
        r = st.ranks[r]
        b, sb = i % 2, step % 2
        n = st.n_r[r]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_run[i - 2])       # unit i - 2 is done reading set b
            if r == st.ranks[0]:                     # the step's shared inputs (set sb)
                for k, v in st.h_shared.items():
                    st.d_shared[sb][k].copy_(v, non_blocking=True)
            for k, v in st.h_inp[r].items():
                st.d_inp[b][k][:n].copy_(v, non_blocking=True)
            ev_in[i].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[i])
            if i >= 2:
                s_run.wait_event(ev_out[i - 2])      # o of unit i - 2 has been read back
            d = st.d_inp[b]
            st.run_shard(r, inp={k: v[:n] for k, v in d.items()}, shared=st.d_shared[sb],
                         o=st.d_o[b][:n])
            ev_run[i].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[i])
            st.h_o[r].copy_(st.d_o[b][:n], non_blocking=True)
            ev_out[i].record(s_out)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, dist, device)

    link = host_link(torch, device, st.h2d_bytes(), st.d2h_bytes())
    errors = dsa.dsa_read_device_errors()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    queries = st.queries() * ws
    value = queries * args.steps / dev_s
    mla_s = parts["mla"] / args.steps
    idx_s = parts["indexer_topk"] / args.steps
    cp_s = parts["split_rerange"] / args.steps
    mla_ach = work["mla_flop"] / mla_s / 1e12
    idx_ach = work["indexer_flop"] / idx_s / 1e12
    cp_ach = work["copy_bytes"] / cp_s / 1e9
    rr_s = parts["rerange"] / args.steps
    rr_ach = work["rerange_bytes"] / rr_s / 1e9
    mla_tr = profiled_traffic("sparse_mla_pair_kernel")
    traffic = None
    if mla_tr is not None:    # DRAM bytes per selected pair from a capture, scaled to a launch
        traffic = int(mla_tr["dram_bytes_per_unit"] * work["selected_pairs"] / len(st.ranks))
    gather = mla_gather_roofline(torch, dsa, W, device, work, mla_s, clk.summary())
    cpu = None
    if not args.no_cpu_baseline and ws == 1:       # the oracle baseline is a one-GPU figure
        cpu = cpu_baseline(args.cpu_baseline_queries)
    wl = st.wl
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dev_s * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded bf16 N(0,1) queries/keys/latents; no weights needed)",
        "config": {"workload": "many_req: 32 requests, lengths U[128,4096] (seed 0, N=71,014), "
                               "sp=4, all 4 shards back to back (71,014 queries); indexer 64x128 "
                               "top-2048; MLA 128 heads 576/512",
                   "queries_per_gpu": st.queries(), "kv_tokens": st.N, "topk": wl.topk,
                   "shard_queries": [st.n_r[r] for r in st.ranks],
                   "l2": "flushed between timed steps (256 MB write)",
                   "step": "per shard: split+gather, rerange (k_idx + latent rows, one launch), "
                           "indexer scores, top-k, sparse MLA",
                   "multi_gpu": "independent replicas of the whole batch (no collective)"},
        "roofline": roofline_obj(
            "sparse_mla_pair_kernel", "tensor", mla_ach, pk["bf16"], "TFLOP/s", NOMINAL["bf16"],
            traffic,
            {"peak_source": f"{pk['source']} bf16 burst (MEASURED_PEAKS.json)",
             "algorithmic_flop_per_launch": work["mla_flop"] / len(st.ranks),
             "unit_of_work": "selected (query, key) pair: 2*128*(576+512) = 278,528 flop",
             "launches_per_step": len(st.ranks),
             "timing": "CUDA events around each MLA call (schedule kernel + MLA) on the launch "
                       "stream, mean over the timed steps",
             "traffic_note": None if traffic is None else
             f"ncu DRAM bytes per selected pair x pairs per launch ({mla_tr['workload']})"}),
        "roofline_indexer": roofline_obj(
            "indexer_plan_kernel + indexer_kernel<64,128> + topk_short_kernel (one call)",
            "tensor", idx_ach, pk["bf16"], "TFLOP/s",
            NOMINAL["bf16"], None,
            {"algorithmic_flop_per_step": work["indexer_flop"],
             "unit_of_work": "causal (query, key) pair of a query whose history exceeds k "
                             "(the others take every key and need no score): 2*64*128 = "
                             "16,384 flop",
             "causal_pairs_all_queries": work["causal_pairs"],
             "timing": "CUDA events around each indexer+top-k call (plan, indexer, top-k)",
             # k int32 indices for every query, those whose history fits in k included
             "topk_output_bytes_per_step": int(st.queries() * st.wl.topk * 4)}),
        "roofline_split_rerange": roofline_obj(
            "split_kernel + rerange_multi_kernel", "hbm", cp_ach, pk["hbm"], "GB/s",
            NOMINAL["hbm"], None,
            {"algorithmic_bytes_per_step": work["copy_bytes"],
             "unit_of_work": "row moved: 2 x row bytes (read + write)",
             "timing": "CUDA events before the split and after the rerange (two launches)"}),
        "roofline_rerange": roofline_obj(
            "rerange_multi_kernel", "hbm", rr_ach, pk["hbm"], "GB/s", NOMINAL["hbm"], None,
            {"algorithmic_bytes_per_launch": work["rerange_bytes"] / len(st.ranks),
             "unit_of_work": "token: 2 x (256 + 1152) B (k_idx and latent rows, read + write)",
             "timing": "CUDA events around each rerange launch, mean over the timed steps"}),
        "roofline_mla_gather": gather,
        "ms_split_rerange": round(cp_s * 1e3, 4), "ms_indexer_topk": round(idx_s * 1e3, 4),
        "ms_mla": round(mla_s * 1e3, 4),
        "e2e": {"value": round(queries * e2e_steps / e2e_s, 2), "unit": "tokens/s",
                "steps": e2e_steps, "h2d_bytes_per_step": st.h2d_bytes(),
                "d2h_bytes_per_step": st.d2h_bytes(),
                "ms_per_step": round(e2e_s * 1e3 / e2e_steps, 2),
                "how": "pinned host inputs uploaded and o read back every step, pipelined per "
                       "shard over 2 buffer sets and 3 streams",
                "host_link": link},
        "gpu_launches": st.launches_per_step * args.steps,
        "clocks": clk.summary(),
        "device_errors": errors,
        "wall_s_timed_region": round(t_end - t_wall, 4),
        "config_long": long_line,
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
    """fp64 inputs of a bounded sample of the many-request batch: n_sample queries spread
    evenly over every shard (all requests, short and long histories), with the whole logical KV.
    Values come from the same seeded generators as the GPU arm (on the GPU when there is one, so
    the sampled rows are the very values the GPU path consumes)."""
    import torch
    import workloads as W
    from oracle import split as osplit
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = W.WORKLOADS[WORKLOAD_ID]
    cu = W.cu_seqlens(wl.lengths)
    n = int(cu[-1])
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    k_all = W.indexer_inputs(wl, 1, n, 0, device=dev).k_idx
    c_all = W.mla_inputs(wl, 1, n, 0, device=dev).c
    parts = {"q_idx": [], "w": [], "q": [], "pos": [], "bid": []}
    per = max(1, n_sample // len(wl.ranks))
    n_total = 0
    for r in wl.ranks:
        meta = osplit.round_robin_split(cu, wl.sp, r)
        n_r = len(meta["pos"])
        n_total += n_r
        sel = np.unique(np.linspace(0, n_r - 1, per).round().astype(np.int64))
        idx = W.indexer_inputs(wl, n_r, 1, r, device=dev)
        mi = W.mla_inputs(wl, n_r, 1, r, device=dev)
        st = torch.as_tensor(sel, device=dev)
        parts["q_idx"].append(f64(idx.q_idx[st]))
        parts["w"].append(f64(idx.w[st]))
        parts["q"].append(f64(mi.q[st]))
        parts["pos"].append(meta["pos"][sel])
        parts["bid"].append(meta["bid"][sel])
        del idx, mi
    sh = {k: np.concatenate(v) for k, v in parts.items()}
    sh["cu"] = cu
    sh["k_idx"] = f64(k_all)
    sh["c"] = f64(c_all)
    return W, wl, sh, n_total


def cpu_baseline(sample_queries=1024, min_seconds=10.0, max_passes=6):
    """Passes of the oracle over the sample until at least `min_seconds` of CPU work (bounded
    by `max_passes`), so the figure rests on 10-30 s of work without stretching the bench."""
    W, wl, sh, n_total = _oracle_inputs(sample_queries)
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
            "sample": f"{len(sel)} of the {n_total} queries of the many-request batch (evenly "
                      f"spaced over all 4 shards), fp64 NumPy indexer + full-sort top-k + sparse "
                      f"MLA, {steps} pass(es), {dt:.1f} s"}


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
    W, wl, sh, n_total = _oracle_inputs(args.cpu_sample)
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
        "config": {"workload": "many_req: 32 requests, lengths U[128,4096] (seed 0, N=71,014), "
                               "sp=4, all 4 shards: a bounded sample of "
                               f"{len(sel)} of its {n_total} queries per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{len(sel)} queries per step, evenly spaced over the 4 shards"},
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
        # the step's rerange (k_idx + latent rows through one row map, one launch) over a range
        # of sizes around the many-request batch, L2 flushed: time = ramp + bytes / rate
        wl3 = W.WORKLOADS[3]
        sizes, times = [], []
        for scale in (0.125, 0.25, 0.5, 1, 2, 4, 8):
            n = int(sum(wl3.lengths) * scale)
            kg = torch.randn(n, wl3.Di, device="cuda").to(torch.bfloat16)
            cg = torch.randn(n, wl3.dqk, device="cuda").to(torch.bfloat16)
            ko, co = torch.empty_like(kg), torch.empty_like(cg)
            nbytes = 2 * n * (wl3.Di + wl3.dqk) * 2
            ms = timeit(lambda: dsa.dsa_rr_rerange_multi([kg, cg], [ko, co], n, wl3.sp, 0), 20, True)
            sizes.append(nbytes)
            times.append(ms * 1e3)
            print(json.dumps({"kernel": "rerange_multi (k_idx 256 B + latent 1,152 B rows)",
                              "tokens": n, "bytes": nbytes, "us": round(ms * 1e3, 1),
                              "GB/s": round(nbytes / ms / 1e6),
                              "frac_of_measured_hbm": round(nbytes / ms / 1e6 / hbm, 3),
                              "l2": "flushed between launches"}), flush=True)
            del kg, cg, ko, co
            torch.cuda.empty_cache()
        slope, ramp = np.polyfit(np.asarray(sizes, dtype=np.float64), np.asarray(times), 1)
        print(json.dumps({"kernel": "rerange_multi", "fit": "us = ramp + bytes / rate",
                          "ramp_us": round(float(ramp), 2),
                          "rate_GB/s": round(1e-3 / float(slope)),
                          "rate_frac_of_measured_hbm": round(1e-3 / float(slope) / hbm, 3)}),
              flush=True)
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
        tot_q = tot_idx = tot_mla = tot_idx8 = 0.0
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
            # the FP8 (E4M3) indexer rows: quantised once, outside the timed region
            q8 = torch.empty(idx.q_idx.shape, dtype=torch.uint8, device="cuda")
            qs = torch.empty(idx.q_idx.shape[:2], dtype=torch.float32, device="cuda")
            k8 = torch.empty(idx.k_idx.shape, dtype=torch.uint8, device="cuda")
            ks = torch.empty(idx.k_idx.shape[0], dtype=torch.float32, device="cuda")
            dsa.dsa_quantize_fp8_rows(idx.q_idx, q8, qs)
            dsa.dsa_quantize_fp8_rows(idx.k_idx, k8, ks)
            topk8 = torch.empty_like(topk)
            f_idx8 = lambda: dsa.dsa_indexer_topk_fp8(q8, qs, idx.w, k8, ks, si["cu"], n_req,
                                                      si["pos"], si["bid"], wl.topk,
                                                      si["max_ctx"], topk8, ws,
                                                      block_table=si["bt"])
            (t_idx8,) = timed([f_idx8])
            tot_idx8 += t_idx8
            del q8, qs, k8, ks, topk8
            p = si["pos"].cpu().numpy().astype(np.int64)
            tot_q += n_q
            tot_idx += t_idx
            tot_mla += t_mla
            idx_flop += 2.0 * wl.Hi * wl.Di * float(np.sum((p + 1)[p + 1 > wl.topk]))
            sel = float(np.sum(np.minimum(p + 1, wl.topk)))
            mla_flop += 2.0 * wl.H * (wl.dqk + wl.dv) * sel
            if wl.decode_queries:
                idx_bytes = float(sum(wl.lengths)) * wl.Di * 2
                mla_bytes += sel * wl.dqk * 2
            si_rows = si["n_rows"]
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
                "indexer_topk_fp8_ms": round(tot_idx8, 4),
                "indexer_topk_fp8_tflops": round(idx_flop / (tot_idx8 * 1e-3) / 1e12, 1),
                "indexer_topk_fp8_frac_fp8": round(idx_flop / (tot_idx8 * 1e-3) / 1e12 /
                                                   (2.0 * pk["bf16"]), 3),
                "mla_tflops": round(mla_flop / (tot_mla * 1e-3) / 1e12, 1),
                "mla_frac_bf16": round(mla_flop / (tot_mla * 1e-3) / 1e12 / pk["bf16"], 3),
                "runs": "median of 20 per shard, L2 flushed before each",
                "fp8_peak": "2 x the measured bf16 burst (the nominal fp8 / bf16 dense ratio)"}
        if args.with_oracle:
            line["oracle"] = {"tokens_per_s": round(or_q / or_s, 3), "kind": "oracle",
                              "cores": _blas_threads(),
                              "sample": f"{or_q} evenly spaced queries of one shard (the longest "
                                        f"included), {or_s:.2f} s, extrapolated per query"}
        # the FP8 latent cache: packing the batch's latent rows (or the decode pool) and
        # expanding them back to the bf16 rows the MLA reads; 1,152 + 656 bytes per row each way
        n_lat = int(sum(wl.lengths)) if not wl.decode_queries else int(si_rows)
        c_lat = torch.randn(n_lat, 576, device="cuda").to(torch.bfloat16)
        p_lat = torch.empty((n_lat, 656), dtype=torch.uint8, device="cuda")
        t_q, t_d = timed([lambda: dsa.dsa_quantize_fp8_latent(c_lat, p_lat),
                          lambda: dsa.dsa_dequantize_fp8_latent(p_lat, c_lat)])
        lat_bytes = n_lat * (1152 + 656)
        line["fp8_latent"] = {"rows": n_lat, "quantize_ms": round(t_q, 4),
                              "dequantize_ms": round(t_d, 4),
                              "dequantize_gbs": round(lat_bytes / (t_d * 1e-3) / 1e9, 1),
                              "dequantize_frac_hbm": round(lat_bytes / (t_d * 1e-3) / 1e9 / pk["hbm"], 3),
                              "bytes_per_row": {"bf16": 1152, "fp8": 656}}
        del c_lat, p_lat
        torch.cuda.empty_cache()
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


def profile_run(args):
    """Small, fixed launch sequences for ncu (no timing, no flush, nothing else on the GPU):
    --profile-steps K: the default workload's whole step, 1 untimed step then K more (32
      launches per step: the launch list);
    --profile-decode: the paged decode batch, indexer + top-k and MLA twice;
    --profile-case: one shard of the many-request batch (rank 1) cut to an evenly spaced
      subset of 2,048 of its queries (every request, short and long histories; about 0.7 GB on
      the device): indexer + top-k, balanced sparse MLA, the FP8 row quantisation and the FP8
      indexer + top-k, each twice (kernel captures)."""
    import torch
    import __graft_entry__ as ge
    ge.build()
    import deepseek_v3_sparse_round_gb300 as dsa
    import workloads as W
    dev = torch.device("cuda", 0)
    if args.profile_decode:
        # the paged decode batch (64 requests x 2 queries over 2.65 M cached tokens, about
        # 4 GB on the device): indexer + top-k and balanced sparse MLA, each twice
        wl = W.WORKLOADS[4]
        table, n_pages = W.random_block_table(wl.lengths, wl.page_size,
                                              W.seed_of(wl, "block_table"))
        bid_np, pos_np = W.decode_queries(wl.lengths, wl.decode_queries)
        n_rows = n_pages * wl.page_size
        cu = torch.zeros(len(wl.lengths) + 1, dtype=torch.int32, device=dev)
        bt = torch.as_tensor(table, device=dev)
        bid = torch.as_tensor(np.asarray(bid_np, np.int32), device=dev)
        pos = torch.as_tensor(np.asarray(pos_np, np.int32), device=dev)
        n_q, max_ctx, n_req = pos.numel(), int(max(wl.lengths)), len(wl.lengths)
        idx = W.indexer_inputs(wl, n_q, n_rows, 0, device=dev)
        mi = W.mla_inputs(wl, n_q, n_rows, 0, device=dev)
        ws = torch.empty(dsa.dsa_indexer_topk_workspace_size(n_q, max_ctx, wl.topk),
                         dtype=torch.uint8, device=dev)
        mws = torch.empty(dsa.dsa_sparse_mla_workspace_size(n_q), dtype=torch.uint8, device=dev)
        topk = torch.empty((n_q, wl.topk), dtype=torch.int32, device=dev)
        o = torch.empty((n_q, wl.H, wl.dv), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((n_q, wl.H), device=dev)
        for _ in range(2):
            dsa.dsa_indexer_topk(idx.q_idx, idx.w, idx.k_idx, cu, n_req, pos, bid, wl.topk,
                                 max_ctx, topk, ws, block_table=bt)
            dsa.dsa_sparse_mla_balanced(mi.q, mi.c, cu, n_req, bid, pos, topk, wl.scale, o, mws,
                                        lse=lse, block_table=bt)
        torch.cuda.synchronize()
        print(json.dumps({"profile_decode": "64 requests x 2 queries, paged", "queries": n_q,
                          "cached_tokens": int(sum(wl.lengths)),
                          "device_errors": dsa.dsa_read_device_errors()}))
        return
    if args.profile_steps:
        st = ConfigStep(torch, dsa, W, WORKLOAD_ID, dev)
        torch.cuda.synchronize()
        for _ in range(1 + args.profile_steps):
            st.run()
        torch.cuda.synchronize()
        print(json.dumps({"profile_steps": args.profile_steps, "launches_per_step":
                          st.launches_per_step, "device_errors": dsa.dsa_read_device_errors()}))
        return
    wl = W.WORKLOADS[WORKLOAD_ID]
    r = 1
    cu_np = W.cu_seqlens(wl.lengths)
    n_tok = int(cu_np[-1])
    n_r = dsa.dsa_rr_shard_len(n_tok, wl.sp, r)
    cu = torch.as_tensor(cu_np, device=dev)
    e = lambda *sh, dt=torch.int32: torch.empty(*sh, dtype=dt, device=dev)
    pos, bid = e(n_r), e(n_r)
    dsa.dsa_rr_split_metadata(cu, n_tok, wl.sp, r, e(len(cu_np)), pos, bid)
    sel = torch.as_tensor(np.unique(np.linspace(0, n_r - 1, 2048).round().astype(np.int64)), device=dev)
    idx = W.indexer_inputs(wl, n_r, n_tok, r, device=dev)
    mi = W.mla_inputs(wl, n_r, n_tok, r, device=dev)
    q_idx, w, q = idx.q_idx[sel].contiguous(), idx.w[sel].contiguous(), mi.q[sel].contiguous()
    k_idx, c = idx.k_idx, mi.c
    del idx, mi
    pos, bid = pos[sel].contiguous(), bid[sel].contiguous()
    n = int(sel.numel())
    torch.cuda.empty_cache()
    max_ctx = int(max(wl.lengths))
    ws = e(dsa.dsa_indexer_topk_workspace_size(n, max_ctx, wl.topk), dt=torch.uint8)
    topk = e(n, wl.topk)
    o = e(n, wl.H, wl.dv, dt=torch.bfloat16)
    lse = e(n, wl.H, dt=torch.float32)
    mws = e(dsa.dsa_sparse_mla_workspace_size(n), dt=torch.uint8)
    q8 = e(*q_idx.shape, dt=torch.uint8)
    qs = e(*q_idx.shape[:2], dt=torch.float32)
    k8 = e(*k_idx.shape, dt=torch.uint8)
    ks = e(k_idx.shape[0], dt=torch.float32)
    topk8 = e(n, wl.topk)
    for _ in range(2):
        dsa.dsa_indexer_topk(q_idx, w, k_idx, cu, len(wl.lengths), pos, bid, wl.topk, max_ctx,
                             topk, ws)
        dsa.dsa_sparse_mla_balanced(q, c, cu, len(wl.lengths), bid, pos, topk, wl.scale, o, mws,
                                    lse=lse)
        dsa.dsa_quantize_fp8_rows(q_idx, q8, qs)
        dsa.dsa_quantize_fp8_rows(k_idx, k8, ks)
        dsa.dsa_indexer_topk_fp8(q8, qs, w, k8, ks, cu, len(wl.lengths), pos, bid, wl.topk,
                                 max_ctx, topk8, ws)
    torch.cuda.synchronize()
    p = pos.cpu().numpy().astype(np.int64)
    print(json.dumps({"profile_case": "many_req rank 1, 2048 evenly spaced queries",
                      "queries": n, "causal_pairs": int(np.sum(p + 1)),
                      "indexer_pairs": int(np.sum((p + 1)[p + 1 > wl.topk])),
                      "selected_pairs": int(np.sum(np.minimum(p + 1, wl.topk))),
                      "device_errors": dsa.dsa_read_device_errors()}))


def gather_probe(args):
    """Rate of the sparse MLA's row gather on its own: 152 CTAs (one per SM) each fill a 3-slot
    ring of 48-row x 576-column bf16 tiles from uniform random rows of the many-request batch's
    latent cache (71,014 rows x 1,152 B, inside L2), by 16-byte cp.async (the kernel's path) and
    by TMA tile::gather4 with 1, 4, 12 or 32 issuing lanes. One JSON line per variant."""
    import torch
    import __graft_entry__ as ge
    ge.build()
    import deepseek_v3_sparse_round_gb300 as dsa
    import workloads as W
    wl = W.WORKLOADS[WORKLOAD_ID]
    n_rows = int(sum(wl.lengths))
    n_ctas = torch.cuda.get_device_properties(0).multi_processor_count
    n_tiles = args.gather_probe
    g = torch.Generator(device="cpu").manual_seed(7)
    c = torch.randn(n_rows, 576, generator=g).to(torch.bfloat16).cuda()
    rows = torch.randint(0, n_rows, (n_ctas * n_tiles * 48,), generator=g, dtype=torch.int32).cuda()
    cycles = torch.zeros(n_ctas, dtype=torch.int64, device="cuda")
    tile_bytes = 48 * 1152
    variants = [(n_ctas, 0, 0), (n_ctas, 1, 1), (n_ctas, 1, 4), (n_ctas, 1, 12), (n_ctas, 1, 32),
                (n_ctas, 2, 0), (n_ctas // 2, 0, 0), (n_ctas // 4, 0, 0), (n_ctas, 4, 0),
                (n_ctas // 2, 4, 0), (n_ctas, 6, 0), (n_ctas, 5, 0), (n_ctas, 3, 0),
                (n_ctas, 7, 0), (n_ctas // 2, 7, 0)]
    for ctas, mode, issuers in variants:
        ms = []
        for rep in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            dsa.dsa_probe_row_gather(c, rows[:ctas * n_tiles * 48], ctas, n_tiles, mode,
                                     max(issuers, 1), cycles[:ctas])
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        cyc = float(cycles[:ctas].double().mean())
        if mode == 3:                                # 192 KB into (and out of) each SM a round
            rounds_bytes = n_tiles * 192 * 1024
            print(json.dumps({
                "dsmem_probe": "bulk copies between the CTAs of each pair, 6 x 32 KB per round",
                "ctas": ctas, "rounds": n_tiles,
                "bytes_per_clk_per_sm_in": round(rounds_bytes / cyc, 2),
                "gb_per_s": round(ctas * rounds_bytes / sorted(ms[1:])[0] / 1e6, 1),
                "device_errors": dsa.dsa_read_device_errors()}), flush=True)
            continue
        t = sorted(ms[1:])[0]
        how = {0: "cp.async 16 B, 3 warps per slot",
               4: "ld.global 16 B + st.shared, 3 warps per slot",
               5: "ld.global + st.shared for columns 0-319, cp.async for 320-575",
               6: "ld.global 16 B + st.shared, every row of a warp in flight",
               1: f"TMA tile::gather4, {issuers} issuing lane(s)",
               2: "cp.async for columns 0-511 + TMA tile::gather4 for 512-575",
               7: "TMA tiled boxes of 48 consecutive rows (not a gather)"}[mode]
        print(json.dumps({
            "gather_probe": how,
            "ctas": ctas, "tiles_per_cta": n_tiles, "tile": "48 rows x 1,152 B (9 SW128 atoms)",
            "bytes_per_clk_per_sm": round(n_tiles * tile_bytes / cyc, 2),
            "cycles_per_tile": round(cyc / n_tiles, 1),
            "gb_per_s": round(ctas * n_tiles * tile_bytes / t / 1e6, 1), "ms": round(t, 4),
            "device_errors": dsa.dsa_read_device_errors()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=128, help="queries per reference-arm step")
    ap.add_argument("--cpu-baseline-queries", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the long-prompt line")
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--next-rows", nargs="?", const="all", default=None,
                    help="measure the widened rows (paged rerange, decode split) and exit")
    ap.add_argument("--configs", action="store_true",
                    help="indexer + top-k + sparse MLA on every workload config, then exit")
    ap.add_argument("--with-oracle", action="store_true",
                    help="with --configs: also time the fp64 oracle on a sample of each config")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="ncu launch list: 1 + K default-workload steps, nothing else, then exit")
    ap.add_argument("--profile-case", action="store_true",
                    help="ncu capture: one 2,048-query cut of a many-request shard, then exit")
    ap.add_argument("--profile-decode", action="store_true",
                    help="ncu capture: the paged decode batch's indexer + top-k and MLA, twice")
    ap.add_argument("--gather-probe", type=int, nargs="?", const=400, default=0,
                    help="row-gather rate probe, cp.async vs TMA gather4 (tiles per CTA), then exit")
    args = ap.parse_args()
    if args.gather_probe:
        gather_probe(args)
        return
    if args.profile_steps or args.profile_case or args.profile_decode:
        profile_run(args)
        return
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
