#!/usr/bin/env python3
"""Benchmark of one MLA tree-verify attention step on GB300.

Headline workload (the largest one-GPU configuration): the batched ragged
step -- 8 requests, H=64 heads, T=16 random draft-tree nodes each, prefixes
drawn uniformly from [1024, 65536], bf16 latent KV gathered through a
page_size=1 slot table scattered over one shared 2^20-slot pool, steps
captured and replayed in CUDA graphs.  A step is one verify call: split-K
partial attention (tree masks computed inside) and the LSE merge.

Prints ONE JSON line: effective KV GB/s (whole job), us/step, the split-K
kernel's roofline fraction (tensor-bound at H=64), the target points (H=8 and
H=64 at prefixes 16k, 65k and 200k, scattered and contiguous) with their
kernel-level fractions, the oracle timed on the host cores, an end-to-end
figure through the C ABI with host buffers, clocks and launches.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "verify-attn µs/step and effective KV GB/s (% of HBM roofline) vs prefix length"
HEADLINE = "batched"
WORKLOAD = ("batched ragged: 8 requests, H=64, T=16 random trees, prefixes U[1024, 65536] "
            "(seeded: 14817, 40180, 26978, 43472, 28365, 46466, 13339, 17238), bf16 latent KV "
            "(576 = 512 + 64), page_size=1 slots scattered over one shared 2^20-slot pool, "
            "sm_scale=1/sqrt(192), captured and replayed in CUDA graphs")
TARGET_P = [16384, 65536, 200000]
SWEEP_P = [4096, 32768, 131072]


def headline_config(step=None) -> dict:
    """The `config` object of both arms' lines (the same dict, so the two
    describe one workload)."""
    s = synth.spec(HEADLINE)
    cfg = {"workload": WORKLOAD, "B": s.B, "H": s.H, "T": s.T, "prefix": list(s.prefix),
           "layout": "scattered", "pool_slots": s.num_slots,
           "kv_bytes_per_step": s.kv_bytes()}
    return cfg


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 FMA, 2 tensor cores")
    ap.add_argument("--nsplit", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--case", default="",
                    help="'batched' or H,prefix,layout[,T]: run only --warmup + --steps plain "
                         "calls of that workload (the captures the ncu summaries are made "
                         "from); prints a timing note, not the benchmark line")
    return ap.parse_args()


KERNEL_SOURCES = ("va_tc.cu", "va_common.cuh", "va_sm100.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "partial_tc_traffic.json")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mla_speculative_decode_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes per launch of the split-K kernel on the benchmark workload,
    from the committed ncu capture -- or None when the kernel sources changed
    since that capture (the counters no longer describe this kernel)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])


def run_case(va, args, dev):
    """A few plain verify calls of one workload, for profiler captures:
    `--case batched` (the headline step) or `--case H,prefix,layout[,T]`."""
    if args.case == HEADLINE:
        s = synth.spec(HEADLINE)
        pool = device_pool(s.num_slots, seed=1, dev=dev)
        st = Step(va, pool, s.H, s.T, list(s.prefix), seed=4, nrot=2, dev=dev, path=args.path,
                  nsplit=args.nsplit)
        label = HEADLINE
    else:
        parts = args.case.split(",")
        H, P, layout = int(parts[0]), int(parts[1]), parts[2]
        T = int(parts[3]) if len(parts) > 3 else 16
        rows = 1 << 18
        while rows < 2 * (P + T):
            rows *= 2
        pool = device_pool(rows, seed=1, dev=dev)
        st = Step(va, pool, H, T, P, seed=7, nrot=2, dev=dev, path=args.path, nsplit=args.nsplit,
                  layout=layout)
        label = f"H={H} T={T} P={P} {layout}"
    for k in range(args.warmup):
        st.call(k)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for k in range(args.steps):
        st.call(k)
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / max(1, args.steps) * 1e3
    print(f"case {label} nsplit={st.nsplit}: {us:.2f} us/call "
          f"(eager launches, not the benchmark figure)", flush=True)


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x: the job takes as long as its slowest rank."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, bytes_per_rank_step: int, steps: int, ms: float) -> float:
    """Whole-job GB/s of `world` replicas, each moving bytes_per_rank_step per step,
    `steps` steps in `ms` (the slowest rank's time): weak scaling."""
    return world * bytes_per_rank_step * steps / (ms / 1e3) / 1e9


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0=None, t1=None):
        rows = []
        for ts, line in self.lines:
            if t0 is not None and not (t0 <= ts <= t1 + 0.15):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i] == "Active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# -------------------------------------------------------------- workload

def device_pool(num_slots: int, seed: int, dev) -> torch.Tensor:
    """The shared latent pool, drawn on the device (seeded) in chunks."""
    g = torch.Generator(device=dev).manual_seed(seed)
    pool = torch.empty(num_slots, synth.D_QK, dtype=torch.bfloat16, device=dev)
    step = 1 << 17
    for r0 in range(0, num_slots, step):
        r1 = min(num_slots, r0 + step)
        pool[r0:r1] = torch.randn(r1 - r0, synth.D_QK, generator=g, device=dev).to(torch.bfloat16)
    return pool


class Step:
    """Device-resident inputs of one verify step plus `nrot` rotated slot tables
    (disjoint random subsets of the pool) so that consecutive steps read rows
    that are not in L2.  `P` is one prefix length or a list, one per request
    (requests take disjoint slots of the shared pool)."""

    def __init__(self, va, pool, H, T, P, seed, nrot, dev, path, nsplit, layout="scattered"):
        self.va = va
        self.pool = pool
        prefixes = [int(P)] if isinstance(P, int) else [int(x) for x in P]
        B = len(prefixes)
        self.B, self.H, self.T, self.P = B, H, T, prefixes[0]
        Ns = [x + T for x in prefixes]
        self.N = sum(Ns)
        g = torch.Generator().manual_seed(seed)
        self.q = (torch.randn(B * T, H, synth.D_QK, generator=g)).to(torch.bfloat16).to(dev)
        self.parents = torch.stack([synth.make_parents(T, "random", g) for _ in range(B)]).to(dev)
        perm = torch.randperm(pool.shape[0], generator=g)
        if nrot * self.N > pool.shape[0]:
            nrot = max(1, pool.shape[0] // self.N)
        self.nrot = nrot
        self.layout = layout
        self.tables = [perm[k * self.N:(k + 1) * self.N].to(torch.int32).to(dev)
                       for k in range(nrot)]
        offs = [0]
        for n in Ns:
            offs.append(offs[-1] + n)
        # contiguous layout: rotation k reads pool rows [k*N, (k+1)*N), request
        # b from k*N + offs[b]
        self.starts = [torch.tensor([k * self.N + o for o in offs[:-1]], dtype=torch.int64,
                                    device=dev) for k in range(nrot)]
        self.indptr = torch.tensor(offs, dtype=torch.int32, device=dev)
        self.prefix = torch.tensor(prefixes, dtype=torch.int32, device=dev)
        self.path = path
        self.ws, self.nsplit = va.alloc_workspace(B, T, H, nsplit, path, dev)
        self.out = torch.empty(B * T, H, synth.D_V, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(B * T, H, dtype=torch.float32, device=dev)
        if layout in ("segmented", "segmented_append"):
            # the extend call's two lists: prefix slots (kv_indices) and the
            # draft nodes' slots (out_cache_loc), and its dense mask rows
            # (prefix columns visible, draft columns the node's ancestors and
            # itself, from a walk up the parent links)
            self.seg_indptr = torch.tensor([0] + list(np.cumsum(prefixes)), dtype=torch.int32,
                                           device=dev)
            self.seg_ind, self.seg_loc = [], []
            for t in self.tables:
                t = t.cpu()
                self.seg_ind.append(torch.cat([t[offs[b]:offs[b] + prefixes[b]]
                                               for b in range(B)]).to(dev))
                self.seg_loc.append(torch.cat([t[offs[b] + prefixes[b]:offs[b + 1]]
                                               for b in range(B)]).to(dev))
            par = self.parents.cpu().tolist()
            rows = []
            for b in range(B):
                for i in range(T):
                    r = np.zeros(prefixes[b] + T, dtype=np.uint8)
                    r[:prefixes[b]] = 1
                    k = i
                    while 0 <= k < T:
                        r[prefixes[b] + k] = 1
                        k = par[b][k] if par[b][k] < k else -1
                    rows.append(r)
            self.mask = torch.from_numpy(np.concatenate(rows)).to(dev)
            # the draft tokens' new latents, written into their slots by the call
            self.draft = ((torch.randn(B * T, synth.D_QK, generator=g)).to(torch.bfloat16).to(dev)
                          if layout == "segmented_append" else None)
        self.prefixes = prefixes
        self.offs = offs
        self.kv_bytes = self.N * synth.D_QK * 2
        # algorithmic tensor work: 2176 flop (2*576 + 2*512) per visible
        # (row, key) pair -- every prefix key, plus each node's ancestors and
        # itself among the draft keys
        par = self.parents.cpu().tolist()
        pairs = 0
        for b in range(B):
            for i in range(T):
                k, depth = i, 0
                while 0 <= k < T:
                    depth += 1
                    k = par[b][k] if par[b][k] < k else -1
                pairs += H * (prefixes[b] + depth)
        self.visible_pairs = pairs
        self.flops = 2176.0 * pairs

    def table_rows(self, k: int) -> torch.Tensor:
        """Pool rows (int64) of rotation k's keys, requests one after the other."""
        if self.layout == "contiguous":
            return torch.arange(k % self.nrot * self.N, (k % self.nrot + 1) * self.N,
                                dtype=torch.int64, device=self.pool.device)
        return self.tables[k % self.nrot].long()

    def call(self, k, stream=None):
        if self.layout in ("segmented", "segmented_append"):
            self.va.verify_attn_segmented(self.q, self.pool, self.seg_ind[k % self.nrot],
                                          self.seg_indptr, self.seg_loc[k % self.nrot],
                                          custom_mask=self.mask, draft_kv=self.draft,
                                          sm_scale=synth.SM_SCALE,
                                          nsplit=self.nsplit, flags=self.path, workspace=self.ws,
                                          out=self.out, lse=self.lse, stream=stream)
            return
        if self.layout == "contiguous":
            self.va.verify_attn_contiguous(self.q, self.pool, self.starts[k % self.nrot],
                                           self.prefix, self.parents, sm_scale=synth.SM_SCALE,
                                           nsplit=self.nsplit, flags=self.path, workspace=self.ws,
                                           out=self.out, lse=self.lse, stream=stream)
            return
        self.va.verify_attn_paged(self.q, self.pool, self.tables[k % self.nrot], self.indptr,
                                  self.prefix, self.parents, sm_scale=synth.SM_SCALE,
                                  nsplit=self.nsplit, flags=self.path, workspace=self.ws,
                                  out=self.out, lse=self.lse, stream=stream)


# Steps per CUDA graph.  A graph boundary costs the overlap of consecutive
# steps (the next step's split-K kernel cannot start while this graph's last
# merge runs; in the end-to-end leg each graph also joins its copy streams, so
# the next graph's first upload cannot overlap this graph's last kernels).
# Measured with 8 and 40 steps per graph: TP8 slice 15.64 -> 15.33 us, H=8
# P=16384 contiguous 18.53 -> 18.17 us, batched step unchanged (535.5 us),
# batched end to end 553.5 -> 543.9 us.
STEPS_PER_GRAPH = 40
E2E_STEPS_PER_GRAPH = STEPS_PER_GRAPH


def capture_graphs(step: Step, K: int, with_events: bool = False):
    """CUDA graphs over the rotated slot tables: graphs of STEPS_PER_GRAPH
    consecutive steps (each on its own table), as a serving loop would capture
    them, and -- when K is not a multiple of that -- one graph of the
    K % STEPS_PER_GRAPH remaining steps, so that exactly K steps can be
    replayed.  With events:
    one-step graphs with event records around the split-K kernel instead."""
    va = step.va
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for k in range(min(step.nrot, 3)):
            step.call(k)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    if with_events:
        graphs, evs = [], []
        for gi in range(min(step.nrot, 8)):
            g = torch.cuda.CUDAGraph()
            eb = torch.cuda.Event(enable_timing=True)
            ea = torch.cuda.Event(enable_timing=True)
            va.set_partial_events(eb, ea)
            evs.append((eb, ea))
            with torch.cuda.graph(g):
                step.call(gi)
            graphs.append(g)
        va.set_partial_events(None, None)
        return graphs, evs
    per = STEPS_PER_GRAPH
    full = []
    for gi in range(max(1, step.nrot // per)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(per):
                step.call(gi * per + j)
        full.append(g)
    tail = None
    if K % per:
        tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tail):
            for j in range(K % per):
                step.call(j)
    return (full, tail), None


def replay_steps(graphs, K: int):
    """Replays exactly K steps: K // STEPS_PER_GRAPH full graphs, then the tail graph."""
    full, tail = graphs
    for r in range(K // STEPS_PER_GRAPH):
        full[r % len(full)].replay()
    if K % STEPS_PER_GRAPH:
        tail.replay()


def time_steps(graphs, K: int, W: int, dist=None) -> float:
    """ms for exactly K timed steps after at least W warm-up steps; barrier and
    device synchronisation on both sides of the timed region."""
    assert W >= 1
    replay_steps(graphs, -(-W // STEPS_PER_GRAPH) * STEPS_PER_GRAPH)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    replay_steps(graphs, K)
    e1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def partial_kernel_us(step: Step) -> float:
    """Average duration of the split-K kernel (CUDA events recorded by the
    library on the launching stream around it), over one-step graphs replayed
    twice after the timed region."""
    egraphs, evs = capture_graphs(step, 1, with_events=True)
    for _ in range(2):
        for g in egraphs:
            g.replay()
    torch.cuda.synchronize()
    us = float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3
    del egraphs
    return us


def measure_dist(step: Step, K: int, W: int, runs: int = 5):
    """Per-step µs of `runs` timed runs of K steps each: (median, p10, p90), and
    the split-K kernel µs."""
    graphs, _ = capture_graphs(step, K)
    vals = [time_steps(graphs, K, W if i == 0 else 1) / K * 1e3 for i in range(runs)]
    del graphs
    k_us = partial_kernel_us(step)
    v = np.array(vals)
    return float(np.median(v)), float(np.percentile(v, 10)), float(np.percentile(v, 90)), k_us


def point_record(step: Step, us: float, p10: float, p90: float, k_us: float, hbm_peak: float,
                 tc_peak: float) -> dict:
    """One measured point: step and split-K kernel figures against both roofs."""
    kvb = step.kv_bytes
    return {"us_per_step": us, "p10": p10, "p90": p90,
            "gbs": kvb / (us * 1e-6) / 1e9, "frac_hbm": kvb / (us * 1e-6) / 1e9 / hbm_peak,
            "tflops": step.flops / (us * 1e-6) / 1e12,
            "frac_tensor": step.flops / (us * 1e-6) / 1e12 / tc_peak,
            "kernel_us": k_us, "kernel_gbs": kvb / (k_us * 1e-6) / 1e9,
            "kernel_frac_hbm": kvb / (k_us * 1e-6) / 1e9 / hbm_peak,
            "kernel_tflops": step.flops / (k_us * 1e-6) / 1e12,
            "kernel_frac_tensor": step.flops / (k_us * 1e-6) / 1e12 / tc_peak,
            "nsplit": step.nsplit, "kv_bytes": kvb, "flops": step.flops}


# --------------------------------------------------------------- oracle

def sample_rows_by_work(step: Step, budget_pairs: float, seed: int):
    """Query rows of a step sampled at random until their visible (row, key)
    pairs reach `budget_pairs`; returns (rows, fraction of the step's pairs)."""
    par = step.parents.cpu().tolist()
    rows_total = step.B * step.T * step.H
    rng = np.random.default_rng(seed)
    order = rng.permutation(rows_total)
    got, pairs = [], 0
    for r in order:
        b, i = divmod(int(r) // step.H, step.T)
        k, depth = i, 0
        while 0 <= k < step.T:
            depth += 1
            k = par[b][k] if par[b][k] < k else -1
        got.append(int(r))
        pairs += step.prefixes[b] + depth
        if pairs >= budget_pairs:
            break
    return np.sort(np.array(got, dtype=np.int64)), pairs / step.visible_pairs


def oracle_inputs(step: Step, k: int):
    """Host copies of step k's inputs for the oracle: the queries, the rows the
    step reads (compacted, in slot-table order), the bounds and the masks."""
    import oracle
    rows_kv = step.pool[step.table_rows(k)].cpu()
    bits, _ = oracle.tree_bits(step.parents.cpu().numpy())
    return (synth.as_u16(step.q.cpu()), synth.as_u16(rows_kv), np.arange(step.N, dtype=np.int32),
            np.array(step.offs, dtype=np.int64), np.array(step.prefixes, dtype=np.int64), bits)


def cpu_baseline_leg(step: Step, budget_s: float = 12.0, threads=None):
    """The fp64 oracle, as it stands, on the host cores: a bounded sample of
    rows of step 0 of the headline workload (about `budget_s` of work), scaled
    to the metric by the sample's share of the step's visible (row, key)
    pairs.  The same rows of the GPU's step 0 are compared with it (the
    parity spot check of the line)."""
    import oracle
    oracle.build()
    threads = threads or oracle.default_threads()
    step.call(0)
    torch.cuda.synchronize()
    go_all = step.out.float().reshape(-1, synth.D_V).cpu().numpy()
    gl_all = step.lse.reshape(-1).cpu().numpy()
    q, kv, slots, indptr, prefix, bits = oracle_inputs(step, 0)
    # calibrate on 1 % of the step's work, then take a sample sized to the
    # budget (at most the whole step)
    rows, frac = sample_rows_by_work(step, step.visible_pairs * 0.01, seed=11)
    t0 = time.perf_counter()
    oracle.verify_attn(q, kv, slots, indptr, prefix, bits, synth.SM_SCALE, rows=rows,
                       threads=threads)
    t_cal = max(time.perf_counter() - t0, 1e-3) / frac      # seconds per whole step
    share = min(1.0, budget_s / t_cal)
    rows, frac = sample_rows_by_work(step, step.visible_pairs * share, seed=12)
    t0 = time.perf_counter()
    ro, rl, _ = oracle.verify_attn(q, kv, slots, indptr, prefix, bits, synth.SM_SCALE, rows=rows,
                                   threads=threads)
    el = time.perf_counter() - t0
    per_step = el / frac
    go, gl = go_all[rows], gl_all[rows]
    err = float(np.abs(go - ro).max())
    mean = float(np.abs(go - ro).mean())
    lerr = float(np.abs(gl - rl).max())
    parity = {"rows": int(len(rows)), "max_abs": err, "mean_abs": mean, "lse_max_abs": lerr,
              "ok": bool(err <= 2e-2 and mean <= 2e-3 and lerr <= 1e-3)}
    cpu = {"value": step.kv_bytes / per_step / 1e9, "unit": "GB/s", "cores": int(threads),
           "kind": "oracle", "us_per_step": per_step * 1e6,
           "sample": f"{len(rows)} of {step.B * step.T * step.H} query rows of one step "
                     f"({frac * 100:.2f} % of its visible (row, key) pairs), fp64, {el:.1f} s; "
                     f"scaled to a whole step by that share"}
    return cpu, parity


def reference_arm(args, rank):
    """--impl reference: the fp64 oracle on the host cores, on the headline
    workload; each step a bounded sample of its query rows (the same rows every
    step), its throughput scaled to a whole step by the sample's share of the
    visible (row, key) pairs."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    s = synth.spec(HEADLINE)
    total = sum(s.n_keys())
    w = synth.make(synth.spec(HEADLINE, num_slots=total))   # a compact pool: the rows used
    bits, _ = oracle.tree_bits(w.parents.numpy())
    q, kv = synth.as_u16(w.q), synth.as_u16(w.kv_pool)
    slots, indptr, prefix = w.slot_idx.numpy(), w.kv_indptr.numpy(), w.prefix_len.numpy()
    par = w.parents.tolist()
    pairs_all, row_pairs = 0, []
    for b in range(s.B):
        for i in range(s.T):
            k, depth = i, 0
            while 0 <= k < s.T:
                depth += 1
                k = par[b][k] if par[b][k] < k else -1
            for _ in range(s.H):
                row_pairs.append(s.prefix[b] + depth)
                pairs_all += s.prefix[b] + depth
    rng = np.random.default_rng(5)
    rows, got = [], 0
    for r in rng.permutation(len(row_pairs)):      # about 2 % of the step's work
        rows.append(int(r))
        got += row_pairs[r]
        if got >= pairs_all * 0.02 and len(rows) >= 4 * threads:
            break
    rows = np.sort(np.array(rows, dtype=np.int64))
    frac = got / pairs_all

    def one():
        oracle.verify_attn(q, kv, slots, indptr, prefix, bits, s.sm_scale, rows=rows,
                           threads=threads)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    ms = el / args.steps / frac * 1e3          # per whole step
    val = s.kv_bytes() / (ms / 1e3) / 1e9
    sample = (f"each step: {len(rows)} of {s.B * s.T * s.H} query rows ({frac * 100:.3f} % of "
              f"the visible (row, key) pairs), fp64 on {threads} host threads; scaled to a "
              f"whole step by that share")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ end to end

def e2e_leg(va, step: Step, K: int, W: int, dist, dev):
    """The headline metric end to end through the public API with host
    buffers.  Every step: its inputs (q, slot table, indptr, prefix lengths,
    parents), packed in one pinned host buffer, are copied to the device with
    one host-to-device copy; the verify call runs on views of that device
    buffer; out and lse, views of one device result buffer, are read back with
    one device-to-host copy into pinned memory.  Two input and two result
    buffers alternate, and the copies run on their own streams, so step k+1's
    upload and step k-1's read-back overlap step k's kernels.  Steps are
    captured E2E_STEPS_PER_GRAPH to a CUDA graph (streams forked and joined
    inside the capture; a last graph holds the remainder) and replayed;
    exactly K steps are timed."""
    def align(n):
        return (n + 255) // 256 * 256

    parts = [("q", step.q), ("tab", step.tables[0]), ("par", step.parents),
             ("ind", step.indptr), ("pre", step.prefix)]
    offs, o = {}, 0
    for name, t in parts:
        offs[name] = (o, t.numel() * t.element_size())
        o = align(o + t.numel() * t.element_size())
    in_bytes = o

    def pack(tab):
        hb = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        for name, t in parts:
            src = tab if name == "tab" else t
            off, n = offs[name]
            hb[off:off + n] = src.detach().cpu().contiguous().view(-1).view(torch.uint8)
        return hb

    hins = [pack(t) for t in step.tables]
    o_bytes = step.out.numel() * step.out.element_size()
    l_off = align(o_bytes)
    res_bytes = l_off + step.lse.numel() * step.lse.element_size()
    dbufs = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    dress = [torch.empty(res_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    hress = [torch.empty(res_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    s_cmp, s_up, s_dn = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def dview(buf, name, like):
        off, n = offs[name]
        return buf[off:off + n].view(like.dtype).view(like.shape)

    calls = []
    for j in range(2):
        dout = dress[j][:o_bytes].view(step.out.dtype).view(step.out.shape)
        dlse = dress[j][l_off:res_bytes].view(step.lse.dtype).view(step.lse.shape)
        calls.append(va.prepare_paged(dview(dbufs[j], "q", step.q), step.pool,
                                      dview(dbufs[j], "tab", step.tables[0]),
                                      dview(dbufs[j], "ind", step.indptr),
                                      dview(dbufs[j], "pre", step.prefix),
                                      dview(dbufs[j], "par", step.parents),
                                      sm_scale=synth.SM_SCALE, nsplit=step.nsplit,
                                      flags=step.path, workspace=step.ws, out=dout, lse=dlse,
                                      stream=s_cmp))

    def run_steps(k0: int, n: int, origin):
        """Enqueue steps k0 .. k0+n-1; `origin` is the stream the work forks
        from and joins back to (the capturing stream inside a capture)."""
        ev_in = [None, None]     # buffer j's inputs consumed (its last call done)
        ev_out = [None, None]    # result buffer j read back
        start = torch.cuda.Event()
        start.record(origin)
        for s_ in (s_cmp, s_up, s_dn):
            s_.wait_event(start)
        for k in range(k0, k0 + n):
            j = k % 2
            up = torch.cuda.Event()
            with torch.cuda.stream(s_up):
                if ev_in[j] is not None:
                    s_up.wait_event(ev_in[j])
                dbufs[j].copy_(hins[k % len(hins)], non_blocking=True)
                up.record(s_up)
            s_cmp.wait_event(up)
            if ev_out[j] is not None:
                s_cmp.wait_event(ev_out[j])
            calls[j]()
            done = torch.cuda.Event()
            done.record(s_cmp)
            ev_in[j] = done
            with torch.cuda.stream(s_dn):
                s_dn.wait_event(done)
                hress[j].copy_(dress[j], non_blocking=True)
                dn = torch.cuda.Event()
                dn.record(s_dn)
            ev_out[j] = dn
        for s_ in (s_cmp, s_up, s_dn):
            e = torch.cuda.Event()
            e.record(s_)
            origin.wait_event(e)

    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    # eager warm-up, and a check that the copy path computes the same step
    run_steps(0, 2, cap)
    torch.cuda.synchronize()
    ref0 = dress[0].clone()
    step.call(0)
    torch.cuda.synchronize()
    dout0 = ref0[:o_bytes].view(step.out.dtype).view(step.out.shape)
    dlse0 = ref0[l_off:res_bytes].view(step.lse.dtype).view(step.lse.shape)
    assert torch.equal(dout0, step.out) and torch.equal(dlse0, step.lse), "e2e path differs"
    assert torch.equal(hress[0], ref0.cpu()), "e2e read-back differs"
    per = E2E_STEPS_PER_GRAPH
    graphs = []
    for gi in range(max(1, min(4, len(hins) // per))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            run_steps(gi * per, per, cap)
        graphs.append(g)
    tail = None
    if K % per:
        tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tail, stream=cap):
            run_steps(0, K % per, cap)
    with torch.cuda.stream(cap):
        for r in range(max(1, -(-W // per))):
            graphs[r % len(graphs)].replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        a.record()
        for r in range(K // per):
            graphs[r % len(graphs)].replay()
        if tail is not None:
            tail.replay()
        b.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e_ms = max_over_ranks(a.elapsed_time(b) / K, dist, dev)
    world = dist.get_world_size() if dist is not None else 1
    return {"value": job_gbs(world, step.kv_bytes, 1, e_ms), "unit": "GB/s",
            "us_per_step": e_ms * 1e3, "steps": K, "h2d_bytes_per_step": int(in_bytes),
            "d2h_bytes_per_step": int(res_bytes),
            "note": "every step: its inputs packed in one pinned buffer and copied in (one H2D "
                    "copy), the verify call (prepared once with va.prepare_paged) launched, out "
                    "and lse read back (one D2H copy); two buffer sets alternate so that the "
                    "copies of neighbouring steps overlap a step's kernels on separate streams; "
                    f"steps captured {E2E_STEPS_PER_GRAPH} to a CUDA graph (the remainder in one "
                    "more) and replayed"}


# ------------------------------------------------------------------ main

def bench_accept(va, dev, hbm_peak) -> dict:
    """Greedy tree acceptance after verify: B=8 requests, T=16 nodes, a
    129280-token vocabulary, fp32 logits (one row after the prefix and one per
    node); rotated logits buffers larger than L2 together, CUDA graphs of 8
    calls."""
    ga = torch.Generator().manual_seed(9)
    Ba, Ta, Va = 8, 16, 129280
    nbuf = max(2, math.ceil(3 * torch.cuda.get_device_properties(dev).L2_cache_size
                            / (Ba * (Ta + 1) * Va * 4)))
    bufs = [(torch.randn(Ba, Va, generator=ga).to(dev), torch.randn(Ba, Ta, Va, generator=ga).to(dev))
            for _ in range(nbuf)]
    par_a = torch.stack([synth.make_parents(Ta, "random", ga) for _ in range(Ba)]).to(dev)
    tok_a = torch.randint(0, Va, (Ba, Ta), generator=ga, dtype=torch.int32).to(dev)
    slot_a = torch.arange(Ba * Ta, dtype=torch.int32, device=dev).reshape(Ba, Ta)
    res = va.tree_accept(bufs[0][0], bufs[0][1], tok_a, par_a, slot_a)
    ws_a, outs_a = res[4], res[:4]
    sa = torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    ga_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga_graph, stream=sa):
        for k in range(8):
            va.tree_accept(bufs[k % nbuf][0], bufs[k % nbuf][1], tok_a, par_a, slot_a,
                           workspace=ws_a, outputs=outs_a, stream=sa)
    for _ in range(3):
        ga_graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    e0.record()
    for _ in range(reps):
        ga_graph.replay()
    e1.record()
    torch.cuda.synchronize()
    a_us = e0.elapsed_time(e1) / (8 * reps) * 1e3
    a_bytes = Ba * (Ta + 1) * Va * 4
    del bufs
    torch.cuda.empty_cache()
    return {"us": a_us, "logits_bytes": a_bytes, "gbs": a_bytes / (a_us * 1e-6) / 1e9,
            "frac_hbm": a_bytes / (a_us * 1e-6) / 1e9 / hbm_peak,
            "timing": "CUDA graphs of 8 calls on rotated logits buffers (> L2 together), events"}


def bench_tree_build(va, dev) -> dict:
    """Device-side draft tree and slot building: B=8 requests, D=8 draft
    positions with K=8 candidates each, T=16 nodes; CUDA graphs of 8 calls
    (the free-list head moves on with every call)."""
    rng = np.random.default_rng(21)
    B, D, K, T = 8, 8, 8, 16
    tok = torch.from_numpy(rng.integers(0, 129280, size=(B, D, K)).astype(np.int32)).to(dev)
    lp = torch.from_numpy(np.log(rng.dirichlet(np.ones(K), size=(B, D))).astype(np.float32)).to(dev)
    free = torch.randperm(1 << 20, dtype=torch.int32, device=dev)
    head = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = va.tree_build(tok, lp, T, free, head)
    s_ = torch.cuda.Stream()
    s_.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s_):
        for _ in range(8):
            va.tree_build(tok, lp, T, free, head, outputs=outs, stream=s_)
    head.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return {"us": e0.elapsed_time(e1) / (8 * reps) * 1e3, "B": B, "D": D, "K": K, "T": T,
            "timing": "CUDA graphs of 8 calls, events; the pages' host tree build took "
                      "1.8 ms per step (sm_120 service, context only)"}


def bench_defrag(va, pool, dev, hbm_peak) -> dict:
    """65536 scattered rows (lower half of the pool) compacted into a
    contiguous range in the upper half."""
    gd = torch.Generator().manual_seed(7)
    n = 65536
    src = torch.randperm(pool.shape[0] // 2, generator=gd)[:n].to(torch.int32).to(dev)
    sind = torch.tensor([0, n], dtype=torch.int32, device=dev)
    dstb = torch.tensor([pool.shape[0] // 2], dtype=torch.int64, device=dev)
    for _ in range(3):
        va.verify_attn_defrag(pool, src, sind, dstb)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record()
    for _ in range(reps):
        va.verify_attn_defrag(pool, src, sind, dstb)
    e1.record()
    torch.cuda.synchronize()
    d_us = e0.elapsed_time(e1) / reps * 1e3
    moved = 2 * n * synth.D_QK * 2
    return {"us": d_us, "bytes_moved": moved, "gbs": moved / (d_us * 1e-6) / 1e9,
            "frac_hbm": moved / (d_us * 1e-6) / 1e9 / hbm_peak}


def bench_contiguous_decode(va, dev, tc_peak) -> dict:
    """The headline workload's shapes (8 requests, H=64, T=16, the same
    prefixes) kept contiguous by the placement policy: each request owns a
    reserved range of rows; one decode step is the draft rows placed after the
    prefix, the contiguous verify and the compaction of a 3-node accepted path
    (the prefix lengths are restored at the start of every step, so every step
    is the same).  Timed as one-step CUDA graphs (events), beside the
    contiguous verify alone; the KV (266 MB) is larger than L2."""
    hs = synth.spec(HEADLINE)
    B, H, T = hs.B, hs.H, hs.T
    prefix = np.array(hs.prefix, dtype=np.int32)
    cap = prefix + 64
    starts = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    pool = device_pool(int(cap.sum()), seed=11, dev=dev)
    g = torch.Generator(device=dev).manual_seed(12)
    q = torch.randn(B * T, H, synth.D_QK, generator=g, device=dev).to(torch.bfloat16)
    draft = torch.randn(B * T, synth.D_QK, generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(13)
    par = np.full((B, T), -1, dtype=np.int32)
    for i in range(1, T):
        par[:, i] = rng.integers(-1, i, size=B)
    par[:, 1] = 0
    par[:, 2] = 1                                  # nodes 0 -> 1 -> 2 form the accepted path
    d_par = torch.from_numpy(par).to(dev)
    d_start = torch.from_numpy(starts).to(dev)
    d_cap = torch.from_numpy(cap).to(dev)
    pl0 = torch.from_numpy(prefix).to(dev)
    d_pl = pl0.clone()
    alen = torch.full((B,), 3, dtype=torch.int32, device=dev)
    nodes = torch.full((B, T), -1, dtype=torch.int32, device=dev)
    nodes[:, :3] = torch.arange(3, dtype=torch.int32, device=dev)
    loc = torch.empty(B * T, dtype=torch.int32, device=dev)
    ws, ns = va.alloc_workspace(B, T, H, 0, va.PATH_AUTO, dev)
    out = torch.empty(B * T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B * T, H, dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)

    def step(full: bool):
        d_pl.copy_(pl0)
        if full:
            va.kv_append_contiguous(pool, d_start, d_pl, d_cap, draft, loc, stream=st)
        va.verify_attn_contiguous(q, pool, d_start, d_pl, d_par, sm_scale=synth.SM_SCALE,
                                  nsplit=ns, workspace=ws, out=out, lse=lse, stream=st)
        if full:
            va.kv_compact_accepted(pool, d_start, d_pl, d_cap, alen, nodes, stream=st)

    res = {}
    for name, full in (("decode_step", True), ("verify_only", False)):
        st.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            step(full)                              # warm-up outside the capture
        st.synchronize()
        with torch.cuda.graph(graph, stream=st):
            step(full)
        for _ in range(5):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 50
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / reps * 1e3
        del graph
    # algorithmic flops of the verify: every prefix key and each node's
    # ancestors-or-self among the draft keys, for every row
    depth_set = np.zeros((B, T), dtype=np.int64)
    for b in range(B):
        for i in range(T):
            n, j = 1, par[b, i]
            while j >= 0:
                n, j = n + 1, par[b, j]
            depth_set[b, i] = n
    pairs = float(sum((prefix[b] * T + depth_set[b].sum()) * H for b in range(B)))
    flops = 2176.0 * pairs
    kv_bytes = float((prefix + T).sum()) * 1152
    return {"us_per_step": res["decode_step"], "verify_only_us": res["verify_only"],
            "placement_and_compaction_us": res["decode_step"] - res["verify_only"],
            "gbs": kv_bytes / (res["decode_step"] * 1e-6) / 1e9,
            "tflops": flops / (res["decode_step"] * 1e-6) / 1e12,
            "frac_tensor": flops / (res["decode_step"] * 1e-6) / 1e12 / tc_peak,
            "nsplit": ns, "timing": "one-step CUDA graphs, events; prefix lengths restored each step"}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
        dist = tdist
    import mla_speculative_decode_gb300 as va
    va.build()
    va.init(local)
    if args.case:
        run_case(va, args, dev)
        return
    hbm_peak, tc_peak, peak_kind = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    # ---- headline: the batched ragged step (8 requests, H=64, T=16)
    hs = synth.spec(HEADLINE)
    pool = device_pool(hs.num_slots, seed=1 + rank, dev=dev)
    step = Step(va, pool, hs.H, hs.T, list(hs.prefix), seed=4 + rank, nrot=2, dev=dev,
                path=args.path, nsplit=args.nsplit)
    kv_step = step.kv_bytes
    assert step.nrot * kv_step > 2 * l2, "rotated slot tables must exceed L2"
    graphs, _ = capture_graphs(step, args.steps)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t_wall0 = time.time()
    ms = time_steps(graphs, args.steps, args.warmup, dist)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    del graphs
    ms = max_over_ranks(ms, dist, dev)
    ms_step = ms / args.steps
    value = job_gbs(world, kv_step, args.steps, ms)
    k_us = partial_kernel_us(step)
    head = point_record(step, ms_step * 1e3, ms_step * 1e3, ms_step * 1e3, k_us, hbm_peak,
                        tc_peak)

    e2e = e2e_leg(va, step, args.steps, args.warmup, dist, dev)

    # ---- the target points: H=8 and H=64, T=16, prefixes 16k / 65k / 200k,
    # scattered and contiguous (kernel-level fractions of both roofs), and the
    # rest of the prefix sweep
    targets, sweep = [], []
    if not args.no_sweep and rank == 0:
        points = [(H_, P_, lay, True) for H_ in (8, 64) for P_ in TARGET_P
                  for lay in ("scattered", "contiguous")]
        points += [(H_, P_, "scattered", False) for H_ in (8, 64) for P_ in SWEEP_P]
        for H_, P_, lay, is_target in points:
            kvb = (P_ + 16) * synth.D_QK * 2
            nr = max(1, min(16, math.ceil(3 * l2 / kvb)))
            st = Step(va, pool, H_, 16, P_, seed=7, nrot=nr, dev=dev, path=args.path,
                      nsplit=0, layout=lay)
            reps = 8 * math.ceil(max(16, min(400, int(2e5 / (P_ / 1024 * H_ / 8)))) / 8)
            us, p10, p90, k_us_ = measure_dist(st, reps, 5)
            rec = {"H": H_, "T": 16, "P": P_, "layout": lay}
            rec.update(point_record(st, us, p10, p90, k_us_, hbm_peak, tc_peak))
            rec["bound"] = "hbm" if 2176 * 16 * H_ / 1152 < tc_peak * 1e12 / (hbm_peak * 1e9) \
                else "tensor"
            (targets if is_target else sweep).append(rec)
            del st
            torch.cuda.empty_cache()

    # ---- the other configurations of the step, and the widened rows
    configs = {}
    if not args.no_sweep and rank == 0:
        # TP8 slice: H=8, T=16, prefix 4096 (launch-bound)
        st = Step(va, pool, 8, 16, 4096, seed=1, nrot=max(2, math.ceil(3 * l2 / (4112 * 1152))),
                  dev=dev, path=args.path, nsplit=0)
        med, p10, p90, k_us_ = measure_dist(st, 64, 8)
        configs["tp8 slice H=8 T=16 P=4096 scattered"] = point_record(
            st, med, p10, p90, k_us_, hbm_peak, tc_peak)
        del st
        # long context: H=8, T=32 random tree, prefix 200000, 2^18-slot pool,
        # nsplit swept (two 128-row blocks per split)
        pool_l = device_pool(1 << 18, seed=3, dev=dev)
        rows = []
        for ns in (16, 32, 64, 96, 128, 0):
            st = Step(va, pool_l, 8, 32, 200000, seed=3, nrot=1, dev=dev, path=args.path,
                      nsplit=ns)
            med, p10, p90, k_us_ = measure_dist(st, 16, 3)
            r = {"auto": ns == 0}
            r.update(point_record(st, med, p10, p90, k_us_, hbm_peak, tc_peak))
            rows.append(r)
            del st
        configs["long H=8 T=32 P=200000 scattered (2^18 pool), nsplit sweep"] = rows
        del pool_l
        torch.cuda.empty_cache()
        # segmented call (two slot lists + dense extend mask) on the TP8 slice,
        # beside the paged call on the same slots
        seg = {}
        for lay in ("segmented", "segmented_append", "scattered"):
            st = Step(va, pool, 8, 16, 4096, seed=1, nrot=16, dev=dev, path=args.path, nsplit=0,
                      layout=lay)
            med, p10, p90, k_us_ = measure_dist(st, 64, 8)
            seg[lay] = {"us_per_step": med, "p10": p10, "p90": p90,
                        "gbs": st.kv_bytes / (med * 1e-6) / 1e9, "kernel_us": k_us_}
            del st
        configs["segmented TP8 H=8 T=16 P=4096 (kv_indices + out_cache_loc + dense mask; "
                "with the draft rows appended in the call) vs paged"] = seg
        torch.cuda.empty_cache()
        configs["tree acceptance B=8 T=16 V=129280 fp32 logits"] = bench_accept(va, dev,
                                                                                   hbm_peak)
        configs["tree build B=8 D=8 K=8 T=16 (draft tree + out_cache_loc on the device)"] = \
            bench_tree_build(va, dev)
        configs["defrag 65536 scattered rows -> contiguous"] = bench_defrag(va, pool, dev,
                                                                            hbm_peak)
        configs["contiguous decode step, batched H=64 T=16 (placement + contiguous verify + "
                "compaction; the same requests as the headline, kept contiguous)"] = \
            bench_contiguous_decode(va, dev, tc_peak)
        torch.cuda.empty_cache()

    cpu, parity = (None, None)
    if rank == 0 and not args.no_cpu:
        cpu, parity = cpu_baseline_leg(step)

    clk = clocks.summary(t_wall0, t_wall1) or clocks.summary()
    achieved = step.flops / (k_us * 1e-6) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q and KV, random trees, random slot scatter)",
        "config": dict(headline_config(),
                       nsplit=step.nsplit, path=["auto", "fma", "tc"][args.path],
                       l2=f"inputs larger than L2: {step.nrot} rotating slot tables "
                          f"({step.nrot * kv_step / 1e6:.0f} MB of rows vs {l2 / 1e6:.0f} MB L2)",
                       launch=f"CUDA graphs of {STEPS_PER_GRAPH} steps"
                              + (f" plus one graph of the remaining {args.steps % STEPS_PER_GRAPH}"
                                 if args.steps % STEPS_PER_GRAPH else "")
                              + ": exactly --steps steps timed; programmatic dependent launch "
                              "between the kernels of a step and between steps",
                       parallelism=f"replicas x{world}"),
        "headline": head,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak, "traffic": recorded_traffic(),
                     "kernel": "split-K partial (partial_tc_kernel)", "kernel_us": k_us,
                     "flops_per_launch": step.flops,
                     "peak_source": f"{peak_kind} bf16_tflops (burst)",
                     "hbm_frac_of_kernel": kv_step / (k_us * 1e-6) / 1e9 / hbm_peak},
        "target_points": targets,
        "cpu_baseline": cpu, "parity": parity, "e2e": e2e,
        "gpu_launches": (3 if args.path == 1 else 2) * args.steps, "clocks": clk,
        "sweep": sweep, "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
