#!/usr/bin/env python3
"""Benchmark of one MLA tree-verify attention step on GB300.

Default workload: one request, H=8 heads, T=16 random draft-tree nodes,
prefix 4096 keys, bf16 latent KV gathered through a page_size=1 slot table
scattered over a 2^20-slot pool (the TP8 slice).  A step is one verify call:
tree-mask evaluation, split-K partial attention and the LSE merge.

Prints ONE JSON line: effective KV GB/s (whole job), us/step, the split-K
kernel's roofline fraction, the oracle timed on the host cores, an
end-to-end figure through the C ABI with host buffers, clocks and launches.

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
WORKLOAD = ("TP8 slice: 1 request, H=8, T=16 random tree, prefix 4096, bf16 latent KV "
            "(576 = 512 + 64), page_size=1 slots scattered over a 2^20-slot pool, "
            "sm_scale=1/sqrt(192)")
SWEEP_P = [4096, 16384, 32768, 65536, 131072, 200000]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 FMA, 2 tensor cores")
    ap.add_argument("--nsplit", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--case", default="",
                    help="H,prefix,layout: run only --warmup + --steps plain calls of that "
                         "workload (the small captures the ncu summaries are made from); "
                         "prints a timing note, not the benchmark line")
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
    """A few plain verify calls of one workload, for profiler captures."""
    H, P, layout = args.case.split(",")
    H, P = int(H), int(P)
    rows = 1 << 18
    while rows < 2 * (P + 16):
        rows *= 2
    pool = device_pool(rows, seed=1, dev=dev)
    st = Step(va, pool, H, 16, P, seed=7, nrot=2, dev=dev, path=args.path, nsplit=args.nsplit,
              layout=layout)
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
    print(f"case H={H} P={P} {layout} nsplit={st.nsplit}: {us:.2f} us/call "
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
        self.kv_bytes = self.N * synth.D_QK * 2
        # tensor-core work: 2176 flop (2*576 + 2*512) for every row and every key
        self.flops = sum(2176.0 * T * H * n for n in Ns)

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


STEPS_PER_GRAPH = 8


def capture_graphs(step: Step, with_events: bool, per_graph: int = 1):
    """CUDA graphs over the rotated slot tables, `per_graph` consecutive steps
    (each on its own table) per graph; with events, one step per graph and
    event records around its split-K kernel."""
    va = step.va
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for k in range(min(step.nrot, 3)):
            step.call(k)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graphs, evs = [], []
    per_graph = 1 if with_events else max(1, per_graph)
    ngraphs = max(1, step.nrot // per_graph)
    for gi in range(ngraphs):
        g = torch.cuda.CUDAGraph()
        if with_events:
            eb = torch.cuda.Event(enable_timing=True)
            ea = torch.cuda.Event(enable_timing=True)
            va.set_partial_events(eb, ea)
            evs.append((eb, ea))
        with torch.cuda.graph(g):
            for j in range(per_graph):
                step.call(gi * per_graph + j)
        graphs.append(g)
    va.set_partial_events(None, None)
    return graphs, evs


def time_graphs(graphs, K, W, dist=None, per_graph: int = 1):
    """Times exactly K steps: K / per_graph replays (K a multiple of per_graph)."""
    assert K % per_graph == 0 and W >= 1
    for k in range(max(1, -(-W // per_graph))):
        graphs[k % len(graphs)].replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(K // per_graph):
        graphs[k % len(graphs)].replay()
    e1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def kernel_ms(evs, used):
    """Average split-K kernel duration over the last replay of each graph used."""
    n = min(len(evs), used)
    return float(np.mean([evs[i][0].elapsed_time(evs[i][1]) for i in range(n)]))


def measure_dist(step: Step, K: int, W: int, runs: int = 5):
    """Per-step µs of `runs` timed runs of K steps each: (median, p10, p90), and
    the split-K kernel µs."""
    per = STEPS_PER_GRAPH if K % STEPS_PER_GRAPH == 0 and step.nrot >= STEPS_PER_GRAPH else 1
    graphs, _ = capture_graphs(step, with_events=False, per_graph=per)
    egraphs, evs = capture_graphs(step, with_events=True)
    vals = [time_graphs(graphs, K, W if i == 0 else 1, None, per_graph=per) / K * 1e3
            for i in range(runs)]
    for g in egraphs:
        g.replay()
    for g in egraphs:
        g.replay()
    torch.cuda.synchronize()
    k_us = kernel_ms(evs, len(egraphs)) * 1e3
    del graphs, egraphs
    v = np.array(vals)
    return float(np.median(v)), float(np.percentile(v, 10)), float(np.percentile(v, 90)), k_us


def measure(step: Step, K: int, W: int, dist=None):
    """(ms for K steps, ms of the split-K kernel).  The step time comes from
    graphs with nothing but the steps' kernels -- eight consecutive steps, each
    on its own rotated slot table, per graph, as a serving loop would capture
    them, so that host-side graph submission does not pace the device -- and
    each kernel may start while its predecessor finishes (programmatic
    dependent launch); the kernel time from a second set of one-step graphs
    with event records around the split-K kernel, replayed after the timed
    region."""
    per = STEPS_PER_GRAPH if K % STEPS_PER_GRAPH == 0 and step.nrot >= STEPS_PER_GRAPH else 1
    graphs, _ = capture_graphs(step, with_events=False, per_graph=per)
    egraphs, evs = capture_graphs(step, with_events=True)
    ms = time_graphs(graphs, K, W, dist, per_graph=per)
    for g in egraphs:
        g.replay()
    for g in egraphs:
        g.replay()
    torch.cuda.synchronize()
    k_ms = kernel_ms(evs, len(egraphs))
    del graphs, egraphs
    return ms, k_ms


def check_parity(step: Step, k: int, nrows: int = 8):
    """Sampled rows of step k against the fp64 oracle (compact copy of the rows used)."""
    import oracle
    step.call(k)
    torch.cuda.synchronize()
    table = step.tables[k % step.nrot].long()
    rows_kv = step.pool[table].cpu()
    rng = np.random.default_rng(k)
    rows = np.sort(rng.choice(step.T * step.H, size=min(nrows, step.T * step.H), replace=False))
    bits, _ = oracle.tree_bits(step.parents.cpu().numpy())
    ro, rl, _ = oracle.verify_attn(synth.as_u16(step.q.cpu()), synth.as_u16(rows_kv),
                                   np.arange(step.N, dtype=np.int32), np.array([0, step.N]),
                                   np.array([step.P]), bits, synth.SM_SCALE, rows=rows)
    go = step.out.float().reshape(-1, 512).cpu().numpy()[rows]
    gl = step.lse.reshape(-1).cpu().numpy()[rows]
    err = float(np.abs(go - ro).max())
    mean = float(np.abs(go - ro).mean())
    lerr = float(np.abs(gl - rl).max())
    return {"rows": int(len(rows)), "max_abs": err, "mean_abs": mean, "lse_max_abs": lerr,
            "ok": bool(err <= 2e-2 and mean <= 2e-3 and lerr <= 1e-3)}


# --------------------------------------------------------------- oracle

def cpu_oracle(P, H, T, seed, budget_s=12.0, threads=None):
    """The fp64 oracle on whole steps of the same workload until ~budget_s."""
    import oracle
    threads = threads or oracle.default_threads()
    g = torch.Generator().manual_seed(seed)
    N = P + T
    q = synth.as_u16(torch.randn(T, H, synth.D_QK, generator=g).to(torch.bfloat16))
    kv = synth.as_u16(torch.randn(N, synth.D_QK, generator=g).to(torch.bfloat16))
    parents = synth.make_parents(T, "random", g).view(1, T).numpy()
    bits, _ = oracle.tree_bits(parents)
    slots = np.random.default_rng(seed).permutation(N).astype(np.int32)
    t0 = time.perf_counter()
    steps = 0
    while True:
        oracle.verify_attn(q, kv, slots, np.array([0, N]), np.array([P]), bits, synth.SM_SCALE,
                           threads=threads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or steps >= 1000:
            break
    per = el / steps
    return {"value": N * synth.D_QK * 2 / per / 1e9, "unit": "GB/s", "cores": int(threads),
            "kind": "oracle", "us_per_step": per * 1e6,
            "sample": f"{steps} whole step(s) of the same shape (P={P}, H={H}, T={T}), "
                      f"fp64, {el:.1f} s"}


def reference_arm(args, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    P, H, T = 4096, 8, 16
    g = torch.Generator().manual_seed(1)
    N = P + T
    q = synth.as_u16(torch.randn(T, H, synth.D_QK, generator=g).to(torch.bfloat16))
    kv = synth.as_u16(torch.randn(N, synth.D_QK, generator=g).to(torch.bfloat16))
    parents = synth.make_parents(T, "random", g).view(1, T).numpy()
    slots = np.random.default_rng(1).permutation(N).astype(np.int32)

    def one():
        bits, _ = oracle.tree_bits(parents)
        oracle.verify_attn(q, kv, slots, np.array([0, N]), np.array([P]), bits, synth.SM_SCALE,
                           threads=threads)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    val = N * synth.D_QK * 2 / (ms / 1e3) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD + " (each step: the whole step on the host cores)"},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{args.steps} whole steps"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main

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

    # ---- headline workload
    H, T, P = 8, 16, 4096
    pool = device_pool(1 << 20, seed=1 + rank, dev=dev)
    kv_step = (P + T) * synth.D_QK * 2
    nrot = max(2, math.ceil(3 * l2 / kv_step))
    step = Step(va, pool, H, T, P, seed=1 + rank, nrot=nrot, dev=dev, path=args.path,
                nsplit=args.nsplit)
    parity = check_parity(step, 0)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t_wall0 = time.time()
    ms, k_ms = measure(step, args.steps, args.warmup, dist)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    ms = max_over_ranks(ms, dist, dev)
    ms_step = ms / args.steps
    value = job_gbs(world, kv_step, args.steps, ms)

    # ---- end to end through the public API with host buffers.  A step's
    # inputs (q, its slot table, indptr, prefix lengths, parents) are packed
    # in one pinned host buffer and land with one host-to-device copy in a
    # device buffer whose views the call takes; out and lse are views of one
    # device result buffer read back with one device-to-host copy.
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
    h2d = in_bytes
    d2h = res_bytes
    Ke = min(args.steps, 500)

    dbuf = torch.empty(in_bytes, dtype=torch.uint8, device=dev)

    def dview(name, like):
        off, n = offs[name]
        return dbuf[off:off + n].view(like.dtype).view(like.shape)

    dres = torch.empty(res_bytes, dtype=torch.uint8, device=dev)
    dout = dres[:o_bytes].view(step.out.dtype).view(step.out.shape)
    dlse = dres[l_off:res_bytes].view(step.lse.dtype).view(step.lse.shape)
    hres = torch.empty(res_bytes, dtype=torch.uint8).pin_memory()
    # The verify call prepared once (checks and marshalling) on stream s; each
    # step copies its packed inputs in, launches it and reads out and lse back.
    # Steps are captured eight to a CUDA graph (the copies are graph nodes, each
    # step's from its own pinned buffer), as a serving loop would replay them,
    # so that Python does not pace the device.
    s_e2e = torch.cuda.Stream()
    s_e2e.wait_stream(torch.cuda.current_stream())
    call = va.prepare_paged(dview("q", step.q), step.pool, dview("tab", step.tables[0]),
                            dview("ind", step.indptr), dview("pre", step.prefix),
                            dview("par", step.parents), sm_scale=synth.SM_SCALE,
                            nsplit=step.nsplit, flags=step.path, workspace=step.ws, out=dout,
                            lse=dlse, stream=s_e2e)

    def e2e_step(k):
        dbuf.copy_(hins[k % len(hins)], non_blocking=True)
        call()
        hres.copy_(dres, non_blocking=True)

    with torch.cuda.stream(s_e2e):
        for k in range(min(args.warmup, 20)):
            e2e_step(k)
        # the packed copy path computes the same step: check one result
        e2e_step(0)
    torch.cuda.synchronize()
    step.call(0)
    torch.cuda.synchronize()
    assert torch.equal(dout, step.out) and torch.equal(dlse, step.lse), "e2e path differs"
    assert torch.equal(hres, dres.cpu()), "e2e read-back differs"
    per = STEPS_PER_GRAPH
    e_graphs = []
    for gi in range(max(1, min(8, len(hins) // per))):
        g_e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e, stream=s_e2e):
            for j2 in range(per):
                e2e_step(gi * per + j2)
        e_graphs.append(g_e)
    Ke = (Ke // per) * per
    with torch.cuda.stream(s_e2e):
        for g_e in e_graphs:
            g_e.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s_e2e):
        a.record()
        for r in range(Ke // per):
            e_graphs[r % len(e_graphs)].replay()
        b.record()
    torch.cuda.synchronize()
    e_ms = max_over_ranks(a.elapsed_time(b) / Ke, dist, dev)
    e2e = {"value": job_gbs(world, kv_step, 1, e_ms), "unit": "GB/s",
           "us_per_step": e_ms * 1e3, "steps": Ke, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h),
           "note": "every step: its inputs packed in one pinned buffer and copied in "
                   "(one H2D copy), the verify call (prepared once with va.prepare_paged) "
                   "launched, out and lse read back (one D2H copy); steps captured eight "
                   "to a CUDA graph and replayed"}

    # ---- prefix sweeps (H=8 and H=64, T=16), scattered slots
    sweep = []
    if not args.no_sweep and rank == 0:
        points = [(Hs, Ps, "scattered") for Hs in (8, 64) for Ps in SWEEP_P]
        points += [(Hs, Ps, "contiguous") for Hs in (8, 64) for Ps in (16384, 65536, 200000)]
        for Hs, Ps, lay in points:
            if True:
                kvb = (Ps + 16) * synth.D_QK * 2
                nr = max(1, min(16, math.ceil(3 * l2 / kvb)))
                st = Step(va, pool, Hs, 16, Ps, seed=7, nrot=nr, dev=dev, path=args.path,
                          nsplit=0, layout=lay)
                reps = 8 * math.ceil(max(20, min(400, int(2e5 / (Ps / 1024 * Hs / 8)))) / 8)
                us, p10, p90, k_us = measure_dist(st, reps, 5)
                sweep.append({"H": Hs, "T": 16, "P": Ps, "layout": lay, "us_per_step": us,
                              "p10": p10, "p90": p90,
                              "gbs": kvb / (us * 1e-6) / 1e9,
                              "frac_hbm": kvb / (us * 1e-6) / 1e9 / hbm_peak,
                              "tflops": st.flops / (us * 1e-6) / 1e12,
                              "partial_kernel_us": k_us,
                              "partial_gbs": kvb / (k_us * 1e-6) / 1e9, "nsplit": st.nsplit,
                              "path": "auto" if args.path == 0 else str(args.path)})
                del st
                torch.cuda.empty_cache()

    # ---- the remaining configurations of the step, and the defrag compaction
    configs = {}
    if not args.no_sweep and rank == 0:
        # long context: H=8, T=32 random tree, prefix 200000, 2^18-slot pool,
        # nsplit swept (two 128-row blocks per split)
        pool_l = device_pool(1 << 18, seed=3, dev=dev)
        rows = []
        for ns in (16, 32, 64, 96, 128, 0):
            st = Step(va, pool_l, 8, 32, 200000, seed=3, nrot=1, dev=dev, path=args.path, nsplit=ns)
            med, p10, p90, k_us = measure_dist(st, 16, 3)
            rows.append({"nsplit": st.nsplit, "auto": ns == 0, "us_per_step": med, "p10": p10,
                         "p90": p90, "gbs": st.kv_bytes / (med * 1e-6) / 1e9,
                         "tflops": st.flops / (med * 1e-6) / 1e12, "partial_kernel_us": k_us})
            del st
        configs["long H=8 T=32 P=200000 scattered (2^18 pool)"] = rows
        del pool_l
        torch.cuda.empty_cache()
        # batched ragged: 8 requests, prefixes U[1024, 65536], H=64, T=16
        prefs = synth.spec("batched").prefix
        st = Step(va, pool, 64, 16, prefs, seed=4, nrot=2, dev=dev, path=args.path, nsplit=0)
        med, p10, p90, k_us = measure_dist(st, 8, 3)
        configs["batched B=8 H=64 T=16 ragged, one graph per step"] = {
            "prefixes": prefs, "nsplit": st.nsplit, "us_per_step": med, "p10": p10, "p90": p90,
            "gbs": st.kv_bytes / (med * 1e-6) / 1e9, "tflops": st.flops / (med * 1e-6) / 1e12,
            "partial_kernel_us": k_us, "kv_bytes": st.kv_bytes}
        del st
        torch.cuda.empty_cache()
        # segmented call (two slot lists + dense extend mask) on the TP8 slice,
        # beside the paged call on the same slots
        seg = {}
        for lay in ("segmented", "segmented_append", "scattered"):
            st = Step(va, pool, 8, 16, 4096, seed=1, nrot=16, dev=dev, path=args.path, nsplit=0,
                      layout=lay)
            med, p10, p90, k_us = measure_dist(st, 64, 8)
            seg[lay] = {"us_per_step": med, "p10": p10, "p90": p90,
                        "gbs": st.kv_bytes / (med * 1e-6) / 1e9, "partial_kernel_us": k_us}
            del st
        configs["segmented TP8 H=8 T=16 P=4096 (kv_indices + out_cache_loc + dense mask; "
                "with the draft rows appended in the call) vs paged"] = seg
        torch.cuda.empty_cache()
        # greedy tree acceptance after verify: B=8 requests, T=16 nodes, a
        # 129280-token vocabulary, fp32 logits (one row after the prefix and
        # one per node); rotated logits buffers larger than L2 together
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
        # graphs of 8 calls, each on its own logits buffer, as for the verify step
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
        configs["tree acceptance B=8 T=16 V=129280 fp32 logits"] = {
            "us": a_us, "logits_bytes": a_bytes, "gbs": a_bytes / (a_us * 1e-6) / 1e9,
            "frac_hbm": a_bytes / (a_us * 1e-6) / 1e9 / hbm_peak,
            "timing": "CUDA graphs of 8 calls on rotated logits buffers (> L2 together), events"}
        del bufs
        torch.cuda.empty_cache()
        # defrag: 65536 scattered rows (lower half of the pool) compacted into a
        # contiguous range in the upper half
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
        configs["defrag 65536 scattered rows -> contiguous"] = {
            "us": d_us, "bytes_moved": moved, "gbs": moved / (d_us * 1e-6) / 1e9,
            "frac_hbm": moved / (d_us * 1e-6) / 1e9 / hbm_peak}

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_oracle(P, H, T, seed=1)

    clk = clocks.summary(t_wall0, t_wall1) or clocks.summary()
    achieved = kv_step / (k_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q and KV, random trees, random slot scatter)",
        "config": {"workload": WORKLOAD, "B": 1, "H": H, "T": T, "prefix": P,
                   "kv_bytes_per_step": kv_step, "nsplit": step.nsplit,
                   "path": ["auto", "fma", "tc"][args.path],
                   "l2": f"inputs larger than L2: {step.nrot} rotating slot tables "
                         f"({step.nrot * kv_step / 1e6:.0f} MB of rows vs {l2 / 1e6:.0f} MB L2)",
                   "launch": f"CUDA graphs of {STEPS_PER_GRAPH} steps, programmatic dependent "
                             "launch between the kernels of a step",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": recorded_traffic(),
                     "kernel": "split-K partial", "kernel_us": k_ms * 1e3,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": (3 if args.path == 1 else 2) * args.steps, "clocks": clk,
        "parity": parity, "sweep": sweep, "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
