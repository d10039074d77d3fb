"""Helpers for the GPU parity tests: move a synthetic workload to the device,
run the library through its binding, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# element-wise bar against the oracle on the same seeded inputs
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def to_device(w: synth.Workload, dev="cuda"):
    d = dict(q=w.q.to(dev), kv_pool=w.kv_pool.to(dev), slot_idx=w.slot_idx.to(dev),
             kv_indptr=w.kv_indptr.to(dev), prefix_len=w.prefix_len.to(dev),
             parents=w.parents.to(dev))
    if w.kv_start is not None:
        d["kv_start"] = w.kv_start.to(dev)
    return d


def run(va, d, w: synth.Workload, *, path=0, nsplit=0, layout=None, bits=None, workspace=None,
        out=None, lse=None):
    layout = layout or w.spec.layout
    kw = dict(sm_scale=w.spec.sm_scale, nsplit=nsplit, flags=path, workspace=workspace, out=out,
              lse=lse)
    par = None if bits is not None else d["parents"]
    if layout == "contiguous":
        return va.verify_attn_contiguous(d["q"], d["kv_pool"], d["kv_start"], d["prefix_len"],
                                         par, bits, **kw)
    return va.verify_attn_paged(d["q"], d["kv_pool"], d["slot_idx"], d["kv_indptr"],
                                d["prefix_len"], par, bits, **kw)


def reference(w: synth.Workload, rows=None, threads=None):
    bits, _ = oracle.tree_bits(w.parents.numpy())
    out, lse, _ = oracle.verify_attn(synth.as_u16(w.q), synth.as_u16(w.kv_pool),
                                     w.slot_idx.numpy(), w.kv_indptr.numpy(),
                                     w.prefix_len.numpy(), bits, w.spec.sm_scale, rows=rows,
                                     threads=threads)
    return out, lse


def compare(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, ref_out, ref_lse, rows=None):
    H = out_gpu.shape[1]
    o = out_gpu.float().reshape(-1, out_gpu.shape[-1]).cpu().numpy().astype(np.float64)
    l = lse_gpu.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    err = np.abs(o - ref_out)
    assert np.all(np.isfinite(o)), "non-finite output"
    with np.errstate(invalid="ignore"):     # -inf - -inf, handled just below
        lerr = np.abs(l - ref_lse)
    same_inf = (np.isinf(l) & np.isinf(ref_lse) & (np.sign(l) == np.sign(ref_lse)))
    lerr = np.where(same_inf, 0.0, lerr)
    stats = dict(max_abs=float(err.max()), mean_abs=float(err.mean()), lse_max=float(lerr.max()))
    assert stats["max_abs"] <= OUT_MAX_ABS, stats
    assert stats["mean_abs"] <= OUT_MEAN_ABS, stats
    assert stats["lse_max"] <= LSE_ABS, stats
    return stats


def sample_rows(w: synth.Workload, n: int, seed: int = 0):
    total = w.spec.B * w.spec.T * w.spec.H
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(total, size=min(n, total), replace=False).tolist())
    rows |= {0, total - 1}
    return np.array(sorted(rows), dtype=np.int64)
