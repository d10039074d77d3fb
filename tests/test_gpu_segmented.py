"""Segmented verify calls on the GPU (two slot lists, dense extend mask) against
the fp64 oracle and against the paged call on the concatenated list.

The Checkpoint Report, "Mistakes and Incorrect Assumptions": the extend call
takes the prefix slots in kv_indices, the draft tokens' own slots at
out_cache_loc, and a custom mask with one row per draft token of stride
prefix + q_len.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _gpu
from tests.test_oracle_pins import _dense_mask

pytestmark = pytest.mark.gpu

PATHS = {"fma": 1, "tc": 2}


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_speculative_decode_gb300 as m
    m.build()
    m.init()
    return m


def _split(w):
    """The workload's per-request lists as (kv_indices, kv_indptr, out_cache_loc)."""
    sl, ip, P, T = w.slot_idx.numpy(), w.kv_indptr.numpy(), w.prefix_len.numpy(), w.spec.T
    B = w.spec.B
    ind = np.concatenate([sl[ip[b]:ip[b] + P[b]] for b in range(B)]).astype(np.int32)
    kip = np.concatenate([[0], np.cumsum(P)]).astype(np.int32)
    loc = np.concatenate([sl[ip[b] + P[b]:ip[b] + P[b] + T] for b in range(B)]).astype(np.int32)
    return ind, kip, loc


def _flat_mask(w, vis=None):
    """Dense extend mask of every request (prefix columns 1, draft columns from
    the tree's closure, or from `vis` [B, T, T] when given), concatenated."""
    P = w.prefix_len.numpy()
    rows = []
    for b in range(w.spec.B):
        m = _dense_mask(w.parents[b].numpy(), int(P[b]))
        if vis is not None:
            m[:, P[b]:] = vis[b]
        rows.append(m.reshape(-1))
    return np.concatenate(rows).astype(np.uint8)


def _reference(w, ind, kip, loc, mask):
    slots, indptr, prefix = oracle.segmented_lists(ind, kip, loc, w.spec.T)
    bits, missing = oracle.dense_mask_bits(mask, kip, w.spec.T)
    out, lse, _ = oracle.verify_attn(synth.as_u16(w.q), synth.as_u16(w.kv_pool), slots, indptr,
                                     prefix, bits, w.spec.sm_scale)
    return out, lse, missing


def _call(va, w, ind, kip, loc, mask=None, parents=None, path=0, ws=None, ns=0, mask_len=None):
    dev = "cuda"
    m = None
    if mask is not None:
        m = torch.from_numpy(mask).to(dev)
        if mask_len is not None:
            m = m[:mask_len]
    return va.verify_attn_segmented(
        w.q.to(dev), w.kv_pool.to(dev), torch.from_numpy(ind).to(dev),
        torch.from_numpy(kip).to(dev), torch.from_numpy(loc).to(dev), custom_mask=m,
        tree_parent=None if parents is None else parents.to(dev), sm_scale=w.spec.sm_scale,
        nsplit=ns, flags=path, workspace=ws)


SPECS = [
    synth.Spec("seg_one", B=1, H=8, T=4, prefix=[256], num_slots=4096, tree="chain", seed=61),
    synth.Spec("seg_ragged", B=3, H=8, T=9, prefix=[0, 300, 77], num_slots=8192, seed=62),
    synth.Spec("seg_tp8", B=1, H=8, T=16, prefix=[4096], num_slots=1 << 16, seed=63),
    synth.Spec("seg_h32", B=2, H=32, T=8, prefix=[1000, 2500], num_slots=1 << 14, seed=64),
]


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("spec", SPECS, ids=[s.name for s in SPECS])
def test_segmented_dense_mask_matches_oracle_and_paged(va, spec, path):
    w = synth.make(spec)
    ind, kip, loc = _split(w)
    mask = _flat_mask(w)
    ws, ns = va.alloc_workspace(spec.B, spec.T, spec.H, 0, path)
    out, lse = _call(va, w, ind, kip, loc, mask=mask, path=path, ws=ws, ns=ns)
    assert va.read_status(ws) == 0
    ref_o, ref_l, missing = _reference(w, ind, kip, loc, mask)
    assert missing == 0
    _gpu.compare(out, lse, ref_o, ref_l)
    # the same kernels on the concatenated list: the same bits
    d = _gpu.to_device(w)
    ws2, _ = va.alloc_workspace(spec.B, spec.T, spec.H, ns, path)
    out2, lse2 = _gpu.run(va, d, w, path=path, nsplit=ns, workspace=ws2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # and the tree given as parents instead of the mask
    out3, lse3 = _call(va, w, ind, kip, loc, parents=w.parents, path=path, ws=ws, ns=ns)
    assert torch.equal(out, out3) and torch.equal(lse, lse3)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_segmented_arbitrary_visibility(va, path):
    """Draft columns that are no tree's closure (self hidden, later nodes seen)
    are taken as given."""
    spec = synth.Spec("seg_vis", B=2, H=8, T=12, prefix=[200, 0], num_slots=4096, seed=65)
    w = synth.make(spec)
    rng = np.random.default_rng(7)
    vis = rng.random((spec.B, spec.T, spec.T)) < 0.4
    vis[1, 3, :] = False               # a node of the prefix-free request sees no key
    ind, kip, loc = _split(w)
    mask = _flat_mask(w, vis)
    ws, ns = va.alloc_workspace(spec.B, spec.T, spec.H, 0, path)
    out, lse = _call(va, w, ind, kip, loc, mask=mask, path=path, ws=ws, ns=ns)
    assert va.read_status(ws) == 0
    ref_o, ref_l, _ = _reference(w, ind, kip, loc, mask)
    _gpu.compare(out, lse, ref_o, ref_l)
    r = (1 * spec.T + 3) * spec.H
    assert torch.isinf(lse.reshape(-1)[r:r + spec.H]).all()


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_segmented_bad_draft_slot_flagged(va, path):
    spec = synth.Spec("seg_bad", B=2, H=8, T=8, prefix=[150, 40], num_slots=4096, seed=66)
    w = synth.make(spec)
    ind, kip, loc = _split(w)
    loc[spec.T + 2] = 4096 + 9          # request 1, draft node 2
    mask = _flat_mask(w)
    ws, ns = va.alloc_workspace(spec.B, spec.T, spec.H, 0, path)
    out, lse = _call(va, w, ind, kip, loc, mask=mask, path=path, ws=ws, ns=ns)
    assert va.read_status(ws) == va.STATUS_BAD_SLOT
    ref_o, ref_l, _ = _reference(w, ind, kip, loc, mask)    # the oracle skips that key
    _gpu.compare(out, lse, ref_o, ref_l)


def test_segmented_short_mask_flagged(va):
    spec = synth.Spec("seg_short", B=2, H=4, T=6, prefix=[30, 20], num_slots=2048, seed=67)
    w = synth.make(spec)
    ind, kip, loc = _split(w)
    mask = _flat_mask(w)
    cut = mask.shape[0] - 4             # the last row of request 1 loses 4 draft columns
    ws, ns = va.alloc_workspace(spec.B, spec.T, spec.H, 0)
    out, lse = _call(va, w, ind, kip, loc, mask=mask, ws=ws, ns=ns, mask_len=cut)
    assert va.read_status(ws) == va.STATUS_BAD_MASK
    ref_o, ref_l, missing = _reference(w, ind, kip, loc, mask[:cut])
    assert missing == 4
    _gpu.compare(out, lse, ref_o, ref_l)


def test_segmented_status_clears_between_calls(va):
    spec = synth.Spec("seg_clear", B=1, H=8, T=4, prefix=[64], num_slots=1024, seed=68)
    w = synth.make(spec)
    ind, kip, loc = _split(w)
    mask = _flat_mask(w)
    ws, ns = va.alloc_workspace(spec.B, spec.T, spec.H, 0)
    _call(va, w, ind, kip, loc, mask=mask, ws=ws, ns=ns, mask_len=mask.shape[0] - 1)
    assert va.read_status(ws) == va.STATUS_BAD_MASK
    _call(va, w, ind, kip, loc, mask=mask, ws=ws, ns=ns)
    assert va.read_status(ws) == 0
