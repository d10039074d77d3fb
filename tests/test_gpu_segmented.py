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

PATHS = {"fma": 1, "tc": 2, "tc1sm": 3}


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


# ------------------------------------------- draft rows appended in the call

def _append_case(va, spec, path, stride=576):
    spec.row_stride = stride
    w = synth.make(spec)
    ind, kip, loc = _split(w)
    mask = _flat_mask(w)
    g = torch.Generator().manual_seed(spec.seed + 1000)
    draft = torch.randn(spec.B * spec.T, synth.D_QK, generator=g).to(torch.bfloat16)
    # the draft slots hold NaN before the call: any read of them before the
    # append shows in the output
    w.kv_pool[torch.from_numpy(loc).long(), :synth.D_QK] = float("nan")
    pool0 = w.kv_pool.clone()
    kv_dev = w.kv_pool.cuda()
    ws, ns = va.alloc_workspace(spec.B, spec.T, spec.H, 0, path)
    out, lse = va.verify_attn_segmented(
        w.q.cuda(), kv_dev, torch.from_numpy(ind).cuda(), torch.from_numpy(kip).cuda(),
        torch.from_numpy(loc).cuda(), custom_mask=torch.from_numpy(mask).cuda(),
        draft_kv=draft.cuda(), sm_scale=w.spec.sm_scale, nsplit=ns, flags=path, workspace=ws)
    assert va.read_status(ws) == 0
    want_pool = oracle.append_rows(synth.as_u16(pool0), synth.as_u16(draft), loc)
    assert np.array_equal(synth.as_u16(kv_dev.cpu()), want_pool)
    slots, indptr, prefix = oracle.segmented_lists(ind, kip, loc, spec.T)
    bits, _ = oracle.dense_mask_bits(mask, kip, spec.T)
    ref_o, ref_l, _ = oracle.verify_attn(synth.as_u16(w.q), want_pool, slots, indptr, prefix, bits,
                                         w.spec.sm_scale)
    _gpu.compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("spec", [
    synth.Spec("app_tp8", B=1, H=8, T=16, prefix=[4096], num_slots=1 << 15, seed=71),
    synth.Spec("app_ragged", B=3, H=8, T=9, prefix=[0, 300, 77], num_slots=8192, seed=72),
    synth.Spec("app_long", B=1, H=8, T=16, prefix=[20000], num_slots=1 << 16, seed=73),
    # two-SM products: the draft keys are read by the QK pair and the PV pair
    synth.Spec("app_h64", B=2, H=64, T=16, prefix=[1500, 333], num_slots=1 << 14, seed=76),
], ids=["tp8", "ragged", "long", "h64"])
def test_segmented_append_then_verify(va, spec, path):
    _append_case(va, spec, path)


def test_segmented_append_wide_rows(va):
    """Pool rows wider than 576: only the first 576 columns are written."""
    _append_case(va, synth.Spec("app_wide", B=2, H=8, T=8, prefix=[500, 64], num_slots=4096,
                                seed=74), 0, stride=640)


def test_segmented_append_in_a_replayed_graph(va):
    """One captured call, replayed with new draft rows each time: every replay
    verifies against the rows it was given."""
    spec = synth.Spec("app_graph", B=1, H=8, T=16, prefix=[2048], num_slots=1 << 14, seed=75)
    w = synth.make(spec)
    ind, kip, loc = _split(w)
    mask = _flat_mask(w)
    dev = "cuda"
    q, kv = w.q.to(dev), w.kv_pool.to(dev)
    ind_d, kip_d, loc_d = (torch.from_numpy(x).to(dev) for x in (ind, kip, loc))
    mask_d = torch.from_numpy(mask).to(dev)
    draft = torch.zeros(spec.T, synth.D_QK, dtype=torch.bfloat16, device=dev)
    ws, ns = va.alloc_workspace(spec.B, spec.T, spec.H, 0)
    out = torch.empty(spec.T, spec.H, synth.D_V, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(spec.T, spec.H, dtype=torch.float32, device=dev)

    def call(stream=None):
        va.verify_attn_segmented(q, kv, ind_d, kip_d, loc_d, custom_mask=mask_d, draft_kv=draft,
                                 sm_scale=w.spec.sm_scale, nsplit=ns, workspace=ws, out=out,
                                 lse=lse, stream=stream)

    call()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(stream=s)
    slots, indptr, prefix = oracle.segmented_lists(ind, kip, loc, spec.T)
    bits, _ = oracle.dense_mask_bits(mask, kip, spec.T)
    for k in range(3):
        gen = torch.Generator().manual_seed(500 + k)
        rows = torch.randn(spec.T, synth.D_QK, generator=gen).to(torch.bfloat16)
        draft.copy_(rows)
        g.replay()
        torch.cuda.synchronize()
        pool_k = oracle.append_rows(synth.as_u16(w.kv_pool), synth.as_u16(rows), loc)
        ref_o, ref_l, _ = oracle.verify_attn(synth.as_u16(w.q), pool_k, slots, indptr, prefix,
                                             bits, w.spec.sm_scale)
        _gpu.compare(out, lse, ref_o, ref_l)
