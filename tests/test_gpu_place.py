"""Contiguous placement of the draft latents and compaction of the accepted
path (va_kv_append_contiguous, va_kv_compact_accepted) against the oracle,
byte for byte, and the decode-side chain that keeps each request contiguous
-- tree build, draft rows placed after the prefix, contiguous verify,
greedy acceptance, compaction -- captured in one CUDA graph and replayed
over several steps (needs an sm_103 GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_speculative_decode_gb300 as m
    m.build()
    m.init()
    return m


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("stride", [576, 640])
def test_append_and_compact_match_the_oracle(va, stride):
    g = torch.Generator().manual_seed(stride)
    rng = np.random.default_rng(stride)
    B, T, cap = 5, 8, 64
    rows = B * cap + 10
    pool = synth._bf16_normal((rows, stride), g)
    ks = np.array([3 + b * cap for b in range(B)], dtype=np.int64)
    # request 3: prefix and draft do not fit its reserve; the others keep
    # room for two rounds of compaction below
    pl = np.array([5, 20, 0, cap - T + 1, 10], dtype=np.int32)
    caps = np.full(B, cap, dtype=np.int32)
    draft = synth._bf16_normal((B * T, 576), g)
    d_pool = pool.cuda()
    d_ks, d_pl, d_cap = (torch.from_numpy(x).cuda() for x in (ks, pl, caps))
    loc = torch.full((B * T,), 7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    va.kv_append_contiguous(d_pool, d_ks, d_pl, d_cap, draft.cuda(), loc, status=status)
    torch.cuda.synchronize()
    p1, loc_w, bad = oracle.append_contiguous(synth.as_u16(pool), synth.as_u16(draft), ks, pl,
                                              caps, T)
    np.testing.assert_array_equal(_u16(d_pool), p1)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_w)
    assert bad == T and int(status.item()) == va.STATUS_BAD_DST

    # accepted paths: increasing, decreasing, empty, full chain, one bad node
    alen = np.array([3, 2, 0, 1, T], dtype=np.int32)
    nodes = np.full((B, T), -1, dtype=np.int32)
    nodes[0, :3] = [1, 4, 6]
    nodes[1, :2] = [5, 2]
    nodes[3, :1] = [0]                        # request 3 has no draft rows: left unchanged
    nodes[4, :] = np.arange(T)
    status.zero_()
    va.kv_compact_accepted(d_pool, d_ks, d_pl, d_cap, torch.from_numpy(alen).cuda(),
                           torch.from_numpy(nodes).cuda(), status=status)
    torch.cuda.synchronize()
    p2, pl_w, bad = oracle.compact_accepted(p1, ks, pl, caps, alen, nodes, T)
    np.testing.assert_array_equal(_u16(d_pool), p2)
    np.testing.assert_array_equal(d_pl.cpu().numpy(), pl_w)
    assert bad == 1 and int(status.item()) == va.STATUS_BAD_DST
    # a node outside the draft: that request alone is left unchanged
    nodes2 = nodes.copy()
    nodes2[0, 1] = T
    status.zero_()
    before = _u16(d_pool).copy()
    pl_before = d_pl.cpu().numpy().copy()
    va.kv_compact_accepted(d_pool, d_ks, d_pl, d_cap, torch.from_numpy(alen).cuda(),
                           torch.from_numpy(nodes2).cuda(), status=status)
    torch.cuda.synchronize()
    p3, pl3, bad = oracle.compact_accepted(before, ks, pl_before, caps, alen, nodes2, T)
    np.testing.assert_array_equal(_u16(d_pool), p3)
    np.testing.assert_array_equal(d_pl.cpu().numpy(), pl3)
    assert bad == 2 and int(status.item()) == va.STATUS_BAD_DST


def test_append_and_compact_64_node_trees(va):
    """T = 64 (the largest tree): the compaction stages up to 64 rows (72 KB,
    past the default 48 KB of dynamic shared memory) before writing any; long
    accepted paths in any order, against the oracle byte for byte."""
    g = torch.Generator().manual_seed(64)
    rng = np.random.default_rng(64)
    B, T, cap = 3, 64, 400
    pool = synth._bf16_normal((B * cap + 7, 576), g)
    ks = np.array([7 + b * cap for b in range(B)], dtype=np.int64)
    pl = np.array([100, 0, cap - T], dtype=np.int32)
    caps = np.full(B, cap, dtype=np.int32)
    draft = synth._bf16_normal((B * T, 576), g)
    d_pool = pool.cuda()
    d_ks, d_pl, d_cap = (torch.from_numpy(x).cuda() for x in (ks, pl, caps))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    loc = torch.full((B * T,), 7, dtype=torch.int32, device="cuda")
    va.kv_append_contiguous(d_pool, d_ks, d_pl, d_cap, draft.cuda(), loc, status=status)
    p1, loc_w, bad = oracle.append_contiguous(synth.as_u16(pool), synth.as_u16(draft), ks, pl,
                                              caps, T)
    torch.cuda.synchronize()
    assert bad == 0 and int(status.item()) == 0
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_w)
    np.testing.assert_array_equal(_u16(d_pool), p1)
    alen = np.array([64, 37, 5], dtype=np.int32)
    nodes = np.full((B, T), -1, dtype=np.int32)
    for b in range(B):
        nodes[b, :alen[b]] = rng.permutation(T)[:alen[b]]
    va.kv_compact_accepted(d_pool, d_ks, d_pl, d_cap, torch.from_numpy(alen).cuda(),
                           torch.from_numpy(nodes).cuda(), status=status)
    torch.cuda.synchronize()
    p2, pl_w, bad = oracle.compact_accepted(p1, ks, pl, caps, alen, nodes, T)
    assert bad == 0 and int(status.item()) == 0
    np.testing.assert_array_equal(_u16(d_pool), p2)
    np.testing.assert_array_equal(d_pl.cpu().numpy(), pl_w)


def _logits_for(rng, par, tok, V, follow=0.8):
    """Target logits whose greedy token at the prefix and at each node is, with
    probability `follow`, the token of one of that position's children."""
    B, T = par.shape
    root = rng.normal(size=(B, V)).astype(np.float32)
    lg = rng.normal(size=(B, T, V)).astype(np.float32)
    for b in range(B):
        for pos in range(-1, T):
            kids = [c for c in range(T) if par[b, c] == pos]
            row = root[b] if pos < 0 else lg[b, pos]
            t = int(tok[b, rng.choice(kids)]) if kids and rng.random() < follow \
                else int(rng.integers(0, V))
            row[t] = 10.0
    return root, lg


def test_contiguous_decode_chain_in_one_graph(va):
    """Tree build -> draft rows after the prefix -> contiguous verify ->
    acceptance -> compaction, captured once and replayed for three decode
    steps on new drafter output, queries, draft rows and target logits; the
    prefix lengths advance on the device.  Every step against the oracle
    chain: tree and acceptance exactly, the pool byte for byte, the verify
    output within the oracle bar."""
    rng = np.random.default_rng(99)
    g = torch.Generator().manual_seed(99)
    B, H, T, D, K, V = 3, 16, 16, 6, 4, 2048
    cap = 2048
    ks = np.array([b * cap for b in range(B)], dtype=np.int64)
    pl = np.array([500, 1200, 64], dtype=np.int32)
    caps = np.full(B, cap, dtype=np.int32)
    pool = synth._bf16_normal((B * cap, 576), g)

    def draw():
        tok = rng.integers(0, V, size=(B, D, K)).astype(np.int32)
        lp = np.log(rng.dirichlet(np.ones(K) * 0.7, size=(B, D))).astype(np.float32)
        q = synth._bf16_normal((B * T, H, 576), g)
        draft = synth._bf16_normal((B * T, 576), g)
        par_w, tok_w, _, _ = oracle.tree_build(tok, lp, T)
        root, lg = _logits_for(rng, par_w, tok_w, V)
        return tok, lp, q, draft, root, lg

    dev = "cuda"
    first = draw()
    d_tok = torch.from_numpy(first[0]).to(dev)
    d_lp = torch.from_numpy(first[1]).to(dev)
    d_q, d_draft = first[2].to(dev), first[3].to(dev)
    d_root, d_lg = torch.from_numpy(first[4]).to(dev), torch.from_numpy(first[5]).to(dev)
    d_pool = pool.to(dev)
    d_ks, d_pl, d_cap = (torch.from_numpy(x).to(dev) for x in (ks, pl, caps))
    par = torch.full((B, T), -1, dtype=torch.int32, device=dev)
    dtok = torch.zeros(B, T, dtype=torch.int32, device=dev)
    depth = torch.zeros(B, T, dtype=torch.int32, device=dev)
    loc = torch.zeros(B * T, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws, ns = va.alloc_workspace(B, T, H)
    out = torch.empty(B * T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B * T, H, dtype=torch.float32, device=dev)
    acc = (torch.empty(B, dtype=torch.int32, device=dev),
           torch.empty(B, T, dtype=torch.int32, device=dev),
           torch.empty(B, T, dtype=torch.int32, device=dev),
           torch.empty(B, dtype=torch.int32, device=dev))
    _, _, _, _, acc_ws = va.tree_accept(d_root, d_lg, dtok, par, loc.view(B, T))
    st = torch.cuda.Stream()

    def chain():
        va.tree_build(d_tok, d_lp, T, outputs=(par, dtok, depth, None), stream=st)
        va.kv_append_contiguous(d_pool, d_ks, d_pl, d_cap, d_draft, loc, status=status, stream=st)
        va.verify_attn_contiguous(d_q, d_pool, d_ks, d_pl, par, sm_scale=synth.SM_SCALE, nsplit=ns,
                                  workspace=ws, out=out, lse=lse, stream=st)
        va.tree_accept(d_root, d_lg, dtok, par, loc.view(B, T), workspace=acc_ws, outputs=acc,
                       stream=st)
        va.kv_compact_accepted(d_pool, d_ks, d_pl, d_cap, acc[0], acc[1], status=status, stream=st)

    st.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        chain()
    torch.cuda.synchronize()
    # capture ran nothing: the pool and the prefix lengths are as drawn
    np.testing.assert_array_equal(d_pl.cpu().numpy(), pl)

    pool_w = synth.as_u16(pool).copy()
    pl_w = pl.copy()
    for step in range(3):
        w = first if step == 0 else draw()
        tok, lp, q, draft, root, lg = w
        if step:
            d_tok.copy_(torch.from_numpy(tok))
            d_lp.copy_(torch.from_numpy(lp))
            d_q.copy_(q)
            d_draft.copy_(draft)
            d_root.copy_(torch.from_numpy(root))
            d_lg.copy_(torch.from_numpy(lg))
        out.fill_(float("nan"))
        status.zero_()
        graph.replay()
        torch.cuda.synchronize()
        # the oracle chain
        par_w, tok_w, _, _ = oracle.tree_build(tok, lp, T)
        np.testing.assert_array_equal(par.cpu().numpy(), par_w)
        np.testing.assert_array_equal(dtok.cpu().numpy(), tok_w)
        p1, loc_w, bad = oracle.append_contiguous(pool_w, synth.as_u16(draft), ks, pl_w, caps, T)
        assert bad == 0
        np.testing.assert_array_equal(loc.cpu().numpy(), loc_w)
        slots = np.concatenate([np.arange(ks[b], ks[b] + pl_w[b] + T) for b in range(B)])
        indptr = np.concatenate([[0], np.cumsum(pl_w + T)]).astype(np.int32)
        bits, nbad = oracle.tree_bits(par_w)
        assert nbad == 0
        ro, rl, _ = oracle.verify_attn(synth.as_u16(q), p1, slots.astype(np.int32), indptr, pl_w,
                                       bits, synth.SM_SCALE)
        _gpu.compare(out, lse, ro, rl)
        assert va.read_status(ws) == 0
        alen_w, nodes_w, _, _, _ = oracle.tree_accept(root, lg, tok_w, par_w, loc_w.reshape(B, T))
        np.testing.assert_array_equal(acc[0].cpu().numpy(), alen_w)
        np.testing.assert_array_equal(acc[1].cpu().numpy(), nodes_w)
        pool_w, pl_w, bad = oracle.compact_accepted(p1, ks, pl_w, caps, alen_w, nodes_w, T)
        assert bad == 0
        np.testing.assert_array_equal(_u16(d_pool), pool_w)
        np.testing.assert_array_equal(d_pl.cpu().numpy(), pl_w)
        assert int(status.item()) == 0
        assert alen_w.max() >= 2          # the walks went past the first level
    assert (pl_w > pl).all()              # every request's prefix grew
