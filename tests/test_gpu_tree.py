"""Device-side draft tree and slot building (va_tree_build) against the oracle,
bit for bit, and the whole decode-side chain -- tree build, segmented verify
with the draft rows appended, greedy acceptance -- captured in one CUDA graph
and replayed on new drafter output (needs an sm_103 GPU)."""
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


def _candidates(rng, B, D, K, kind):
    tok = rng.integers(0, 32000, size=(B, D, K)).astype(np.int32)
    if kind == "dirichlet":
        lp = np.log(rng.dirichlet(np.ones(K) * 0.7, size=(B, D))).astype(np.float32)
    elif kind == "ties":                         # few levels: many equal scores
        lp = -rng.integers(0, 3, size=(B, D, K)).astype(np.float32) * 0.5
    elif kind == "specials":                     # NaN, -inf, +inf, positive values
        lp = rng.normal(-1.0, 1.0, size=(B, D, K)).astype(np.float32)
        flat = lp.reshape(-1)
        idx = rng.permutation(flat.size)
        flat[idx[:3]] = np.nan
        flat[idx[3:6]] = -np.inf
        flat[idx[6:8]] = np.inf
    else:
        raise ValueError(kind)
    return tok, lp


@pytest.mark.parametrize("B,D,K,T,kind", [
    (5, 6, 5, 16, "dirichlet"),
    (3, 4, 3, 40, "ties"),
    (9, 8, 8, 64, "dirichlet"),     # more requests than warps of the CTA
    (2, 15, 16, 64, "specials"),
    (4, 3, 2, 14, "ties"),          # T = every node of the candidate tree
    (3, 8, 1, 8, "dirichlet"),      # one candidate per depth: a chain
    (1, 1, 16, 16, "specials"),     # one depth: the candidates in order
    (2, 5, 4, 1, "dirichlet"),
    (200, 8, 8, 16, "dirichlet"),   # many requests: 25 rounds of the CTA's warps
])
def test_tree_build_matches_oracle(va, B, D, K, T, kind):
    rng = np.random.default_rng(B * 1000 + D * 10 + K)
    tok, lp = _candidates(rng, B, D, K, kind)
    free = rng.permutation(100000)[:3 * B * T + 5].astype(np.int32)
    head0 = 5
    d_tok, d_lp = torch.from_numpy(tok).cuda(), torch.from_numpy(lp).cuda()
    d_free = torch.from_numpy(free).cuda()
    d_head = torch.tensor([head0], dtype=torch.int32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    par_w, tok_w, dep_w, _ = oracle.tree_build(tok, lp, T)
    head = head0
    for _ in range(2):                 # the head moves on: new slots each call
        par, tk, dep, loc = va.tree_build(d_tok, d_lp, T, d_free, d_head, status=status)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(par.cpu().numpy(), par_w)
        np.testing.assert_array_equal(tk.cpu().numpy(), tok_w)
        np.testing.assert_array_equal(dep.cpu().numpy(), dep_w)
        loc_w, head = oracle.pop_slots(free, head, B, T)
        np.testing.assert_array_equal(loc.cpu().numpy(), loc_w)
        assert int(d_head.item()) == head
        assert int(status.item()) == 0
    # every node's parent precedes it and sits one level up
    p = par.cpu().numpy()
    dp = dep.cpu().numpy()
    for b in range(B):
        for i in range(T):
            assert p[b, i] < i
            assert dp[b, i] == (0 if p[b, i] < 0 else dp[b, p[b, i]] + 1)


def test_tree_build_free_list_running_out(va):
    rng = np.random.default_rng(7)
    B, D, K, T = 3, 4, 4, 10
    tok, lp = _candidates(rng, B, D, K, "dirichlet")
    free = np.arange(1000, 1025, dtype=np.int32)          # 25 slots for 30 nodes
    d_head = torch.tensor([0], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    par, tk, dep, loc = va.tree_build(torch.from_numpy(tok).cuda(), torch.from_numpy(lp).cuda(),
                                      T, torch.from_numpy(free).cuda(), d_head, status=status)
    torch.cuda.synchronize()
    loc_w, head = oracle.pop_slots(free, 0, B, T)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_w)
    assert (loc_w[25:] == -1).all() and int(d_head.item()) == head
    assert int(status.item()) == va.STATUS_BAD_SLOT
    # the tree itself does not depend on the slots
    par_w, tok_w, _, _ = oracle.tree_build(tok, lp, T)
    np.testing.assert_array_equal(par.cpu().numpy(), par_w)
    np.testing.assert_array_equal(tk.cpu().numpy(), tok_w)


def _logits_for(rng, par, tok, V, follow=0.7):
    """Target logits whose greedy token at the prefix and at each node is, with
    probability `follow`, the token of one of that position's children (so the
    acceptance walk goes deep), else a random token."""
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


def test_decode_chain_in_one_graph(va):
    """Tree build -> segmented verify (draft rows written into the new slots
    first) -> greedy acceptance, captured once and replayed on two draws of
    drafter candidates, draft rows, queries and target logits copied into the
    same buffers; every output against the oracle chain."""
    rng = np.random.default_rng(2024)
    B, H, T, D, K, V = 4, 8, 16, 6, 4, 4096
    prefix = [300, 1000, 64, 2000]
    num_slots = 8192
    g = torch.Generator().manual_seed(77)
    pool = synth._bf16_normal((num_slots, 576), g)
    perm = torch.randperm(num_slots, generator=g).to(torch.int32)
    kv_indices = perm[:sum(prefix)]
    free = perm[sum(prefix):].numpy().copy()            # slots no prefix uses
    kv_indptr = torch.tensor(np.concatenate([[0], np.cumsum(prefix)]), dtype=torch.int32)

    def draw():
        tok, lp = _candidates(rng, B, D, K, "dirichlet")
        tok = tok % V
        q = synth._bf16_normal((B * T, H, 576), g)
        draft_kv = synth._bf16_normal((B * T, 576), g)
        par_w, tok_w, _, _ = oracle.tree_build(tok, lp, T)
        root, lg = _logits_for(rng, par_w, tok_w, V)
        return tok, lp, q, draft_kv, root, lg

    dev = "cuda"
    d_pool = pool.to(dev)
    d_ind, d_ip = kv_indices.to(dev), kv_indptr.to(dev)
    d_free = torch.from_numpy(free).to(dev)
    d_head = torch.zeros(1, dtype=torch.int32, device=dev)
    first = draw()
    d_tok = torch.from_numpy(first[0]).to(dev)
    d_lp = torch.from_numpy(first[1]).to(dev)
    d_q, d_dkv = first[2].to(dev), first[3].to(dev)
    d_root, d_lg = torch.from_numpy(first[4]).to(dev), torch.from_numpy(first[5]).to(dev)
    par = torch.full((B, T), -1, dtype=torch.int32, device=dev)
    dtok = torch.zeros(B, T, dtype=torch.int32, device=dev)
    depth = torch.zeros(B, T, dtype=torch.int32, device=dev)
    loc = torch.zeros(B * T, dtype=torch.int32, device=dev)
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
        va.tree_build(d_tok, d_lp, T, d_free, d_head, outputs=(par, dtok, depth, loc), stream=st)
        va.verify_attn_segmented(d_q, d_pool, d_ind, d_ip, loc, draft_kv=d_dkv, tree_parent=par,
                                 sm_scale=synth.SM_SCALE, nsplit=ns, workspace=ws, out=out,
                                 lse=lse, stream=st)
        va.tree_accept(d_root, d_lg, dtok, par, loc.view(B, T), workspace=acc_ws, outputs=acc,
                       stream=st)

    st.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        chain()
    torch.cuda.synchronize()
    d_head.zero_()
    torch.cuda.synchronize()

    pool_w = synth.as_u16(pool).copy()
    head = 0
    for rep, w in enumerate([first, draw()]):
        tok, lp, q, draft_kv, root, lg = w
        if rep:
            d_tok.copy_(torch.from_numpy(tok))
            d_lp.copy_(torch.from_numpy(lp))
            d_q.copy_(q)
            d_dkv.copy_(draft_kv)
            d_root.copy_(torch.from_numpy(root))
            d_lg.copy_(torch.from_numpy(lg))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        # the oracle chain
        par_w, tok_w, dep_w, _ = oracle.tree_build(tok, lp, T)
        loc_w, head = oracle.pop_slots(free, head, B, T)
        np.testing.assert_array_equal(par.cpu().numpy(), par_w)
        np.testing.assert_array_equal(dtok.cpu().numpy(), tok_w)
        np.testing.assert_array_equal(loc.cpu().numpy(), loc_w)
        assert int(d_head.item()) == head
        pool_w = oracle.append_rows(pool_w, synth.as_u16(draft_kv), loc_w)
        got_pool = d_pool.cpu().view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(got_pool, pool_w)
        slots, indptr, pre = oracle.segmented_lists(kv_indices.numpy(), kv_indptr.numpy(),
                                                    loc_w, T)
        bits, bad = oracle.tree_bits(par_w)
        assert bad == 0
        ro, rl, _ = oracle.verify_attn(synth.as_u16(q), pool_w, slots, indptr, pre, bits,
                                       synth.SM_SCALE)
        _gpu.compare(out, lse, ro, rl)
        assert va.read_status(ws) == 0
        alen_w, nodes_w, aslots_w, bonus_w, _ = oracle.tree_accept(root, lg, tok_w, par_w,
                                                                   loc_w.reshape(B, T))
        np.testing.assert_array_equal(acc[0].cpu().numpy(), alen_w)
        np.testing.assert_array_equal(acc[1].cpu().numpy(), nodes_w)
        np.testing.assert_array_equal(acc[2].cpu().numpy(), aslots_w)
        np.testing.assert_array_equal(acc[3].cpu().numpy(), bonus_w)
        assert alen_w.max() >= 2          # the walks went past the first level
