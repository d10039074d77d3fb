"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test would fail on a plausible mistake in the oracle: a dropped rotary
term, a wrong scale, a mask off by one, a transposed operand, a wrong LSE
base, a wrong merge weight.
"""
import math
import os

import numpy as np
import pytest
import torch

import synth
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


def _tiny(B=1, H=2, T=3, prefix=(5,), tree="random", seed=11, num_slots=64, stride=576, scale=None):
    s = synth.Spec("pin", B=B, H=H, T=T, prefix=list(prefix), num_slots=num_slots, tree=tree,
                   seed=seed, row_stride=stride)
    w = synth.make(s)
    if scale is not None:
        w.spec.sm_scale = scale
    return w


def _run(oracle_mod, w, **kw):
    bits, bad = oracle_mod.tree_bits(w.parents.numpy())
    assert bad == 0
    out, lse, skipped = oracle_mod.verify_attn(
        synth.as_u16(w.q), synth.as_u16(w.kv_pool), w.slot_idx.numpy(), w.kv_indptr.numpy(),
        w.prefix_len.numpy(), bits, w.spec.sm_scale, **kw)
    return out, lse, skipped


def _dense_mask(parent, P):
    """Visibility [T, P+T] via transitive closure of the parent relation
    (boolean matrix powers), independent of walking parent links."""
    T = len(parent)
    A = np.zeros((T, T), dtype=bool)
    for i, p in enumerate(parent):
        if p >= 0:
            A[i, p] = True
    reach = np.eye(T, dtype=bool)
    step = np.eye(T, dtype=bool)
    for _ in range(T):
        step = (step.astype(np.int64) @ A.astype(np.int64)) > 0
        reach |= step
    m = np.zeros((T, P + T), dtype=bool)
    m[:, :P] = True
    m[:, P:] = reach
    return m


def _np_inputs(w):
    q = w.q.to(torch.float64).numpy()                   # [B*T, H, 576]
    kv = w.kv_pool.to(torch.float64).numpy()[:, :576]
    return q, kv


# ---------------------------------------------------------------- tree sets

def test_tree_bits_golden(oracle_mod):
    g = _parse(os.path.join(GOLDEN, "tree_small.txt"))
    parent = np.array([int(x) for x in g["parent"].split()], dtype=np.int32)
    want = np.array([int(x) for x in g["bits"].split()], dtype=np.uint64)
    bits, bad = oracle_mod.tree_bits(parent)
    assert bad == 0
    np.testing.assert_array_equal(bits, want)


def test_tree_bits_vs_topdown_paths(oracle_mod):
    gen = torch.Generator().manual_seed(3)
    for T in (1, 2, 5, 17, 33, 64):
        for tree in ("random", "chain", "flat"):
            parent = synth.make_parents(T, tree, gen).tolist()
            bits, bad = oracle_mod.tree_bits(np.array(parent, dtype=np.int32))
            assert bad == 0
            paths = _brute.tree_paths(parent)
            for i in range(T):
                assert int(bits[i]) == sum(1 << k for k in paths[i]), (T, tree, i)


def test_tree_bits_bad_parent_counted(oracle_mod):
    parent = np.array([-1, 0, 5, 1, -3], dtype=np.int32)   # node 2 forward, node 4 < -1
    bits, bad = oracle_mod.tree_bits(parent)
    assert bad == 2
    assert int(bits[2]) == 1 << 2 and int(bits[4]) == 1 << 4
    assert int(bits[3]) == (1 << 3) | (1 << 1) | 1


def test_tree_bits_child_of_bad_node(oracle_mod):
    """A node whose parent is invalid hangs off the prefix; its children see
    it and nothing above it (worked by hand)."""
    parent = np.array([-1, 0, 7, 2, -1, 3], dtype=np.int32)   # node 2's parent is not earlier
    bits, bad = oracle_mod.tree_bits(parent)
    assert bad == 1
    np.testing.assert_array_equal(bits, np.array([0b1, 0b11, 0b100, 0b1100, 0b10000, 0b101100],
                                                 dtype=np.uint64))


def test_extend_mask_golden_through_attention(oracle_mod):
    """q = 0 gives uniform weights over the visible keys; one-hot value rows then
    read the visible set straight out of the attention output."""
    g = _parse(os.path.join(GOLDEN, "extend_mask_small.txt"))
    P = int(g["prefix"])
    parent = np.array([int(x) for x in g["parent"].split()], dtype=np.int32)
    T = len(parent)
    rows = [np.array([int(x) for x in g[f"row{i}"].split()]) for i in range(T)]
    N = P + T
    kv = torch.zeros(N, 576, dtype=torch.bfloat16)
    for j in range(N):
        kv[j, j] = 1.0
    q = torch.zeros(T, 1, 576, dtype=torch.bfloat16)
    bits, _ = oracle_mod.tree_bits(parent[None])
    out, lse, _ = oracle_mod.verify_attn(synth.as_u16(q), synth.as_u16(kv), np.arange(N, dtype=np.int32),
                                         np.array([0, N]), np.array([P]), bits, 0.1)
    for i in range(T):
        vis = rows[i].astype(bool)
        np.testing.assert_allclose(out[i, :N], vis / vis.sum(), rtol=0, atol=1e-15)
        np.testing.assert_allclose(out[i, N:], 0.0, atol=0)
        assert abs(lse[i] - math.log(vis.sum())) < 1e-15


def test_segmented_lists_golden(oracle_mod):
    g = _parse(os.path.join(GOLDEN, "segmented_small.txt"))
    T = int(g["T"])
    ints = lambda k: [int(x) for x in g[k].split()]
    slots, indptr, prefix = oracle_mod.segmented_lists(ints("kv_indices"), ints("kv_indptr"),
                                                       ints("out_cache_loc"), T)
    assert slots.tolist() == ints("slots")
    assert indptr.tolist() == ints("indptr")
    assert prefix.tolist() == ints("prefix")


def test_dense_mask_bits_golden(oracle_mod):
    g = _parse(os.path.join(GOLDEN, "segmented_small.txt"))
    T = int(g["T"])
    mask = np.array([int(x) for x in g["mask"].split()], dtype=np.uint8)
    bits, missing = oracle_mod.dense_mask_bits(mask, [int(x) for x in g["kv_indptr"].split()], T)
    assert missing == 0
    assert bits.reshape(-1).tolist() == [int(x) for x in g["bits"].split()]


def test_dense_mask_bits_of_the_extend_mask_golden(oracle_mod):
    g = _parse(os.path.join(GOLDEN, "extend_mask_small.txt"))
    P = int(g["prefix"])
    parent = [int(x) for x in g["parent"].split()]
    T = len(parent)
    mask = np.concatenate([np.array([int(x) for x in g[f"row{i}"].split()]) for i in range(T)])
    bits, missing = oracle_mod.dense_mask_bits(mask, [0, P], T)
    want, _ = oracle_mod.tree_bits(np.array(parent, dtype=np.int32)[None])
    assert missing == 0 and bits.tolist() == want.tolist()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dense_mask_bits_vs_tree_bits(oracle_mod, seed):
    """Masks from the transitive closure of the parent relation, read back as
    bits, equal the parent walk's sets; requests of different prefix lengths
    (one empty) place their rows one after the other."""
    rng = np.random.default_rng(seed)
    B, T = 4, 9
    prefixes = [0, 5, 1, 12]
    parents = np.array([[rng.integers(-1, i) for i in range(T)] for _ in range(B)], dtype=np.int32)
    flat = np.concatenate([_dense_mask(parents[b], prefixes[b]).reshape(-1) for b in range(B)])
    indptr = np.concatenate([[3], 3 + np.cumsum(prefixes)])   # non-zero start
    bits, missing = oracle_mod.dense_mask_bits(flat.astype(np.uint8), indptr, T)
    want, bad = oracle_mod.tree_bits(parents)
    assert missing == 0 and bad == 0
    assert bits.tolist() == want.tolist()


def test_dense_mask_bits_short_mask_reads_zero(oracle_mod):
    mask = np.ones(2 * (3 + 2), dtype=np.uint8)            # T=2 rows of prefix 3 + 2
    bits, missing = oracle_mod.dense_mask_bits(mask[:-1], [0, 3], 2)
    assert missing == 1 and bits.tolist() == [[3, 1]]


def test_append_rows_small(oracle_mod):
    pool = np.arange(4 * 6, dtype=np.uint16).reshape(4, 6)
    rows = np.array([[100, 101, 102], [200, 201, 202], [300, 301, 302]], dtype=np.uint16)
    out = oracle_mod.append_rows(pool, rows, [2, 9, 0])      # slot 9 is outside the pool
    want = pool.copy()
    want[2, :3] = [100, 101, 102]
    want[0, :3] = [300, 301, 302]
    assert np.array_equal(out, want) and np.array_equal(pool, np.arange(24).reshape(4, 6))


def test_tree_accept_golden(oracle_mod):
    g = _parse(os.path.join(GOLDEN, "accept_small.txt"))
    ints = lambda k: [int(x) for x in g[k].split()]
    T = len(ints("parent"))
    root = np.array([[float(x) for x in g["root"].split()]])
    lg = np.array([[[float(x) for x in g[f"node{i}"].split()] for i in range(T)]])
    alen, nodes, aslots, bonus, bad = oracle_mod.tree_accept(
        root, lg, [ints("tokens")], [ints("parent")], [ints("slots")])
    assert bad == 0
    assert alen.tolist() == [int(g["accept_len"])]
    assert nodes[0].tolist() == ints("accept_nodes")
    assert aslots[0].tolist() == ints("accept_slots")
    assert bonus.tolist() == [int(g["bonus"])]


def _nan_argmax(row):
    row = np.asarray(row, dtype=np.float64)
    return 0 if np.isnan(row).all() else int(np.nanargmax(row))


def test_target_token_is_nanargmax(oracle_mod):
    rng = np.random.default_rng(3)
    for _ in range(200):
        row = rng.integers(0, 4, size=int(rng.integers(1, 40))).astype(np.float64)
        row[rng.random(row.shape[0]) < 0.2] = np.nan
        if rng.random() < 0.1:
            row[:] = np.nan
        assert oracle_mod.target_token(row) == _nan_argmax(row)


@pytest.mark.parametrize("seed", range(4))
def test_tree_accept_is_the_longest_matching_root_path(oracle_mod, seed):
    """With distinct tokens among siblings, the accepted path is the longest
    root path whose every token is the target's token at its parent (found
    here by checking every node's path), and the bonus token is the target's
    token at its end."""
    rng = np.random.default_rng(seed)
    B, T, V = 6, 12, 16          # V > T: a free token always exists among siblings
    root = rng.normal(size=(B, V))
    lg = rng.normal(size=(B, T, V))
    parents = np.array([[rng.integers(-1, i) for i in range(T)] for _ in range(B)])
    tokens = np.zeros((B, T), dtype=np.int64)
    for b in range(B):
        for c in range(T):
            sib = [tokens[b, d] for d in range(c) if parents[b, d] == parents[b, c]]
            want = _nan_argmax(root[b] if parents[b, c] < 0 else lg[b, parents[b, c]])
            # often the target's token, never a sibling's
            tok = want if (rng.random() < 0.7 and want not in sib) else int(rng.integers(0, V))
            while tok in sib:
                tok = (tok + 1) % V
            tokens[b, c] = tok
    alen, nodes, _, bonus, _ = oracle_mod.tree_accept(root, lg, tokens, parents)
    for b in range(B):
        best = []
        for c in range(T):
            path, k = [], c
            while k >= 0:
                path.append(k)
                k = parents[b, k]
            path = path[::-1]
            ok = tokens[b, path[0]] == _nan_argmax(root[b]) and all(
                tokens[b, path[m + 1]] == _nan_argmax(lg[b, path[m]]) for m in range(len(path) - 1))
            if ok and len(path) > len(best):
                best = path
        assert alen[b] == len(best) and nodes[b, :len(best)].tolist() == best
        end = _nan_argmax(lg[b, best[-1]]) if best else _nan_argmax(root[b])
        assert bonus[b] == end


def test_tree_accept_bad_parent_hangs_off_the_prefix(oracle_mod):
    root = np.array([[0.0, 5.0]])
    lg = np.zeros((1, 3, 2))
    lg[0, 2, 0] = 1.0
    alen, nodes, _, bonus, bad = oracle_mod.tree_accept(root, lg, [[0, 0, 1]], [[-1, 0, 2]])
    assert bad == 1 and alen.tolist() == [1] and nodes[0, 0] == 2 and bonus.tolist() == [0]


def test_segmented_attention_is_slot_relocation_invariant(oracle_mod):
    """Draft rows moved to other pool slots, with out_cache_loc following them,
    give bit-identical attention."""
    w = _tiny(B=2, H=2, T=3, prefix=(4, 0), num_slots=64, seed=5)
    sl, ip = w.slot_idx.numpy(), w.kv_indptr.numpy()
    P = w.prefix_len.numpy()
    T = w.spec.T
    ind = np.concatenate([sl[ip[b]:ip[b] + P[b]] for b in range(2)])
    kip = np.concatenate([[0], np.cumsum(P)])
    loc = np.concatenate([sl[ip[b] + P[b]:ip[b + 1]] for b in range(2)])
    bits, _ = oracle_mod.tree_bits(w.parents.numpy())

    def attn(kv, loc_):
        s2, ip2, p2 = oracle_mod.segmented_lists(ind, kip, loc_, T)
        return oracle_mod.verify_attn(synth.as_u16(w.q), synth.as_u16(kv), s2, ip2, p2, bits,
                                      w.spec.sm_scale)[:2]

    o1, l1 = attn(w.kv_pool, loc)
    used = set(sl.tolist())
    free = [r for r in range(w.kv_pool.shape[0]) if r not in used][:len(loc)]
    kv2 = w.kv_pool.clone()
    for a, b2 in zip(loc, free):
        kv2[b2] = w.kv_pool[a]
        kv2[a] = 0
    o2, l2 = attn(kv2, np.array(free, dtype=np.int32))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    o0, l0 = oracle_mod.verify_attn(synth.as_u16(w.q), synth.as_u16(w.kv_pool), sl, ip, P, bits,
                                    w.spec.sm_scale)[:2]
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


# ------------------------------------------------------ brute force / library

@pytest.mark.parametrize("seed,H,T,P,tree", [(1, 2, 3, 4, "random"), (2, 1, 4, 0, "random"),
                                             (3, 3, 2, 6, "chain"), (4, 2, 5, 1, "flat")])
def test_oracle_vs_pure_python_brute_force(oracle_mod, seed, H, T, P, tree):
    w = _tiny(H=H, T=T, prefix=(P,), tree=tree, seed=seed, num_slots=32)
    out, lse, _ = _run(oracle_mod, w)
    qb = synth.as_u16(w.q).astype(int).tolist()
    kb = synth.as_u16(w.kv_pool).astype(int).tolist()
    bo, bl = _brute.brute_attention(qb, kb, w.slot_idx.tolist(), w.kv_indptr.tolist(),
                                    w.prefix_len.tolist(), w.parents.tolist(), w.spec.sm_scale)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def test_oracle_vs_torch_sdpa_fp64(oracle_mod):
    """Library routine: fp64 scaled_dot_product_attention with an explicit mask
    built by transitive closure; lse from torch.logsumexp of the masked logits."""
    w = _tiny(B=2, H=3, T=6, prefix=(9, 4), seed=5, num_slots=128)
    out, lse, _ = _run(oracle_mod, w)
    q, kv = _np_inputs(w)
    B, T, H = 2, 6, 3
    r = 0
    for b in range(B):
        P = int(w.prefix_len[b])
        N = P + T
        sl = w.slot_idx[int(w.kv_indptr[b]):int(w.kv_indptr[b]) + N].long()
        K = torch.from_numpy(kv)[sl]                                  # [N, 576]
        Q = torch.from_numpy(q[b * T:(b + 1) * T]).permute(1, 0, 2)   # [H, T, 576]
        mask = torch.from_numpy(_dense_mask(w.parents[b].tolist(), P))
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, K.expand(H, N, 576), K[:, :512].expand(H, N, 512), attn_mask=mask,
            scale=w.spec.sm_scale)                                     # [H, T, 512]
        logits = (Q @ K.T) * w.spec.sm_scale
        l = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)  # [H, T]
        o_rows = o.permute(1, 0, 2).reshape(T * H, 512).numpy()
        l_rows = l.permute(1, 0).reshape(T * H).numpy()
        np.testing.assert_allclose(out[r:r + T * H], o_rows, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r:r + T * H], l_rows, rtol=0, atol=1e-12)
        r += T * H


def test_rotary_columns_enter_scores(oracle_mod):
    """Changing only the 64 rotary columns of q changes the result; changing
    columns beyond 576 of a wider pool row does not."""
    w = _tiny(H=2, T=3, prefix=(4,), seed=21, stride=640)
    out0, lse0, _ = _run(oracle_mod, w)
    w.kv_pool[:, 576:] = 7.0
    out1, lse1, _ = _run(oracle_mod, w)
    np.testing.assert_array_equal(out0, out1)
    w.q[:, :, 512:] *= -1.0
    out2, lse2, _ = _run(oracle_mod, w)
    assert np.abs(lse2 - lse0).max() > 1e-3


# ------------------------------------------------------------- identities

def test_chain_tree_equals_causal(oracle_mod):
    """A chain-shaped tree is bottom-right aligned causal attention: node i sees
    keys 0 .. P+i."""
    from scipy.special import logsumexp, softmax
    P, T, H = 7, 5, 2
    w = _tiny(H=H, T=T, prefix=(P,), tree="chain", seed=8, num_slots=64)
    out, lse, _ = _run(oracle_mod, w)
    q, kv = _np_inputs(w)
    K = kv[w.slot_idx.numpy()]
    causal = np.tril(np.ones((T, P + T), dtype=bool), k=P)
    for i in range(T):
        for h in range(H):
            s = w.spec.sm_scale * (K @ q[i, h])
            s = np.where(causal[i], s, -np.inf)
            np.testing.assert_allclose(out[i * H + h], softmax(s) @ K[:, :512], rtol=0, atol=1e-12)
            assert abs(lse[i * H + h] - logsumexp(s)) < 1e-12


def test_single_node_equals_decode(oracle_mod):
    """T = 1: plain decode attention over all P + 1 keys."""
    from scipy.special import logsumexp, softmax
    P, H = 9, 3
    w = _tiny(H=H, T=1, prefix=(P,), seed=9, num_slots=64)
    out, lse, _ = _run(oracle_mod, w)
    q, kv = _np_inputs(w)
    K = kv[w.slot_idx.numpy()]
    for h in range(H):
        s = w.spec.sm_scale * (K @ q[0, h])
        np.testing.assert_allclose(out[h], softmax(s) @ K[:, :512], rtol=0, atol=1e-12)
        assert abs(lse[h] - logsumexp(s)) < 1e-12


def test_slot_relocation_is_exact(oracle_mod):
    """Moving rows to other pool slots and remapping the table gives identical bits."""
    w = _tiny(B=2, H=2, T=4, prefix=(6, 3), seed=12, num_slots=64)
    out0, lse0, _ = _run(oracle_mod, w)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(1))
    newpool = torch.empty_like(w.kv_pool)
    newpool[perm] = w.kv_pool
    w.kv_pool = newpool
    w.slot_idx = perm[w.slot_idx.long()].to(torch.int32)
    out1, lse1, _ = _run(oracle_mod, w)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)


def test_prefix_order_invariance(oracle_mod):
    w = _tiny(H=2, T=3, prefix=(11,), seed=13, num_slots=64)
    out0, lse0, _ = _run(oracle_mod, w)
    perm = torch.randperm(11, generator=torch.Generator().manual_seed(2))
    w.slot_idx[:11] = w.slot_idx[:11][perm]
    out1, lse1, _ = _run(oracle_mod, w)
    np.testing.assert_allclose(out0, out1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse0, lse1, rtol=0, atol=1e-12)


def test_tree_key_order_matters(oracle_mod):
    """Swapping the slots of two tree nodes must change the result (the mask is
    positional over the tree keys) -- guards against a mask that ignores k."""
    w = _tiny(H=1, T=3, prefix=(2,), tree="chain", seed=14, num_slots=32)
    out0, _, _ = _run(oracle_mod, w)
    a, b = int(w.slot_idx[2]), int(w.slot_idx[4])
    w.slot_idx[2], w.slot_idx[4] = b, a
    out1, _, _ = _run(oracle_mod, w)
    assert np.abs(out0 - out1).max() > 1e-6


def test_head_permutation(oracle_mod):
    w = _tiny(H=4, T=3, prefix=(5,), seed=15, num_slots=64)
    out0, lse0, _ = _run(oracle_mod, w)
    perm = torch.tensor([2, 0, 3, 1])
    w.q = w.q[:, perm].contiguous()
    out1, lse1, _ = _run(oracle_mod, w)
    T, H = 3, 4
    o0 = out0.reshape(T, H, 512)[:, perm.numpy()]
    np.testing.assert_array_equal(o0.reshape(-1, 512), out1)
    np.testing.assert_array_equal(lse0.reshape(T, H)[:, perm.numpy()].reshape(-1), lse1)


# ----------------------------------------------------------- split algebra

def test_lse_merge_of_splits_equals_unsplit(oracle_mod):
    w = _tiny(B=1, H=2, T=5, prefix=(23,), seed=16, num_slots=64)
    out, lse, _ = _run(oracle_mod, w)
    N = 28
    gen = np.random.default_rng(0)
    for trial in range(4):
        cuts = sorted(set([0, N] + list(gen.integers(0, N + 1, size=trial + 2))))
        cuts = [0] + cuts if cuts[0] != 0 else cuts
        # add an empty split and a split entirely past the end
        windows = list(zip(cuts[:-1], cuts[1:])) + [(5, 5), (N, N + 10)]
        lps, ops = [], []
        for k0, k1 in windows:
            o, l, _ = _run(oracle_mod, w, k0=k0, k1=k1)
            lps.append(l)
            ops.append(o)
        mo, ml = oracle_mod.lse_merge(np.stack(lps), np.stack(ops))
        np.testing.assert_allclose(mo, out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(ml, lse, rtol=0, atol=1e-12)


def test_lse_merge_closed_forms(oracle_mod):
    o = np.array([[[1.0, -2.0]], [[3.0, 4.0]]])
    lp = np.array([[0.5], [0.5]])
    mo, ml = oracle_mod.lse_merge(lp, o)
    assert abs(ml[0] - (0.5 + math.log(2.0))) < 1e-15
    np.testing.assert_allclose(mo[0], [2.0, 1.0], atol=1e-15)
    lp2 = np.array([[math.log(3.0)], [-np.inf]])
    mo2, ml2 = oracle_mod.lse_merge(lp2, o)
    assert abs(ml2[0] - math.log(3.0)) < 1e-15
    np.testing.assert_allclose(mo2[0], o[0, 0], atol=0)
    mo3, ml3 = oracle_mod.lse_merge(np.full((2, 1), -np.inf), o)
    assert ml3[0] == -np.inf and np.all(mo3 == 0)


# ------------------------------------------------------------ closed forms

def test_zero_query_gives_mean_of_visible_values(oracle_mod):
    P, T, H = 6, 4, 2
    w = _tiny(H=H, T=T, prefix=(P,), seed=17, num_slots=64)
    w.q.zero_()
    out, lse, _ = _run(oracle_mod, w)
    _, kv = _np_inputs(w)
    K = kv[w.slot_idx.numpy()]
    mask = _dense_mask(w.parents[0].tolist(), P)
    for i in range(T):
        vis = mask[i]
        for h in range(H):
            np.testing.assert_allclose(out[i * H + h], K[vis, :512].mean(0), rtol=0, atol=1e-13)
            assert abs(lse[i * H + h] - math.log(vis.sum())) < 1e-13


def test_identical_keys(oracle_mod):
    P, T, H = 5, 3, 2
    w = _tiny(H=H, T=T, prefix=(P,), seed=18, num_slots=32)
    w.kv_pool[:] = w.kv_pool[3]
    out, lse, _ = _run(oracle_mod, w)
    q, kv = _np_inputs(w)
    mask = _dense_mask(w.parents[0].tolist(), P)
    for i in range(T):
        for h in range(H):
            s = w.spec.sm_scale * float(q[i, h] @ kv[3])
            assert abs(lse[i * H + h] - (s + math.log(mask[i].sum()))) < 1e-12
            np.testing.assert_allclose(out[i * H + h], kv[3, :512], rtol=0, atol=1e-12)


def test_dominant_key(oracle_mod):
    """One key whose scaled logit exceeds all others by > 50 takes all the weight."""
    P, T, H = 8, 2, 1
    w = _tiny(H=H, T=T, prefix=(P,), tree="chain", seed=19, num_slots=32)
    w.q.zero_()
    w.q[:, :, 0] = 4.0
    w.kv_pool[:, 0] = 0.0
    dom = int(w.slot_idx[3])
    w.kv_pool[dom, 0] = 256.0        # logit gap = 4 * 256 / sqrt(192) ~ 73.9
    out, lse, _ = _run(oracle_mod, w)
    _, kv = _np_inputs(w)
    for r in range(T * H):
        np.testing.assert_allclose(out[r], kv[dom, :512], rtol=0, atol=1e-20 + 1e-25)
        assert abs(lse[r] - 4.0 * 256.0 * w.spec.sm_scale) < 1e-12


def test_scale_enters_linearly(oracle_mod):
    """lse(scale=0) = ln|K|; and out depends on the scale (guards a dropped scale)."""
    w = _tiny(H=1, T=2, prefix=(4,), tree="chain", seed=20, num_slots=32)
    w.spec.sm_scale = 0.0
    out0, lse0, _ = _run(oracle_mod, w)
    np.testing.assert_allclose(lse0, [math.log(5), math.log(6)], atol=1e-15)
    w.spec.sm_scale = 0.3
    out1, _, _ = _run(oracle_mod, w)
    assert np.abs(out1 - out0).max() > 1e-3


# ------------------------------------------------------ skips and windows

def test_out_of_range_slot_is_skipped(oracle_mod):
    w = _tiny(H=2, T=2, prefix=(6,), tree="chain", seed=22, num_slots=32)
    ref = _tiny(H=2, T=2, prefix=(5,), tree="chain", seed=22, num_slots=32)
    ref.q, ref.kv_pool = w.q, w.kv_pool
    ref.slot_idx = torch.cat([w.slot_idx[:2], w.slot_idx[3:]])
    ref.kv_indptr = torch.tensor([0, 7], dtype=torch.int32)
    w.slot_idx[2] = 32 + 5
    out, lse, skipped = _run(oracle_mod, w)
    assert skipped == 2 * 2          # every row of both nodes skips that prefix key
    out_r, lse_r, _ = _run(oracle_mod, ref)
    np.testing.assert_allclose(out, out_r, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_r, rtol=0, atol=1e-13)


def test_row_subset_matches_full(oracle_mod):
    w = _tiny(B=2, H=3, T=4, prefix=(7, 2), seed=23, num_slots=64)
    out, lse, _ = _run(oracle_mod, w)
    rows = [0, 5, 13, 23]
    o2, l2, _ = _run(oracle_mod, w, rows=rows)
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(l2, lse[rows])


# ------------------------------------------------------------------ defrag

def test_defrag_copies_rows_and_preserves_attention(oracle_mod):
    # live rows in [0, 64) of a 128-row pool; destinations in the free upper half
    w = _tiny(B=2, H=2, T=3, prefix=(5, 4), seed=24, num_slots=64)
    w.kv_pool = torch.cat([w.kv_pool, synth._bf16_normal((64, 576), torch.Generator().manual_seed(9))])
    out0, lse0, _ = _run(oracle_mod, w)
    pool = synth.as_u16(w.kv_pool)
    ip = w.kv_indptr.numpy().astype(np.int64)
    dst = np.array([80, 100], dtype=np.int64)
    src = w.slot_idx.numpy()
    newpool, newslots = oracle_mod.defrag(pool, src, ip, dst)
    touched = set()
    for b in range(2):
        for i in range(ip[b + 1] - ip[b]):
            assert newslots[ip[b] + i] == dst[b] + i
            np.testing.assert_array_equal(newpool[dst[b] + i], pool[src[ip[b] + i]])
            touched.add(int(dst[b] + i))
    for r in range(128):
        if r not in touched:
            np.testing.assert_array_equal(newpool[r], pool[r])
    bits, _ = oracle_mod.tree_bits(w.parents.numpy())
    out1, lse1, _ = oracle_mod.verify_attn(synth.as_u16(w.q), newpool, newslots, ip,
                                           w.prefix_len.numpy(), bits, w.spec.sm_scale)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)


# ------------------------------------------------------- draft tree build

def test_tree_build_golden(oracle_mod):
    g = _parse(os.path.join(GOLDEN, "tree_build_small.txt"))
    D = sum(1 for k in g if k.startswith("tokens") and k[6:].isdigit())
    tok = np.array([[[int(x) for x in g[f"tokens{d}"].split()] for d in range(D)]])
    lp = np.array([[[float(x) for x in g[f"logp{d}"].split()] for d in range(D)]],
                  dtype=np.float32)
    T = int(g["T"])
    par, tk, dp, _ = oracle_mod.tree_build(tok, lp, T)
    ints = lambda k: [int(x) for x in g[k].split()]
    assert par[0].tolist() == ints("parent")
    assert tk[0].tolist() == ints("tokens")
    assert dp[0].tolist() == ints("depth")


def _brute_paths(lp_sorted, D, K):
    """Every node of the candidate tree (rank paths of length 1..D) with its
    float32 running score, by exhaustive enumeration."""
    import itertools
    out = []
    for d in range(1, D + 1):
        for ranks in itertools.product(range(K), repeat=d):
            s = np.float32(0)
            for i, r in enumerate(ranks):
                s = np.float32(s + lp_sorted[i][r])
            out.append((ranks, s))
    return out


def _sorted_candidates(tok, lp):
    """Per depth: candidates by log-probability (NaN/+inf -> -inf), highest first."""
    D, K = tok.shape
    ts, ls = [], []
    for d in range(D):
        v = [np.float32(-np.inf) if (x != x or x == np.inf) else np.float32(x) for x in lp[d]]
        o = sorted(range(K), key=lambda k: (-float(v[k]), k))
        ts.append([int(tok[d][k]) for k in o])
        ls.append([v[k] for k in o])
    return ts, ls


def _as_tree(paths, ts):
    """(parent, tokens, depth) of rank paths listed in tree order."""
    idx = {p: i for i, p in enumerate(paths)}
    parent = [idx[p[:-1]] if len(p) > 1 else -1 for p in paths]
    return parent, [ts[len(p) - 1][p[-1]] for p in paths], [len(p) - 1 for p in paths]


@pytest.mark.parametrize("seed", range(6))
def test_tree_build_is_the_global_top_T_for_log_probabilities(oracle_mod, seed):
    """With log-probabilities (all <= 0) a child never outscores its parent,
    so growing the tree best first selects the T best nodes of the whole
    candidate tree: here every node is enumerated and sorted (score desc,
    depth asc, rank path asc) and the first T compared with the oracle."""
    rng = np.random.default_rng(seed)
    B, D, K = 3, 4, 3
    tok = rng.integers(0, 50, size=(B, D, K))
    lp = np.log(rng.dirichlet(np.ones(K), size=(B, D))).astype(np.float32)
    if seed % 2:               # quantise to force ties
        lp = (np.round(lp * 2) / 2).astype(np.float32)
    if seed == 5:
        lp[0, 1, 2] = np.nan
        lp[1, 0, 0] = -np.inf
    T = int(rng.integers(1, 30))
    par, tk, dp, _ = oracle_mod.tree_build(tok, lp, T)
    for b in range(B):
        ts, ls = _sorted_candidates(tok[b], lp[b])
        nodes = _brute_paths(ls, D, K)
        nodes.sort(key=lambda n: (-float(n[1]), len(n[0]), n[0]))
        want = _as_tree([n[0] for n in nodes[:T]], ts)
        assert par[b].tolist() == want[0]
        assert tk[b].tolist() == want[1]
        assert dp[b].tolist() == want[2]


@pytest.mark.parametrize("seed", range(6))
def test_tree_build_equals_a_scan_of_every_attachable_node(oracle_mod, seed):
    """Best first with no heap: at each step every node whose parent is already
    in the tree is scored and the best taken (same tie rule).  Holds for any
    scores, including positive ones (raw logits passed by mistake), where the
    tree is no longer the global top T."""
    rng = np.random.default_rng(100 + seed)
    B, D, K = 2, 3, 4
    tok = rng.integers(0, 9, size=(B, D, K))
    lp = rng.normal(0, 1.5, size=(B, D, K)).astype(np.float32)
    if seed % 2:
        lp = np.round(lp).astype(np.float32)
    T = int(rng.integers(1, 40))
    par, tk, dp, _ = oracle_mod.tree_build(tok, lp, T)
    for b in range(B):
        ts, ls = _sorted_candidates(tok[b], lp[b])
        score = {p: s for p, s in _brute_paths(ls, D, K)}
        chosen = []
        for _ in range(T):
            have = set(chosen)
            cand = [p for p in score if p not in have and (len(p) == 1 or p[:-1] in have)]
            best = min(cand, key=lambda p: (-float(score[p]), len(p), p))
            chosen.append(best)
        want = _as_tree(chosen, ts)
        assert par[b].tolist() == want[0]
        assert tk[b].tolist() == want[1]
        assert dp[b].tolist() == want[2]


def test_tree_build_peaked_drafter_gives_a_chain(oracle_mod):
    """A drafter certain of one token per depth (log-prob 0 there, -30 for the
    others): the first D nodes are the chain of those tokens."""
    D, K = 6, 4
    tok = np.arange(D * K).reshape(1, D, K)
    lp = np.full((1, D, K), -30.0, dtype=np.float32)
    lp[0, np.arange(D), np.arange(D) % K] = 0.0
    par, tk, dp, _ = oracle_mod.tree_build(tok, lp, D)
    assert par[0].tolist() == [-1] + list(range(D - 1))
    assert tk[0].tolist() == [d * K + d % K for d in range(D)]
    assert dp[0].tolist() == list(range(D))


def test_pop_slots(oracle_mod):
    free = np.array([7, 3, 9, 1, 4, 8], dtype=np.int32)
    loc, head = oracle_mod.pop_slots(free, 1, 2, 2)
    assert loc.tolist() == [3, 9, 1, 4] and head == 5
    loc, head = oracle_mod.pop_slots(free, 4, 2, 2)    # the list runs out
    assert loc.tolist() == [4, 8, -1, -1] and head == 8


# ---------------------------------------------- contiguous placement and compaction

def _pool(rows, cols=3):
    """Row r of a small pool holds r*10 + c in column c (easy to read back)."""
    return (np.arange(rows)[:, None] * 10 + np.arange(cols)[None, :]).astype(np.uint16)


def test_append_contiguous_golden(oracle_mod):
    """Two requests owning rows [0, 6) and [6, 12): prefixes of 2 and 1 rows,
    three draft nodes each, so request 0's nodes land in rows 2-4 and request
    1's in rows 7-9 (worked by hand)."""
    pool = _pool(12)
    draft = (900 + np.arange(6)[:, None] * 10 + np.arange(2)[None, :]).astype(np.uint16)
    new, loc, bad = oracle_mod.append_contiguous(pool, draft, [0, 6], [2, 1], [6, 6], 3)
    assert loc.tolist() == [2, 3, 4, 7, 8, 9] and bad == 0
    want = pool.copy()
    for r, row in zip([2, 3, 4, 7, 8, 9], range(6)):
        want[r, :2] = [900 + row * 10, 901 + row * 10]
    np.testing.assert_array_equal(new, want)


def test_append_contiguous_capacity_and_pool_bounds(oracle_mod):
    pool = _pool(10)
    draft = np.ones((6, 3), dtype=np.uint16)
    # request 0: 4 + 3 > 6 reserved rows; request 1: rows 8, 9, 10 -- the last
    # outside the pool
    new, loc, bad = oracle_mod.append_contiguous(pool, draft, [0, 7], [4, 1], [6, 6], 3)
    assert loc.tolist() == [-1, -1, -1, 8, 9, -1] and bad == 4
    np.testing.assert_array_equal(new[:8], pool[:8])
    assert (new[8:10] == 1).all()


def test_compact_accepted_golden(oracle_mod):
    """Continues the append example: request 0 accepts nodes 0 and 2 (rows 2
    and 4), request 1 accepts node 1 (row 8).  Request 0's rows become
    2 <- 2, 3 <- 4 and its prefix 2 -> 4; request 1's row 7 <- 8, prefix 1 -> 2
    (worked by hand)."""
    pool = _pool(12)
    new, pl, bad = oracle_mod.compact_accepted(pool, [0, 6], [2, 1], [6, 6], [2, 1],
                                               [[0, 2, -1], [1, -1, -1]], 3, cols=3)
    assert pl.tolist() == [4, 2] and bad == 0
    want = pool.copy()
    want[3] = pool[4]
    want[7] = pool[8]
    np.testing.assert_array_equal(new, want)


def test_compact_accepted_reads_before_writing(oracle_mod):
    """A path in decreasing node order (node 2, then node 0) with P = 1: row
    1 takes node 2's row (row 3) and row 2 takes node 0's row, which is row 1's
    old content -- right only when every row is read before any is written."""
    pool = _pool(8)
    new, pl, _ = oracle_mod.compact_accepted(pool, [0], [1], [8], [2], [[2, 0, -1]], 3, cols=3)
    np.testing.assert_array_equal(new[1], pool[3])
    np.testing.assert_array_equal(new[2], pool[1])
    assert pl.tolist() == [3]


def test_compact_accepted_edge_cases(oracle_mod):
    pool = _pool(20)
    # nothing accepted: unchanged pool and prefix; a full chain: identity moves
    new, pl, bad = oracle_mod.compact_accepted(pool, [0, 10], [3, 2], [8, 8], [0, 4],
                                               [[-1] * 4, [0, 1, 2, 3]], 4, cols=3)
    np.testing.assert_array_equal(new, pool)
    assert pl.tolist() == [3, 6] and bad == 0
    # a node outside [0, T), an accept count past T, a range past the reserve:
    # each request left unchanged and counted
    new, pl, bad = oracle_mod.compact_accepted(pool, [0, 5, 10], [1, 1, 6], [8, 8, 8],
                                               [1, 5, 1], [[4, -1, -1, -1], [0, 1, 2, 3],
                                                           [0, -1, -1, -1]], 4, cols=3)
    np.testing.assert_array_equal(new, pool)
    assert pl.tolist() == [1, 1, 6] and bad == 3


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_append_then_compact_keeps_the_logical_sequence(oracle_mod, seed):
    """Invariant: after the append and the compaction, request b's first
    prefix_len'[b] rows from kv_start[b] are, in order, its prefix rows and then
    the draft latents of its accepted nodes in path order -- the key sequence a
    paged step over (prefix slots, accepted nodes' slots) would read next.
    Written as a gather by list, independently of the in-place moves."""
    rng = np.random.default_rng(seed)
    B, T, cols = 3, 5, 4
    cap = 12
    ks = np.array([0, cap, 2 * cap]) + 3
    pl = rng.integers(0, cap - T + 1, size=B)
    pool = rng.integers(0, 60000, size=(3 * cap + 6, cols)).astype(np.uint16)
    draft = rng.integers(0, 60000, size=(B * T, cols)).astype(np.uint16)
    p1, loc, bad = oracle_mod.append_contiguous(pool, draft, ks, pl, [cap] * B, T)
    assert bad == 0
    alen = rng.integers(0, T + 1, size=B)
    nodes = np.full((B, T), -1, dtype=np.int32)
    for b in range(B):
        path = np.sort(rng.choice(T, size=alen[b], replace=False))
        nodes[b, :alen[b]] = path
    p2, pl2, bad = oracle_mod.compact_accepted(p1, ks, pl, [cap] * B, alen, nodes, T, cols=cols)
    assert bad == 0 and pl2.tolist() == (pl + alen).tolist()
    for b in range(B):
        logical = [p1[ks[b] + j] for j in range(pl[b])] + \
                  [draft[b * T + int(x)] for x in nodes[b, :alen[b]]]
        got = [p2[ks[b] + j] for j in range(pl2[b])]
        for a, g in zip(logical, got):
            np.testing.assert_array_equal(a, g)
        # rows outside the request's reserved range are untouched
    owned = np.zeros(p2.shape[0], dtype=bool)
    for b in range(B):
        owned[ks[b]:ks[b] + cap] = True
    np.testing.assert_array_equal(p2[~owned], pool[~owned])
