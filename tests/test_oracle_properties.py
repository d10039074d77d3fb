"""Randomised pins of the oracle (CPU): hypothesis draws small shapes, trees,
prefix lengths and segmentations; each example is checked against an
evaluation that shares nothing with the oracle.  Skipped where hypothesis is
not installed."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import synth  # noqa: E402
from tests import _brute  # noqa: E402
from tests.test_oracle_pins import _dense_mask  # noqa: E402

SETTINGS = dict(max_examples=25, deadline=None, derandomize=True)


@st.composite
def trees(draw, max_t=6):
    T = draw(st.integers(1, max_t))
    return [draw(st.integers(-1, i - 1)) for i in range(T)]


@settings(**SETTINGS)
@given(parent=trees(), P=st.integers(0, 6), H=st.integers(1, 3), seed=st.integers(0, 10_000))
def test_attention_matches_brute_force(oracle_mod, parent, P, H, seed):
    T = len(parent)
    s = synth.Spec("hyp", B=1, H=H, T=T, prefix=[P], num_slots=32, tree="random", seed=seed)
    w = synth.make(s)
    import torch
    w.parents = torch.tensor([parent], dtype=torch.int32)
    bits, bad = oracle_mod.tree_bits(w.parents.numpy())
    assert bad == 0
    out, lse, _ = oracle_mod.verify_attn(synth.as_u16(w.q), synth.as_u16(w.kv_pool),
                                         w.slot_idx.numpy(), w.kv_indptr.numpy(),
                                         w.prefix_len.numpy(), bits, s.sm_scale)
    bo, bl = _brute.brute_attention(synth.as_u16(w.q).astype(int).tolist(),
                                    synth.as_u16(w.kv_pool).astype(int).tolist(),
                                    w.slot_idx.tolist(), w.kv_indptr.tolist(),
                                    w.prefix_len.tolist(), [parent], s.sm_scale)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


@settings(**SETTINGS)
@given(parents=st.lists(trees(max_t=7), min_size=1, max_size=4).filter(
           lambda ps: len({len(p) for p in ps}) == 1),
       prefixes=st.lists(st.integers(0, 9), min_size=4, max_size=4))
def test_dense_mask_bits_are_the_ancestor_sets(oracle_mod, parents, prefixes):
    B, T = len(parents), len(parents[0])
    P = prefixes[:B]
    flat = np.concatenate([_dense_mask(np.array(parents[b]), P[b]).reshape(-1) for b in range(B)])
    indptr = np.concatenate([[0], np.cumsum(P)])
    bits, missing = oracle_mod.dense_mask_bits(flat.astype(np.uint8), indptr, T)
    want = [[sum(1 << k for k in path) for path in _brute.tree_paths(p)] for p in parents]
    assert missing == 0 and bits.tolist() == want


@settings(**SETTINGS)
@given(parent=trees(max_t=8), V=st.integers(9, 12), seed=st.integers(0, 10_000),
       hit=st.floats(0.0, 1.0))
def test_accept_is_the_longest_matching_root_path(oracle_mod, parent, V, seed, hit):
    rng = np.random.default_rng(seed)
    T = len(parent)
    root = rng.integers(0, 4, size=(1, V)).astype(np.float64)      # ties are common
    lg = rng.integers(0, 4, size=(1, T, V)).astype(np.float64)

    def greedy(row):
        return int(np.nanargmax(row))

    tokens = []
    for c in range(T):
        sib = [tokens[d] for d in range(c) if parent[d] == parent[c]]
        want = greedy(root[0] if parent[c] < 0 else lg[0, parent[c]])
        tok = want if (rng.random() < hit and want not in sib) else int(rng.integers(0, V))
        while tok in sib:
            tok = (tok + 1) % V
        tokens.append(tok)
    alen, nodes, _, bonus, _ = oracle_mod.tree_accept(root, lg, [tokens], [parent])
    best = []
    for path in (sorted(p) for p in _brute.tree_paths(parent)):
        ok = tokens[path[0]] == greedy(root[0]) and all(
            tokens[path[m + 1]] == greedy(lg[0, path[m]]) for m in range(len(path) - 1))
        if ok and len(path) > len(best):
            best = path
    assert alen[0] == len(best) and nodes[0, :len(best)].tolist() == best
    assert bonus[0] == (greedy(lg[0, best[-1]]) if best else greedy(root[0]))
