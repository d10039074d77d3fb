"""Greedy tree acceptance on the GPU against the oracle (integer results, so
compared exactly).  The argmax decides an integer: both sides compare the same
fp32 values with the same rule (lowest index among the largest non-NaN)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_speculative_decode_gb300 as m
    m.build()
    m.init()
    return m


def _case(B, T, V, seed, levels=None, nan_rows=0, p_hit=0.7):
    """Random logits (quantised to `levels` values to force ties when given),
    random trees, and draft tokens that are the target's token at the parent
    with probability p_hit (so that paths are accepted deep)."""
    rng = np.random.default_rng(seed)
    if levels:
        root = rng.integers(0, levels, size=(B, V)).astype(np.float32)
        lg = rng.integers(0, levels, size=(B, T, V)).astype(np.float32)
    else:
        root = rng.normal(size=(B, V)).astype(np.float32)
        lg = rng.normal(size=(B, T, V)).astype(np.float32)
    for _ in range(nan_rows):
        b, c = int(rng.integers(0, B)), int(rng.integers(0, T))
        if rng.random() < 0.5:
            lg[b, c, :] = np.nan
        else:
            lg[b, c, rng.random(V) < 0.3] = np.nan
    parents = np.array([[rng.integers(-1, i) for i in range(T)] for _ in range(B)], dtype=np.int32)
    tokens = rng.integers(0, V, size=(B, T)).astype(np.int32)
    for b in range(B):
        for c in range(T):
            if rng.random() < p_hit:
                src = root[b] if parents[b, c] < 0 else lg[b, parents[b, c]]
                tokens[b, c] = oracle.target_token(src)
    slots = rng.permutation(1 << 20)[:B * T].reshape(B, T).astype(np.int32)
    return root, lg, tokens, parents, slots


def _check(va, root, lg, tokens, parents, slots, want_bad=0):
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    alen, nodes, aslots, bonus, ws = va.tree_accept(d(root), d(lg), d(tokens), d(parents),
                                                    None if slots is None else d(slots))
    status = va.read_status(ws)
    r_len, r_nodes, r_slots, r_bonus, bad = oracle.tree_accept(root, lg, tokens, parents, slots)
    assert bad == want_bad
    assert status == (va.STATUS_BAD_PARENT if want_bad else 0)
    assert alen.cpu().numpy().tolist() == r_len.tolist()
    assert nodes.cpu().numpy().tolist() == r_nodes.tolist()
    assert aslots.cpu().numpy().tolist() == r_slots.tolist()
    assert bonus.cpu().numpy().tolist() == r_bonus.tolist()
    return r_len


@pytest.mark.parametrize("B,T,V,seed", [(1, 4, 37, 0), (3, 16, 5003, 1), (8, 16, 32000, 2),
                                        (2, 64, 9000, 3), (1, 16, 129280, 4)])
def test_accept_matches_oracle(va, B, T, V, seed):
    r_len = _check(va, *_case(B, T, V, seed))
    assert r_len.max() >= 1          # the case accepts something


def test_accept_ties_across_chunks(va):
    """Logits of only two values: the largest appears many times in every row,
    in several argmax chunks; the lowest index must win."""
    _check(va, *_case(4, 8, 70000, 5, levels=2))


def test_accept_nan_rows(va):
    _check(va, *_case(4, 12, 20000, 6, nan_rows=10))


def test_accept_without_slots(va):
    root, lg, tokens, parents, _ = _case(2, 8, 1000, 7)
    _check(va, root, lg, tokens, parents, None)


def test_accept_bad_parent_flagged(va):
    root, lg, tokens, parents, slots = _case(2, 8, 1000, 8)
    parents[1, 5] = 7
    _check(va, root, lg, tokens, parents, slots, want_bad=1)


def test_accept_nothing_accepted(va):
    root, lg, tokens, parents, slots = _case(3, 8, 500, 9, p_hit=0.0)
    tokens[:] = 499
    root[:, 499] = -1e9
    lg[:, :, 499] = -1e9
    r_len = _check(va, root, lg, tokens, parents, slots)
    assert r_len.tolist() == [0, 0, 0]
