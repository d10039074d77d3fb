"""Independent pure-Python evaluations used to pin the oracle (tiny inputs only).

Nothing here is shared with the oracle: the visible-key sets are derived by a
depth-first walk from the prefix over child lists (the oracle walks parent
links upward), and the softmax is the textbook ratio exp(s_j) / sum_k exp(s_k)
with no max shift (inputs are kept small enough not to overflow).
"""
from __future__ import annotations

import math
import struct
from typing import Dict, List


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def tree_paths(parent: List[int]) -> List[set]:
    """For every node, the set of nodes on the path from the prefix to it (inclusive).

    Built top-down: start at the nodes hanging off the prefix and carry the path
    downward through the children lists.
    """
    T = len(parent)
    children: Dict[int, List[int]] = {i: [] for i in range(-1, T)}
    for i, p in enumerate(parent):
        children[p].append(i)
    paths: List[set] = [set() for _ in range(T)]
    stack = [(c, frozenset()) for c in children[-1]]
    while stack:
        node, above = stack.pop()
        here = set(above) | {node}
        paths[node] = here
        for c in children[node]:
            stack.append((c, frozenset(here)))
    return paths


def brute_attention(q_bits, kv_bits, slots, indptr, prefix, parent, sm_scale):
    """q_bits [B*T][H][576] ints, kv_bits [S][>=576] ints -> (out [rows][512], lse [rows])."""
    B = len(prefix)
    T = len(parent[0])
    H = len(q_bits[0])
    outs, lses = [], []
    for b in range(B):
        paths = tree_paths(list(parent[b]))
        P = prefix[b]
        for i in range(T):
            keys = list(range(P)) + [P + k for k in sorted(paths[i])]
            for h in range(H):
                qv = [bf16_value(x) for x in q_bits[b * T + i][h]]
                ex = []
                vs = []
                for j in keys:
                    row = kv_bits[slots[indptr[b] + j]]
                    kvals = [bf16_value(x) for x in row[:576]]
                    s = sm_scale * sum(a * c for a, c in zip(qv, kvals))
                    ex.append(math.exp(s))
                    vs.append(kvals[:512])
                z = sum(ex)
                outs.append([sum(ex[t] / z * vs[t][d] for t in range(len(keys))) for d in range(512)])
                lses.append(math.log(z))
    return outs, lses
