"""fp64 CPU oracle for MLA tree-verify attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
(``mla_speculative_decode_gb300``) and imports nothing from it; the product
path never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one thread
per group of output rows).  This module only compiles that file with gcc and
marshals numpy arrays into it.  bf16 tensors cross as their raw 16-bit
patterns (numpy ``uint16``); the C side widens them exactly.

Functions and the passages they follow (page titles and sections):
  tree_bits     -- The Checkpoint Report, "Mistakes and Incorrect Assumptions"
                   (draft rows of the extend mask) and "Input Knowledge
                   Required" (the DDTree draft tree).
  verify_attn   -- The Milestone Commit, "Input Knowledge Required" (attention
                   of the draft tokens against the full KV cache) and
                   "Context" (MLA latent cache, page_size=1 slots).
  lse_merge     -- The Commit That Locked In 6x Decode, "Input Knowledge
                   Required" (NSPLIT partial-reduce); The Milestone Commit,
                   "The Deeper Significance" (reduction kernel).
  defrag        -- The Checkpoint Report, "Input Knowledge Required" (KV
                   defragmentation keeps per-request KV contiguous).
  tree_accept   -- The Milestone Commit, "Input Knowledge Required" (the verify
                   step checks whether the draft predictions are correct); The
                   Checkpoint Report, "Input Knowledge Required to Understand
                   This Message" (a drafter proposes a tree of candidate tokens,
                   the target model checks them in one parallel pass).
  tree_build, pop_slots
                -- The Checkpoint Report, "Input Knowledge Required to
                   Understand This Message" (a drafter proposes candidate
                   tokens; DDTree builds a tree of draft tokens from them) and
                   The Commit That Locked In 6x Decode, "4. The Marshaling
                   Realization" (the per-step tree build, done on the host);
                   the draft tokens' slots are out_cache_loc (The Checkpoint
                   Report, "Mistakes and Incorrect Assumptions").  The pages
                   give no selection rule: this is the best-first reading
                   (highest cumulative log-probability first).
  segmented_lists, dense_mask_bits, append_rows
                -- The Checkpoint Report, "Mistakes and Incorrect Assumptions"
                   (the extend call takes the prefix slots in kv_indices, the
                   draft tokens' own slots at out_cache_loc, and a custom mask
                   with one row per draft token of stride prefix + q_len;
                   out_cache_loc is where the draft tokens' KV goes).
  append_contiguous, compact_accepted
                -- The Checkpoint Report, "Input Knowledge Required" (KV
                   defragmentation keeps per-request KV contiguous) and "The
                   Architecture of the Report" (defragmentation, the deferred
                   phase; its placement policy, "Tier 1 defrag", is named on
                   the pages but not specified).  The reading: a request owns
                   a reserved range of rows; its draft latents land right after
                   its prefix, and after acceptance the accepted path's rows
                   are moved to directly after the prefix, which grows by the
                   accepted count.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

D_QK = 576   # latent 512 + rotary 64
D_V = 512    # value = first 512 columns of the latent row

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_tree_bits.argtypes = [P, i32, P]
    lib.oracle_tree_bits.restype = i32
    lib.oracle_verify_attn.argtypes = [P, P, i64, i64, P, P, P, P, i32, i32, i32, i32, i32,
                                       dbl, i64, i64, P, i64, P, P, i32]
    lib.oracle_verify_attn.restype = i64
    lib.oracle_lse_merge.argtypes = [i32, P, P, i32, P, P]
    lib.oracle_lse_merge.restype = None
    lib.oracle_defrag.argtypes = [P, i64, i64, P, P, P, i32, P]
    lib.oracle_defrag.restype = i32
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def tree_bits(parent) -> tuple[np.ndarray, int]:
    """parent int32 [B, T] (or [T]) -> (ancestor-or-self bits uint64 same shape, #bad parents)."""
    par = _c(parent, np.int32)
    shape = par.shape
    par2 = par.reshape(-1, shape[-1])
    out = np.zeros(par2.shape, dtype=np.uint64)
    lib = _load()
    bad = 0
    for b in range(par2.shape[0]):
        row = np.ascontiguousarray(par2[b])
        ob = np.zeros(shape[-1], dtype=np.uint64)
        bad += lib.oracle_tree_bits(_ptr(row), int(shape[-1]), _ptr(ob))
        out[b] = ob
    return out.reshape(shape), bad


def verify_attn(q_bits, kv_bits, slots, kv_indptr, prefix_len, bits, sm_scale: float,
                k0: int = 0, k1: int = np.iinfo(np.int64).max,
                rows: Optional[Sequence[int]] = None, threads: Optional[int] = None):
    """Masked softmax attention of every (request, node, head) row.

    q_bits   uint16 [B*T, H, 576]      bf16 bit patterns
    kv_bits  uint16 [num_slots, stride] bf16 bit patterns (stride >= 576)
    slots    int32  [sum_b N_b]         request b's keys: prefix slots then T tree slots
    kv_indptr int   [B+1]               offsets of each request in ``slots``
    prefix_len int  [B]
    bits     uint64 [B, T]              ancestor-or-self sets
    Returns (out float64 [rows, 512], lse float64 [rows], skipped_keys).
    ``rows`` selects flat row indices ((b*T + i)*H + h); default all rows.
    ``[k0, k1)`` restricts every request to that window of key indices.
    """
    q = _c(q_bits, np.uint16)
    kv = _c(kv_bits, np.uint16)
    assert q.ndim == 3 and q.shape[2] == D_QK, q.shape
    assert kv.ndim == 2 and kv.shape[1] >= D_QK, kv.shape
    bits_ = _c(bits, np.uint64)
    B, T = bits_.shape
    H = q.shape[1]
    assert q.shape[0] == B * T
    sl = _c(slots, np.int32)
    ip = _c(kv_indptr, np.int64)
    pl = _c(prefix_len, np.int32)
    assert ip.shape == (B + 1,) and pl.shape == (B,)
    if rows is None:
        rows_arr = None
        nrows = B * T * H
    else:
        rows_arr = _c(rows, np.int64)
        nrows = rows_arr.shape[0]
    out = np.zeros((nrows, D_V), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    lib = _load()
    skipped = lib.oracle_verify_attn(
        _ptr(q), _ptr(kv), kv.shape[0], kv.shape[1], _ptr(sl), _ptr(ip), _ptr(pl),
        _ptr(bits_), B, T, H, D_QK, D_V, float(sm_scale), int(k0), int(k1),
        _ptr(rows_arr) if rows_arr is not None else None, nrows, _ptr(out), _ptr(lse),
        int(threads or default_threads()))
    if skipped < 0:
        raise ValueError("oracle_verify_attn: bad arguments")
    return out, lse, int(skipped)


def lse_merge(lse_parts, o_parts):
    """lse_parts [S, rows], o_parts [S, rows, Dv] -> (out [rows, Dv], lse [rows])."""
    lp = _c(lse_parts, np.float64)
    op = _c(o_parts, np.float64)
    S, nrows = lp.shape
    Dv = op.shape[2]
    out = np.zeros((nrows, Dv), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    lib = _load()
    for r in range(nrows):
        lr = np.ascontiguousarray(lp[:, r])
        orr = np.ascontiguousarray(op[:, r, :])
        o1 = np.zeros(Dv, dtype=np.float64)
        l1 = np.zeros(1, dtype=np.float64)
        lib.oracle_lse_merge(S, _ptr(lr), _ptr(orr), Dv, _ptr(o1), _ptr(l1))
        out[r] = o1
        lse[r] = l1[0]
    return out, lse


def segmented_lists(kv_indices, kv_indptr, out_cache_loc, T: int):
    """Two slot lists -> one list per request, prefix first, then the draft nodes.

    Request b's prefix slots are kv_indices[kv_indptr[b]:kv_indptr[b+1]] and its
    draft nodes' slots out_cache_loc[b*T:(b+1)*T].  Returns (slots int32,
    indptr int64 [B+1], prefix_len int32 [B]) in the layout ``verify_attn`` takes.
    """
    ind = [int(x) for x in np.asarray(kv_indices).reshape(-1)]
    ip = [int(x) for x in np.asarray(kv_indptr).reshape(-1)]
    loc = [int(x) for x in np.asarray(out_cache_loc).reshape(-1)]
    B = len(ip) - 1
    slots, indptr, prefix = [], [0], []
    for b in range(B):
        pre = ind[ip[b]:ip[b + 1]]
        slots += pre + loc[b * T:(b + 1) * T]
        indptr.append(len(slots))
        prefix.append(len(pre))
    return (np.array(slots, dtype=np.int32), np.array(indptr, dtype=np.int64),
            np.array(prefix, dtype=np.int32))


def dense_mask_bits(custom_mask, kv_indptr, T: int):
    """Dense extend-mask rows -> the draft-key part of each node's visible set.

    Request b (prefix P_b = kv_indptr[b+1] - kv_indptr[b]) owns T rows of P_b + T
    entries, after the rows of the requests before it; bit k of node i's set is
    row i, column P_b + k (non-zero = visible).  Entries past the end of the mask
    count as 0.  Returns (bits uint64 [B, T], number of entries past the end).
    """
    m = np.asarray(custom_mask).reshape(-1)
    ip = [int(x) for x in np.asarray(kv_indptr).reshape(-1)]
    B = len(ip) - 1
    bits = np.zeros((B, T), dtype=np.uint64)
    missing = 0
    start = 0                      # first entry of request b's rows
    for b in range(B):
        P = max(ip[b + 1] - ip[b], 0)
        for i in range(T):
            row = start + i * (P + T)
            v = 0
            for k in range(T):
                e = row + P + k
                if 0 <= e < m.shape[0]:
                    if m[e]:
                        v |= 1 << k
                else:
                    missing += 1
            bits[b, i] = v
        start += T * (P + T)
    return bits, missing


def append_rows(pool_bits, rows_bits, slots):
    """A copy of the pool with rows_bits[r] written into the first columns of
    pool row slots[r] (slots outside the pool are skipped)."""
    pool = np.array(pool_bits, dtype=np.uint16, copy=True, order="C")
    rows = np.asarray(rows_bits, dtype=np.uint16)
    for r, s in enumerate(np.asarray(slots).reshape(-1).tolist()):
        if 0 <= s < pool.shape[0]:
            pool[s, :rows.shape[1]] = rows[r]
    return pool


def target_token(row) -> int:
    """The target's greedy token for one logits row: the lowest index among the
    largest non-NaN values, 0 when every value is NaN."""
    best, idx = None, 0
    for i, v in enumerate(np.asarray(row, dtype=np.float64).tolist()):
        if v != v:                 # NaN
            continue
        if best is None or v > best:
            best, idx = v, i
    return idx


def tree_accept(root_logits, logits, tokens, parent, slots=None):
    """Greedy acceptance of each request's draft tree.

    Starting at the prefix with the target's token after it, repeatedly accept
    the lowest-numbered child of the current position whose draft token is the
    target's token there; stop when no child matches.  A node whose parent is
    not an earlier node counts as a child of the prefix.  Returns
    (accept_len [B], accept_nodes [B, T] (-1 padded), accept_slots [B, T]
    (-1 padded; all -1 without slots), bonus [B], #bad parents).
    """
    rl = np.asarray(root_logits)
    lg = np.asarray(logits)
    tk = np.asarray(tokens).tolist()
    par = np.asarray(parent).tolist()
    sl = None if slots is None else np.asarray(slots).tolist()
    B, T = lg.shape[0], lg.shape[1]
    alen = np.zeros(B, dtype=np.int64)
    nodes = -np.ones((B, T), dtype=np.int64)
    aslots = -np.ones((B, T), dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    bad = 0
    for b in range(B):
        p = [q if -1 <= q < i else -1 for i, q in enumerate(par[b])]
        bad += sum(1 for i, q in enumerate(par[b]) if not (-1 <= q < i))
        cur, n, t = -1, 0, target_token(rl[b])
        while True:
            kids = [c for c in range(T) if p[c] == cur and tk[b][c] == t]
            if not kids:
                break
            c = kids[0]
            nodes[b, n] = c
            if sl is not None:
                aslots[b, n] = sl[b][c]
            n += 1
            cur, t = c, target_token(lg[b, c])
        alen[b], bonus[b] = n, t
    return alen, nodes, aslots, bonus, bad


def _valid_logp(x: np.float32) -> np.float32:
    """A log-probability as the tree build reads it: NaN and +inf are not
    log-probabilities and count as -inf."""
    return np.float32(-np.inf) if (x != x or x == np.inf) else np.float32(x)


def tree_build(cand_tokens, cand_logp, T: int):
    """Draft tree of each request from the drafter's per-depth candidates.

    cand_tokens int [B, D, K], cand_logp float32 [B, D, K]: at depth d (the
    d+1-th draft position) the drafter proposes K tokens with their
    log-probabilities.  A tree node is a path of candidate choices, one per
    depth from depth 0 down; its score is the float32 running sum of the
    chosen log-probabilities, root first.  The tree is grown best first:
      1. at each depth, order the candidates by log-probability, highest
         first, ties by lower candidate index (NaN and +inf count as -inf);
      2. start from the empty tree; T times, add the highest-scoring node
         whose parent is in the tree (depth-0 nodes hang off the prefix),
         ties going to the shallower node, then to the path whose ranks are
         lexicographically smaller.
    Nodes are numbered in the order they were added, so a parent always
    precedes its children.  Returns (parent int32 [B, T] (-1: hangs off the
    prefix), tokens int32 [B, T], depth int32 [B, T] (0-based), ranks:
    a list per request of each node's rank path).
    """
    import heapq
    tok = np.asarray(cand_tokens)
    lp = np.asarray(cand_logp, dtype=np.float32)
    B, D, K = tok.shape
    parent = np.zeros((B, T), dtype=np.int32)
    tokens = np.zeros((B, T), dtype=np.int32)
    depth = np.zeros((B, T), dtype=np.int32)
    all_paths = []
    for b in range(B):
        # 1. candidates of each depth in order
        order, slp = [], []
        for d in range(D):
            vals = [_valid_logp(lp[b, d, k]) for k in range(K)]
            o = sorted(range(K), key=lambda k: (-float(vals[k]), k))
            order.append(o)
            slp.append([vals[k] for k in o])
        # 2. best first.  Every node whose parent is in the tree is reachable
        # as either the first child of a node in the tree or the next sibling
        # (next rank) of a node in the tree, so a heap holding, for each node
        # added, its first child and its next sibling always contains the best
        # candidate.  Heap entries: (-score, depth, ranks, score, parent
        # index, parent score), so the heap pops the order of step 2.
        zero = np.float32(0)
        heap = [(-float(slp[0][0]), 0, (0,), np.float32(zero + slp[0][0]), -1, zero)]
        paths = []
        for i in range(T):
            _, d, ranks, sc, par, psc = heapq.heappop(heap)
            parent[b, i] = par
            tokens[b, i] = int(tok[b, d, order[d][ranks[-1]]])
            depth[b, i] = d
            paths.append(ranks)
            if d + 1 < D:                       # first child
                c = np.float32(sc + slp[d + 1][0])
                heapq.heappush(heap, (-float(c), d + 1, ranks + (0,), c, i, sc))
            if ranks[-1] + 1 < K:               # next sibling
                c = np.float32(psc + slp[d][ranks[-1] + 1])
                heapq.heappush(heap, (-float(c), d, ranks[:-1] + (ranks[-1] + 1,), c, par, psc))
        all_paths.append(paths)
    return parent, tokens, depth, all_paths


def pop_slots(free_slots, head: int, B: int, T: int):
    """Draft node i of request b takes free_slots[head + b*T + i]; returns
    (out_cache_loc int32 [B*T] (-1 where the list has run out), new head)."""
    fs = np.asarray(free_slots).reshape(-1)
    loc = np.full(B * T, -1, dtype=np.int32)
    for j in range(B * T):
        if 0 <= head + j < fs.shape[0]:
            loc[j] = fs[head + j]
    return loc, head + B * T


def defrag(pool_bits, src_slots, src_indptr, dst_base):
    """Out-of-place compaction: returns (new pool uint16 copy, new slot table int32)."""
    pool = np.array(pool_bits, dtype=np.uint16, copy=True, order="C")
    src = _c(src_slots, np.int32)
    ip = _c(src_indptr, np.int64)
    db = _c(dst_base, np.int64)
    B = db.shape[0]
    slots_out = np.array(src, dtype=np.int32, copy=True)
    lib = _load()
    rc = lib.oracle_defrag(_ptr(pool), pool.shape[0], pool.shape[1], _ptr(src), _ptr(ip),
                           _ptr(db), B, _ptr(slots_out))
    if rc != 0:
        raise ValueError("oracle_defrag: slot out of range")
    return pool, slots_out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))


def append_contiguous(pool_bits, draft_bits, kv_start, prefix_len, capacity, T: int):
    """Draft latents of request b into the rows after its prefix.

    Node i of request b goes to row kv_start[b] + prefix_len[b] + i when the
    request's reserved range of capacity[b] rows holds prefix and draft
    (prefix_len[b] + T <= capacity[b]) and the row lies in the pool (and below
    2^31); otherwise the node gets no row.  Returns (a copy of the pool with
    draft_bits[b*T + i] written into the first columns of that row,
    out_cache_loc int32 [B*T] with the row or -1, the number of nodes without
    a row)."""
    pool = np.array(pool_bits, dtype=np.uint16, copy=True, order="C")
    draft = np.asarray(draft_bits, dtype=np.uint16)
    ks = np.asarray(kv_start).reshape(-1).tolist()
    pl = np.asarray(prefix_len).reshape(-1).tolist()
    cap = np.asarray(capacity).reshape(-1).tolist()
    B = len(ks)
    loc = np.full(B * T, -1, dtype=np.int32)
    bad = 0
    for b in range(B):
        fits = 0 <= pl[b] and pl[b] + T <= cap[b]
        for i in range(T):
            row = ks[b] + pl[b] + i
            if fits and 0 <= row < pool.shape[0] and row < 2 ** 31:
                pool[row, :draft.shape[1]] = draft[b * T + i]
                loc[b * T + i] = row
            else:
                bad += 1
    return pool, loc, bad


def compact_accepted(pool_bits, kv_start, prefix_len, capacity, accept_len, accept_nodes,
                     T: int, cols: int = D_QK):
    """Accepted path of request b moved to directly after its prefix.

    With P = prefix_len[b] and n = accept_len[b], the k-th accepted node
    (accept_nodes[b, k], a draft node whose row is kv_start[b] + P + node)
    has its first `cols` columns copied to row kv_start[b] + P + k, all n rows
    read before any is written; then prefix_len[b] becomes P + n.  A request
    whose n is outside [0, T], whose accepted nodes are outside [0, T), or
    whose rows fall outside its reserved range (P + T <= capacity[b]) or the
    pool is left unchanged and counted.  Returns (a copy of the pool, the new
    prefix_len int32 [B], the number of requests left unchanged)."""
    pool = np.array(pool_bits, dtype=np.uint16, copy=True, order="C")
    ks = np.asarray(kv_start).reshape(-1).tolist()
    pl = np.asarray(prefix_len).reshape(-1).astype(np.int64).tolist()
    cap = np.asarray(capacity).reshape(-1).tolist()
    alen = np.asarray(accept_len).reshape(-1).tolist()
    nodes = np.asarray(accept_nodes).reshape(len(ks), T)
    new_pl = np.array(pl, dtype=np.int32)
    bad = 0
    for b in range(len(ks)):
        P, n = pl[b], alen[b]
        path = [int(x) for x in nodes[b, :max(0, min(n, T))]]
        ok = (0 <= n <= T and 0 <= P and P + T <= cap[b]
              and ks[b] + P >= 0 and ks[b] + P + T <= pool.shape[0]
              and all(0 <= x < T for x in path))
        if not ok:
            bad += 1
            continue
        rows = [pool[ks[b] + P + x, :cols].copy() for x in path]
        for k, r in enumerate(rows):
            pool[ks[b] + P + k, :cols] = r
        new_pl[b] = P + n
    return pool, new_pl, bad
