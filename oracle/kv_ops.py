"""Oracle for the paged-cache steps around tree verification (plain numpy).

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU legs use it; the
product path never imports it, and it shares no code with the CUDA library.

The verify-kernel page ("The Shared Memory Ceiling", section "The Broader
Context") places the draft tree's latents in the same paged KV cache that the
verify kernel reads, and names the step after verification a KV-cache
"defrag" of the accepted path; the pages give no further detail.  The reading
implemented here:

* append: the T_b tree tokens of request b (rows of 576 bf16 values, c_kv then
  k_rope, tokens back to back as in q) are written at KV positions
  P_b + i, i < T_b, with P_b = seq_len_b - T_b, through the block table;
* accept: the accepted tokens form a path from a root of the draft tree
  (``accept_idx`` holds, in each request's segment, ``accept_len[b]`` node
  indices in path order: the first has parent -1, each next one is a child
  of the one before).  Accepted node k's row moves to position P_b + k and the
  new sequence length is P_b + accept_len[b].  Every row is read before any
  row is written (a node's old position can be another node's new one).

Both leave a request untouched and report it in the status bits when its tree
or path is malformed (bit 1 << 6) or a block id it touches is out of range
(bit 1 << 7).  A request's rows of the per-token arrays (tree_kv, tree_parent,
accept_idx, all [total_q, ...]) start at the sum of the earlier counts, a
negative count taken as 0; a request whose rows would reach past total_q is
malformed too (a reading: the pages define no error contract, and this one
never reads outside the arrays).  Rows are moved as raw 16-bit patterns: the
results are exact.
"""
from __future__ import annotations

import numpy as np

D_KV = 576
MAX_TREE = 64
STATUS_BAD_TREE = 1 << 6
STATUS_BAD_BLOCK = 1 << 7


def _offsets(n_tree):
    """First tree token of each request: the running sum of the counts, a negative
    count taken as 0 (such a request is itself rejected as malformed)."""
    n_tree = np.maximum(np.asarray(n_tree, dtype=np.int64), 0)
    return np.concatenate([[0], np.cumsum(n_tree)]).astype(np.int64)


def _row(block_table, b, pos, page_size, num_pages):
    """Cache row of KV position `pos` of request b, or None if its block id is out of range."""
    page_idx = pos // page_size
    if page_idx >= block_table.shape[1]:
        return None
    page = int(block_table[b, page_idx])
    if page < 0 or page >= num_pages:
        return None
    return page * page_size + pos % page_size


def _tree_ok(parent, T):
    return all(-1 <= int(parent[i]) < i for i in range(T))


def tree_kv_append(kv_cache, block_table, seq_lens, n_tree, tree_kv, page_size):
    """Returns (new cache [num_pages, page_size, 576] uint16, status bits)."""
    cache = np.array(kv_cache, dtype=np.uint16, copy=True)
    num_pages = cache.shape[0]
    flat = cache.reshape(num_pages * page_size, D_KV)
    tree_kv = np.asarray(tree_kv, dtype=np.uint16).reshape(-1, D_KV)
    total_q = tree_kv.shape[0]
    off = _offsets(n_tree)
    status = 0
    for b in range(len(seq_lens)):
        T, L = int(n_tree[b]), int(seq_lens[b])
        if T < 0 or T > MAX_TREE or T > L or off[b] + T > total_q:
            status |= STATUS_BAD_TREE
            continue
        P = L - T
        rows = [_row(block_table, b, P + i, page_size, num_pages) for i in range(T)]
        if any(r is None for r in rows):
            status |= STATUS_BAD_BLOCK
            continue
        for i, r in enumerate(rows):
            flat[r] = tree_kv[off[b] + i]
    return cache, status


def tree_kv_accept(kv_cache, block_table, seq_lens, n_tree, tree_parent, accept_len, accept_idx, page_size):
    """Returns (new cache, new_seq_lens int32 [batch], status bits)."""
    cache = np.array(kv_cache, dtype=np.uint16, copy=True)
    num_pages = cache.shape[0]
    flat = cache.reshape(num_pages * page_size, D_KV)
    off = _offsets(n_tree)
    total_q = len(tree_parent)
    new_lens = np.array(seq_lens, dtype=np.int32, copy=True)
    status = 0
    for b in range(len(seq_lens)):
        T, L, A = int(n_tree[b]), int(seq_lens[b]), int(accept_len[b])
        if T < 0 or T > MAX_TREE or T > L or off[b] + T > total_q:
            status |= STATUS_BAD_TREE
            continue
        P = L - T
        parent = [int(v) for v in tree_parent[off[b]:off[b] + T]]
        path = [int(v) for v in accept_idx[off[b]:off[b] + max(A, 0)]]
        ok = _tree_ok(parent, T) and 0 <= A <= T and all(0 <= v < T for v in path)
        if ok:
            for k, v in enumerate(path):
                if parent[v] != (path[k - 1] if k > 0 else -1):
                    ok = False
        if not ok:
            status |= STATUS_BAD_TREE
            continue
        rows = [_row(block_table, b, P + i, page_size, num_pages) for i in range(T)]
        if any(r is None for r in rows):
            status |= STATUS_BAD_BLOCK
            continue
        moved = [flat[rows[v]].copy() for v in path]      # read every accepted row first
        for k, data in enumerate(moved):
            flat[rows[k]] = data
        new_lens[b] = P + A
    return cache, new_lens, status
