"""Work and traffic counts of a verify batch (for throughput and roofline figures).

Algorithmic work is what the method must do, not what a dense kernel would:
per (row, visible key) 2*576 flops for q.k and 2*512 for p*v; masked tree
pairs are not counted.  KV bytes count each request's rows once (logical) or
each physical page once (unique; shared prefix pages counted once).
"""
from __future__ import annotations

import hashlib
import os
import re

import numpy as np

FLOPS_PER_ROW_KEY = 2 * (512 + 64) + 2 * 512
KV_ROW_BYTES = (512 + 64) * 2


def visible_tree_pairs(parent: np.ndarray) -> int:
    """Number of (node, ancestor-or-self) pairs of one draft tree."""
    depth = np.zeros(len(parent), dtype=np.int64)
    for i, p in enumerate(parent):
        depth[i] = 1 + (depth[p] if p >= 0 else 0)
    return int(depth.sum())


def algorithmic_flops(inp) -> int:
    total = 0
    off = 0
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        P = int(inp.seq_lens[b]) - T
        total += inp.num_heads * FLOPS_PER_ROW_KEY * (T * P + visible_tree_pairs(inp.tree_parent[off:off + T]))
        off += T
    return int(total)


def sparse_visible_keys(inp, topk_idx: np.ndarray) -> int:
    """Sum over tree tokens of their visible keys in the sparse variant: listed
    slots plus ancestor-or-self tree tokens."""
    total = int((np.asarray(topk_idx) >= 0).sum())
    off = 0
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        total += visible_tree_pairs(inp.tree_parent[off:off + T])
        off += T
    return total


def sparse_flops(inp, topk_idx: np.ndarray) -> int:
    return int(inp.num_heads * FLOPS_PER_ROW_KEY * sparse_visible_keys(inp, topk_idx))


def sparse_kv_bytes(inp, topk_idx: np.ndarray) -> int:
    """KV rows the sparse variant must read: each visible key once per tree token."""
    return int(sparse_visible_keys(inp, topk_idx) * KV_ROW_BYTES)


def kv_bytes(inp, unique: bool = False) -> int:
    if not unique:
        return int(inp.seq_lens.astype(np.int64).sum()) * KV_ROW_BYTES
    pages = set()
    for b in range(inp.batch):
        n = (int(inp.seq_lens[b]) + inp.page_size - 1) // inp.page_size
        pages.update(int(p) for p in inp.block_table[b, :n])
    return len(pages) * inp.page_size * KV_ROW_BYTES


def io_bytes(inp) -> dict:
    """Bytes of the call's inputs (host -> device) and outputs (device -> host)."""
    inputs = sum(a.nbytes for a in (inp.q_lat, inp.q_rope, inp.kv_cache, inp.block_table,
                                    inp.seq_lens, inp.tree_parent, inp.n_tree))
    outputs = inp.total_q * inp.num_heads * (512 + 1) * 4
    return {"h2d": int(inputs), "d2h": int(outputs)}


VERIFY_KERNEL_SOURCES = ("sm103_ptx.cuh", "verify_kernel.cuh")


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed (string
    literals in these files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(files=VERIFY_KERNEL_SOURCES) -> str:
    """Hash of the code the fused verify kernel is compiled from (comments and
    layout ignored); profile figures taken on other code are stale."""
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc")
    h = hashlib.sha256()
    for name in sorted(files):
        with open(os.path.join(here, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]
