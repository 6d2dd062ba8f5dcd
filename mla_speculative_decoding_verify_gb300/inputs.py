"""Seeded synthetic inputs for MLA tree-verify attention.

This module only builds inputs: it draws random values, rounds them to bf16,
shapes draft trees and lays the latent KV cache out in pages.  It holds none
of the attention arithmetic, so the CUDA path and the fp64 oracle can both
consume what it produces without sharing any of the method's code.

Five verify-attention workloads, shaped as the verify-kernel page describes
the problem (page "The Shared Memory Ceiling", sections "The Broader Context"
and "Technical Deep Dive": 64 heads, a 512-dim latent c_kv plus a 64-dim k_rope per KV row,
a draft tree of query tokens per request, prefixes up to 65,536 tokens).

Readings taken where the pages are silent:
  * values are N(0,1) drawn as float32 from numpy's PCG64 (ziggurat), then
    rounded to bf16 with round-to-nearest-even;
  * the tree tokens' own latents sit in the same paged cache right after the
    prefix, so ``seq_lens = prefix + n_tree``;
  * ``tree_parent`` holds request-local parents, -1 for a root, parent < i;
  * outlier rows (the 4 x 4096-token workload) scale the 512 c_kv dims by 8,
    not k_rope;
  * shared-prefix groups (the 64-request ragged workload) of 8 requests share
    the physical pages
    of their first floor(min_prefix / page) pages, with identical content;
  * unused cache rows (tail of a last page, unreferenced pages) and unused
    block-table slots are poisoned (NaN rows, -1 slots) so a read out of
    range shows up in the result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

NUM_HEADS = 64
D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE
PAGE = 64
BF16_NAN = np.uint16(0x7FC0)


def bf16_bits_from_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (round-to-nearest-even) and return the bits.

    Exact for every finite value in the normal bf16 range: the f64 mantissa is
    rounded to 7 bits in integer arithmetic, and the result (exactly
    representable in float32) is narrowed to its top 16 bits.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    keep = np.uint64(45)  # 52 - 7 mantissa bits dropped
    lsb = (b >> keep) & np.uint64(1)
    rounded = (b + (np.uint64((1 << 44) - 1) + lsb)) >> keep << keep
    f32 = rounded.view(np.float64).astype(np.float32)
    out = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even) and return the bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    out = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


@dataclasses.dataclass
class VerifyInputs:
    """One batch of verify-attention inputs, host side (bf16 kept as uint16 bits)."""

    name: str
    q_lat: np.ndarray        # uint16 [total_q, H, 512]
    q_rope: np.ndarray       # uint16 [total_q, H, 64]
    kv_cache: np.ndarray     # uint16 [num_pages, page_size, 576]  (c_kv | k_rope)
    block_table: np.ndarray  # int32  [B, max_pages_per_seq]
    seq_lens: np.ndarray     # int32  [B]   prefix + n_tree
    tree_parent: np.ndarray  # int32  [total_q] request-local parent, -1 = root
    n_tree: np.ndarray       # int32  [B]
    scale: float
    page_size: int
    unique_pages: int        # physical pages referenced by the block table

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.tree_parent.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.q_lat.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_tree(self) -> int:
        return int(self.n_tree.max()) if self.batch else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    @property
    def prefix_lens(self) -> np.ndarray:
        return (self.seq_lens - self.n_tree).astype(np.int64)

    @property
    def q_offsets(self) -> np.ndarray:
        off = np.zeros(self.batch + 1, dtype=np.int64)
        np.cumsum(self.n_tree, out=off[1:])
        return off

    def nbytes(self) -> int:
        return sum(a.nbytes for a in (self.q_lat, self.q_rope, self.kv_cache,
                                      self.block_table, self.seq_lens,
                                      self.tree_parent, self.n_tree))


def first_requests(inp: VerifyInputs, k: int) -> VerifyInputs:
    """The first k requests of `inp`, sharing its KV cache (same pages and block
    table rows): smaller batches of one cache, as a serving loop sees them."""
    k = int(k)
    nq = int(inp.q_offsets[k])
    return dataclasses.replace(
        inp, name=f"{inp.name}[:{k}]", q_lat=inp.q_lat[:nq], q_rope=inp.q_rope[:nq],
        block_table=inp.block_table[:k], seq_lens=inp.seq_lens[:k], tree_parent=inp.tree_parent[:nq],
        n_tree=inp.n_tree[:k])


# ---------------------------------------------------------------- draft trees

def _tree(kind: str, n: int, rng: np.random.Generator) -> np.ndarray:
    """Request-local parent array of one draft tree (parent[i] < i, -1 = root)."""
    par = np.full(n, -1, dtype=np.int32)
    if n == 0:
        return par
    if kind == "forest":            # parent[i] uniform in [-1, i)
        for i in range(n):
            par[i] = rng.integers(-1, i) if i > 0 else -1
        return par
    if kind == "chain":             # parent[i] = i - 1
        par[1:] = np.arange(n - 1, dtype=np.int32)
        return par
    if kind == "star":              # every node hangs off the root
        par[1:] = 0
        return par
    if kind == "roots":             # every node is its own root
        return par
    depth = np.zeros(n, dtype=np.int64)
    kids = np.zeros(n, dtype=np.int64)
    depth[0] = 1
    for i in range(1, n):
        if kind == "uniform":       # parent uniform in [0, i)
            cand = np.arange(i)
        elif kind.startswith("depth"):   # parent uniform over nodes of depth < D
            cap = int(kind[5:] or 6)
            cand = np.nonzero(depth[:i] < cap)[0]
        elif kind.startswith("branch"):  # parent uniform over nodes with < K children
            cap = int(kind[6:] or 4)
            cand = np.nonzero(kids[:i] < cap)[0]
        else:
            raise ValueError(f"unknown tree kind {kind!r}")
        p = int(cand[rng.integers(0, cand.size)])
        par[i] = p
        depth[i] = depth[p] + 1
        kids[p] += 1
    return par


# ---------------------------------------------------------------- generator

def make_inputs(prefix_lens: Sequence[int], tree_sizes: Sequence[int], *,
                tree_kind: str = "uniform", page_size: int = PAGE,
                seed: int = 0, stream: int = 0, shuffle: bool = True,
                outlier_frac: float = 0.0, outlier_scale: float = 8.0,
                share_group: int = 0, num_heads: int = NUM_HEADS,
                scale: Optional[float] = None, extra_pages: int = 2,
                poison: bool = True, q_zero: bool = False,
                trees: Optional[Sequence[Sequence[int]]] = None,
                name: str = "custom") -> VerifyInputs:
    """Build a batch: request b has ``prefix_lens[b]`` prefix tokens and a draft
    tree of ``tree_sizes[b]`` nodes whose latents follow the prefix in its pages.
    """
    B = len(prefix_lens)
    assert len(tree_sizes) == B
    ss = np.random.SeedSequence([int(stream), int(seed)])
    r_tree, r_kv, r_q, r_perm, r_out = (np.random.default_rng(s) for s in ss.spawn(5))
    prefix = np.asarray(prefix_lens, dtype=np.int64)
    ntree = np.asarray(tree_sizes, dtype=np.int64)
    seq = prefix + ntree
    if trees is not None:
        parents = [np.asarray(t, dtype=np.int32) for t in trees]
        assert [len(p) for p in parents] == list(ntree)
    else:
        parents = [_tree(tree_kind, int(n), r_tree) for n in ntree]
    tree_parent = (np.concatenate(parents) if B else np.zeros(0)).astype(np.int32)
    total_q = int(ntree.sum())
    pages_per = [(int(s) + page_size - 1) // page_size for s in seq]
    max_pages = max(pages_per) if B else 1
    max_pages = max(max_pages, 1)

    # shared-prefix groups: members reuse the leader's first pages
    shared = np.zeros(B, dtype=np.int64)
    leader = np.arange(B)
    if share_group and share_group > 1:
        for g0 in range(0, B, share_group):
            members = list(range(g0, min(B, g0 + share_group)))
            n_sh = int(prefix[members].min()) // page_size
            for m in members:
                leader[m] = g0
                shared[m] = n_sh if m != g0 else 0
    own_pages = [pages_per[b] - int(shared[b]) for b in range(B)]
    n_used = int(sum(own_pages))
    num_pages = n_used + int(extra_pages)
    phys = (r_perm.permutation(num_pages) if shuffle else np.arange(num_pages)).astype(np.int32)
    block_table = np.full((B, max_pages), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        if leader[b] != b:
            block_table[b, :shared[b]] = block_table[leader[b], :shared[b]]
        k = int(shared[b])
        block_table[b, k:pages_per[b]] = phys[cursor:cursor + own_pages[b]]
        cursor += own_pages[b]

    D = D_LATENT + D_ROPE
    kv = np.empty((num_pages, page_size, D), dtype=np.uint16)
    kv[...] = BF16_NAN if poison else np.uint16(0)
    for b in range(B):
        L = int(seq[b])
        vals = r_kv.standard_normal((L, D), dtype=np.float32)
        if outlier_frac > 0 and L > 0:
            n_out = int(math.floor(outlier_frac * L))
            if n_out:
                rows = r_out.choice(L, size=n_out, replace=False)
                vals[rows, :D_LATENT] *= np.float32(outlier_scale)
        bits = bf16_bits_from_f32(vals)
        for p in range(int(shared[b]), pages_per[b]):
            r0 = p * page_size
            r1 = min(L, r0 + page_size)
            kv[block_table[b, p], :r1 - r0] = bits[r0:r1]
        del vals, bits

    if q_zero:
        q_lat = np.zeros((total_q, num_heads, D_LATENT), dtype=np.uint16)
        q_rope = np.zeros((total_q, num_heads, D_ROPE), dtype=np.uint16)
    else:
        q_lat = bf16_bits_from_f32(r_q.standard_normal((total_q, num_heads, D_LATENT),
                                                       dtype=np.float32))
        q_rope = bf16_bits_from_f32(r_q.standard_normal((total_q, num_heads, D_ROPE),
                                                        dtype=np.float32))
    if scale is None:
        scale = 1.0 / math.sqrt(192.0)
    return VerifyInputs(name=name, q_lat=q_lat, q_rope=q_rope, kv_cache=kv,
                        block_table=block_table, seq_lens=seq.astype(np.int32),
                        tree_parent=tree_parent, n_tree=ntree.astype(np.int32),
                        scale=float(scale), page_size=int(page_size),
                        unique_pages=n_used)


# ---------------------------------------------------------------- the five workloads

CONFIG_NAMES = {
    1: "c1_b1_p256_t8_contig",
    2: "c2_b4_p4096_t16_outliers",
    3: "c3_b16_p16384_t32",
    4: "c4_b2_p65536_t64",
    5: "c5_b64_ragged_shared",
}


def config_shape(cfg: int, seed: int = 0):
    """(prefix_lens, tree_sizes, kwargs) of workload ``cfg`` (1..5)."""
    if cfg == 1:
        # one request, prefix 256, 8-node forest, contiguous KV (a single page)
        return [256], [8], dict(tree_kind="forest", page_size=320, shuffle=False)
    if cfg == 2:
        return [4096] * 4, [16] * 4, dict(tree_kind="depth6", outlier_frac=0.01)
    if cfg == 3:
        return [16384] * 16, [32] * 16, dict(tree_kind="uniform")
    if cfg == 4:
        return [65536] * 2, [64] * 2, dict(tree_kind="branch4")
    if cfg == 5:
        rng = np.random.default_rng(np.random.SeedSequence([5, int(seed), 99]))
        lo, hi = math.log(1024), math.log(32768)
        prefix = np.floor(np.exp(rng.uniform(lo, hi, size=64))).astype(np.int64)
        prefix = np.clip(prefix, 1024, 32768)
        trees = rng.choice(np.array([4, 8, 16, 32]), size=64)
        return prefix.tolist(), trees.tolist(), dict(tree_kind="uniform", share_group=8)
    raise ValueError(cfg)


def config_inputs(cfg: int, seed: int = 0, **overrides) -> VerifyInputs:
    prefix, trees, kw = config_shape(cfg, seed)
    kw.update(overrides)
    return make_inputs(prefix, trees, seed=seed, stream=cfg, name=CONFIG_NAMES[cfg], **kw)


def scaled_config_inputs(cfg: int, seed: int = 0, prefix_div: int = 16,
                         batch_cap: Optional[int] = None, **overrides) -> VerifyInputs:
    """A reduced copy of workload ``cfg`` (prefixes divided by ``prefix_div``,
    batch capped) with the same tree generator, paging and value recipe, small
    enough for the oracle to evaluate every output row in seconds."""
    prefix, trees, kw = config_shape(cfg, seed)
    prefix = [max(1, p // prefix_div) for p in prefix]
    if batch_cap is not None:
        prefix, trees = prefix[:batch_cap], trees[:batch_cap]
    kw.update(overrides)
    if cfg == 1:
        kw["page_size"] = max(64, ((prefix[0] + trees[0] + 63) // 64) * 64)
    return make_inputs(prefix, trees, seed=seed, stream=100 + cfg,
                       name=CONFIG_NAMES[cfg] + f"_div{prefix_div}", **kw)


def sample_rows(inp: VerifyInputs, n: int, seed: int = 1234) -> np.ndarray:
    """A seeded sample of global output rows (q_index * H + head), always
    including the first and last row of every request."""
    H = inp.num_heads
    total = inp.total_q * H
    rng = np.random.default_rng(seed)
    must = []
    off = inp.q_offsets
    for b in range(inp.batch):
        if inp.n_tree[b]:
            must += [int(off[b]) * H, int(off[b + 1]) * H - 1]
    pick = rng.choice(total, size=min(n, total), replace=False) if total else np.zeros(0)
    return np.unique(np.concatenate([np.asarray(must, dtype=np.int64),
                                     np.asarray(pick, dtype=np.int64)]))


def tree_rows(inp: VerifyInputs, seed: int = 0) -> np.ndarray:
    """Seeded latent rows for the draft tree tokens: bf16 bits [total_q, 576] drawn
    like the cache (N(0,1) rounded to bf16)."""
    rng = np.random.default_rng(seed)
    return bf16_bits_from_f32(rng.standard_normal((inp.total_q, 576), dtype=np.float32))


def accept_paths(inp: VerifyInputs, seed: int = 0):
    """Seeded accepted paths: per request a random node, its root-to-node path,
    cut at a random length (possibly 0).  Returns (accept_len int32 [batch],
    accept_idx int32 [total_q]) in the layout of tree_parent."""
    rng = np.random.default_rng(seed)
    off = inp.q_offsets
    acc_len = np.zeros(inp.batch, dtype=np.int32)
    acc_idx = np.full(inp.total_q, -1, dtype=np.int32)
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        if T == 0:
            continue
        par = inp.tree_parent[off[b]:off[b] + T]
        node, path = int(rng.integers(0, T)), []
        while node >= 0:
            path.append(node)
            node = int(par[node])
        path = path[::-1][: int(rng.integers(0, len(path) + 1))]
        acc_len[b] = len(path)
        acc_idx[off[b]:off[b] + len(path)] = path
    return acc_len, acc_idx


def topk_indices(inp: VerifyInputs, topk: int, seed: int = 0, unused_frac: float = 0.0,
                 duplicates: bool = False) -> np.ndarray:
    """Seeded top-k slot lists, int32 [total_q, topk]: per tree token, distinct
    prefix positions in random order (all of them, then -1, when the prefix is
    shorter than topk).  `unused_frac` of the slots become -1; `duplicates`
    repeats some listed positions in other slots."""
    rng = np.random.default_rng(seed)
    out = np.full((inp.total_q, topk), -1, dtype=np.int32)
    off = inp.q_offsets
    for b in range(inp.batch):
        P = int(inp.seq_lens[b] - inp.n_tree[b])
        for g in range(int(off[b]), int(off[b + 1])):
            if P <= 0:
                continue
            k = min(topk, P)
            pos = rng.choice(P, size=k, replace=False) if P > 4 * k else rng.permutation(P)[:k]
            row = np.full(topk, -1, dtype=np.int64)
            row[:k] = pos
            if duplicates and k > 1:
                n_dup = max(1, k // 8)
                row[rng.choice(topk, size=n_dup, replace=False)] = rng.choice(pos, size=n_dup)
            if unused_frac > 0:
                row[rng.random(topk) < unused_frac] = -1
            out[g] = rng.permutation(row)
    return out

