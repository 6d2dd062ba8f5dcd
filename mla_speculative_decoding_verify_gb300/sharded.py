"""Split-KV across GPUs: one long request's prefix sharded over ranks.

The verify path shards over requests and row tiles with no exchange at all
(independent replicas).  A single long request is the exception: its KV cache
can be divided along the key axis, each GPU holding and attending only its
share of the pages, after which the GPUs exchange their partial results once
and merge them by log-sum-exp weights -- the flash-decoding split of the
single-GPU path stretched across devices (one process per GPU).

  rank r of W with k splits per rank computes splits r*k .. r*k + k - 1 of W*k
  (mla_verify_attn_split_range); every rank all-gathers the W*k partials
  (o_s fp32 [rows, 512], lse_s fp32 [rows]) and merges them with
  mla_split_combine.

Split s of S covers KV tiles [n*s // S, n*(s+1) // S) of a request of n tiles
(64 keys each), the partition the kernel uses, so the tree's own keys fall in
the last split only.  A rank needs the pages under its tiles and nothing else;
``shard_inputs`` builds such a local cache (pages renumbered, positions outside
the rank's tiles pointed at local page 0, which the kernel never reads there).

The exchange goes through torch.distributed (NCCL on GPUs, gloo on the host in
the tests); nothing else in the path is collective.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Tuple

import numpy as np

BLOCK_N = 64      # keys per KV tile of the verify kernel


def split_tiles(n_tiles: int, s: int, num_splits: int) -> Tuple[int, int]:
    """KV tiles [t0, t1) that split s of num_splits covers (equal shares, integer division)."""
    return (n_tiles * s) // num_splits, (n_tiles * (s + 1)) // num_splits


def rank_splits(world: int, rank: int, per_rank: int = 1) -> Tuple[int, int, int]:
    """(num_splits, split_begin, split_count) of rank `rank` of `world`."""
    if world < 1 or not 0 <= rank < world or per_rank < 1:
        raise ValueError("bad rank layout")
    return world * per_rank, rank * per_rank, per_rank


def rank_key_ranges(seq_lens, num_splits: int, begin: int, count: int) -> List[Tuple[int, int]]:
    """Per request, the KV positions [k0, k1) the splits begin .. begin + count - 1 cover."""
    out = []
    for L in np.asarray(seq_lens, dtype=np.int64):
        n = (int(L) + BLOCK_N - 1) // BLOCK_N
        t0 = split_tiles(n, begin, num_splits)[0]
        t1 = split_tiles(n, begin + count - 1, num_splits)[1]
        out.append((min(t0 * BLOCK_N, int(L)), min(t1 * BLOCK_N, int(L))))
    return out


def rank_pages(block_table, seq_lens, page_size: int, num_splits: int, begin: int, count: int) -> List[List[int]]:
    """Per request, the (global) page ids under the rank's KV positions, in position order."""
    pages = []
    for b, (k0, k1) in enumerate(rank_key_ranges(seq_lens, num_splits, begin, count)):
        if k1 <= k0:
            pages.append([])
            continue
        idx = range(k0 // page_size, (k1 - 1) // page_size + 1)
        pages.append([int(block_table[b, i]) for i in idx])
    return pages


def shard_inputs(inp, num_splits: int, begin: int, count: int):
    """A copy of `inp` holding only the pages a rank reads: the local cache has
    the needed pages (each once, renumbered in first-use order) and the local
    block table maps the rank's positions to them; every other position names
    local page 0 (valid, never read by the rank's splits)."""
    ps = inp.page_size
    need = rank_pages(inp.block_table, inp.seq_lens, ps, num_splits, begin, count)
    local_id = {}
    for plist in need:
        for g in plist:
            local_id.setdefault(g, len(local_id))
    order = sorted(local_id, key=local_id.get)
    n_local = max(1, len(order))
    cache = np.zeros((n_local,) + inp.kv_cache.shape[1:], dtype=inp.kv_cache.dtype)
    if order:
        cache[: len(order)] = inp.kv_cache[np.array(order)]
    table = np.zeros_like(inp.block_table)
    for b, (k0, k1) in enumerate(rank_key_ranges(inp.seq_lens, num_splits, begin, count)):
        if k1 <= k0:
            continue
        for i in range(k0 // ps, (k1 - 1) // ps + 1):
            table[b, i] = local_id[int(inp.block_table[b, i])]
    return dataclasses.replace(inp, kv_cache=cache, block_table=table, unique_pages=len(order),
                               name=f"{inp.name}_shard{begin}of{num_splits}")


def all_gather_partials(part_out, part_lse, group=None):
    """Concatenate every rank's partials along the split axis (rank order):
    part_out [k, rows, 512] and part_lse [k, rows] per rank -> [W*k, ...]."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    if world == 1:
        return part_out, part_lse
    outs = [torch.empty_like(part_out) for _ in range(world)]
    lses = [torch.empty_like(part_lse) for _ in range(world)]
    dist.all_gather(outs, part_out.contiguous(), group=group)
    dist.all_gather(lses, part_lse.contiguous(), group=group)
    return torch.cat(outs, 0), torch.cat(lses, 0)


def verify_sharded(db_local, world: int, rank: int, per_rank: int = 1, group=None,
                   exchange: Callable = all_gather_partials, stream=None):
    """This rank's share of the verify attention of db_local (a DeviceBatch of
    ``shard_inputs``), one exchange, and the merge on this GPU.  Returns
    (out [total_q, 64, 512], lse [total_q, 64], workspace) -- the same result on
    every rank."""
    import torch

    from . import binding
    inp = db_local.inp
    S, b0, k = rank_splits(world, rank, per_rank)
    part_out, part_lse, ws = binding.verify_split_range(db_local, S, b0, k, stream=stream)
    all_out, all_lse = exchange(part_out, part_lse, group)
    rows = inp.total_q * inp.num_heads
    out = torch.empty((inp.total_q, inp.num_heads, binding.D_LATENT), dtype=torch.float32, device=db_local.device)
    lse = torch.empty((inp.total_q, inp.num_heads), dtype=torch.float32, device=db_local.device)
    if stream is None:
        stream = torch.cuda.current_stream(db_local.device)
    binding.check(binding.split_combine(all_out.data_ptr(), all_lse.data_ptr(), S, rows, out.data_ptr(),
                                        lse.data_ptr(), stream.cuda_stream), "mla_split_combine")
    return out, lse, ws
