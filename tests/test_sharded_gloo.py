"""Split-KV across ranks (mla_speculative_decoding_verify_gb300/sharded.py) on the
host: the partition of a request's KV tiles into splits, the per-rank page
shards, and the one exchange of partials, run as two gloo ranks (world size 2).

Each rank computes its partials with the fp64 oracle on its OWN shard (the
local cache and block table shard_inputs builds, restricted to its keys), the
ranks exchange them with all_gather_partials, and the merge of the gathered
partials must equal the unsplit result of the whole cache to 1e-12.  On the
GPU the same orchestration runs the CUDA kernels (tests/test_gpu_sharded.py).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from mla_speculative_decoding_verify_gb300 import inputs as I
from mla_speculative_decoding_verify_gb300 import sharded as SH

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_splits_partition_every_request_and_keep_the_tree_in_the_last():
    for n in (1, 2, 5, 64, 257, 1025):
        for S in (1, 2, 3, 7, 16):
            spans = [SH.split_tiles(n, s, S) for s in range(S)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))     # contiguous, disjoint
            assert all(t0 <= t1 for t0, t1 in spans)
    # keys: the tree's own keys (the last n_tree positions) lie in the last split
    inp = I.make_inputs([1000, 64, 3000], [9, 32, 1], tree_kind="forest", seed=41, stream=970)
    S = 4
    for s in range(S):
        for (k0, k1), L, T in zip(SH.rank_key_ranges(inp.seq_lens, S, s, 1), inp.seq_lens, inp.n_tree):
            if s < S - 1:
                assert k1 <= L - T or k1 == k0
            else:
                assert k1 == L
    assert SH.rank_splits(4, 2, 3) == (12, 6, 3)
    with pytest.raises(ValueError):
        SH.rank_splits(2, 2)


@pytest.mark.parametrize("world,per_rank", [(2, 1), (3, 2), (4, 1)])
def test_shard_holds_exactly_the_pages_of_its_keys(world, per_rank):
    inp = I.make_inputs([5000, 130, 900], [16, 3, 64], tree_kind="uniform", seed=42, stream=971)
    ps = inp.page_size
    covered = np.zeros(inp.num_pages, dtype=bool)
    for r in range(world):
        S, b0, k = SH.rank_splits(world, r, per_rank)
        loc = SH.shard_inputs(inp, S, b0, k)
        ranges = SH.rank_key_ranges(inp.seq_lens, S, b0, k)
        needed = {int(inp.block_table[b, t // ps]) for b, (k0, k1) in enumerate(ranges) for t in range(k0, k1)}
        assert loc.unique_pages == len(needed) and loc.num_pages == max(1, len(needed))
        for b, (k0, k1) in enumerate(ranges):
            for t in range(k0, k1):
                g = inp.kv_cache[inp.block_table[b, t // ps], t % ps]
                l_ = loc.kv_cache[loc.block_table[b, t // ps], t % ps]
                assert np.array_equal(g, l_)
            covered[[int(inp.block_table[b, t // ps]) for t in range(k0, k1)]] = True
        assert (loc.block_table >= 0).all() and (loc.block_table < loc.num_pages).all()
    referenced = {int(inp.block_table[b, i]) for b in range(inp.batch)
                  for i in range((int(inp.seq_lens[b]) + ps - 1) // ps)}
    assert set(np.flatnonzero(covered)) == referenced     # the shards cover every used page


def _rank_body(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = I.make_inputs([4000], [16], tree_kind="branch4", seed=43, stream=972)   # one long request
        S, b0, k = SH.rank_splits(world, rank, 1)
        loc = SH.shard_inputs(inp, S, b0, k)
        (k0, k1), = SH.rank_key_ranges(inp.seq_lens, S, b0, k)
        o, l = oracle.verify_rows(loc, None, key_range=(k0, k1))          # this rank's shard only
        po = torch.from_numpy(o.reshape(1, *o.shape))
        pl = torch.from_numpy(l.reshape(1, -1))
        all_o, all_l = SH.all_gather_partials(po, pl)
        out, lse = oracle.combine(all_o.numpy(), all_l.numpy())
        if rank == 0:
            ref_o, ref_l = oracle.verify_rows(inp, None)
            q.put((float(np.abs(out - ref_o).max()), float(np.abs(lse - ref_l).max()), tuple(all_o.shape)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_merge_to_the_unsplit_result():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_body, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    err_o, err_l, shape = q.get(timeout=5)
    assert shape[0] == 2
    assert err_o < 1e-12 and err_l < 1e-12, (err_o, err_l)
