"""GPU tests of the replayable verify step (mla_verify_graph_*, through the C
ABI): a graph captured for a bucket of requests, replayed for smaller batches
padded up to it, must give exactly what the eager call gives on the same
requests, and match the fp64 oracle."""
import dataclasses

import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import assert_close, ensure_gpu

pytestmark = pytest.mark.gpu

PREFIXES = [700, 130, 64, 1000, 333, 2048]
TREES = [9, 33, 4, 16, 1, 64]


def bucket_inputs(seed=21, kind="uniform"):
    return I.make_inputs(PREFIXES, TREES, seed=seed, tree_kind=kind, stream=503)


def make_graph(full, splits, topk=0):
    import torch
    ensure_gpu()
    kv = binding.DeviceBatch(full, "cuda:0").kv_cache
    g = binding.VerifyGraph(kv, full.batch, full.total_q, full.max_tree, full.max_seq_len, full.page_size,
                            full.max_pages_per_seq, full.scale, topk=topk, num_splits_req=splits,
                            stream=torch.cuda.current_stream())
    return g


def eager(inp, splits, topk_idx=None):
    import torch
    db = binding.DeviceBatch(inp, "cuda:0")
    if topk_idx is None:
        out, lse, ws = binding.verify(db, splits)
    else:
        t = torch.from_numpy(np.ascontiguousarray(topk_idx)).to("cuda:0")
        out, lse, ws = binding.verify_sparse(db, t, splits)
    torch.cuda.synchronize()
    assert binding.read_status(ws.data_ptr()) == 0
    return out.cpu(), lse.cpu()


def replay(g, inp, topk_idx=None):
    import torch
    g.load(inp, topk_idx)
    g.out.fill_(float("nan"))
    g.launch()
    torch.cuda.synchronize()
    return g.out[:inp.total_q].cpu(), g.lse[:inp.total_q].cpu(), binding.read_status(g.workspace.data_ptr())


@pytest.mark.parametrize("splits", [1, 3])
def test_graph_bucket_padding_matches_eager_bitwise(splits):
    """Batches 6, 4, 1 and 6 again through one graph captured for 6 requests:
    the padded requests add nothing and the real ones are bit-identical to eager."""
    import torch
    full = bucket_inputs()
    g = make_graph(full, splits)
    try:
        for k in (6, 4, 1, 6):
            sub = I.first_requests(full, k)
            o, l, st = replay(g, sub)
            assert st == 0, (k, st)
            eo, el = eager(sub, splits)
            assert torch.equal(o, eo) and torch.equal(l, el), f"batch {k}: replay differs from eager"
    finally:
        g.close()


def test_graph_replay_matches_oracle_and_reads_new_inputs():
    """A replay reads the buffers at replay time: new queries give the oracle's new result."""
    full = bucket_inputs()
    other = bucket_inputs(seed=22)
    g = make_graph(full, 2)
    try:
        for tag, inp in (("first", I.first_requests(full, 4)),
                         ("new queries", dataclasses.replace(I.first_requests(full, 4),
                                                             q_lat=other.q_lat[:full.q_offsets[4]],
                                                             q_rope=other.q_rope[:full.q_offsets[4]]))):
            o, l, st = replay(g, inp)
            assert st == 0
            ref_o, ref_l = oracle.verify(inp)
            assert_close(o.numpy().astype(np.float64), l.numpy().astype(np.float64), ref_o, ref_l, tag)
    finally:
        g.close()


def test_graph_sparse_bucket_matches_eager_bitwise():
    import torch
    full = bucket_inputs(kind="forest")
    idx = I.topk_indices(full, 100, seed=5, unused_frac=0.1, duplicates=True)
    # three splits: with two, the split point follows the launch's sizes (bucket vs batch)
    g = make_graph(full, 3, topk=100)
    try:
        for k in (6, 3):
            sub = I.first_requests(full, k)
            sidx = idx[:sub.total_q]
            o, l, st = replay(g, sub, sidx)
            assert st == 0
            eo, el = eager(sub, 3, sidx)
            assert torch.equal(o, eo) and torch.equal(l, el), f"sparse batch {k}"
        ref_o, ref_l = oracle.verify_sparse(sub, sidx)
        assert_close(o.numpy().astype(np.float64), l.numpy().astype(np.float64), ref_o, ref_l, "sparse replay")
    finally:
        g.close()


def test_graph_status_is_per_replay():
    """A malformed step sets its status bit; the next good step reads 0 again."""
    full = bucket_inputs()
    g = make_graph(full, 1)
    try:
        sub = I.first_requests(full, 3)
        bad_parent = sub.tree_parent.copy()
        bad_parent[sub.q_offsets[1] + 2] = 5          # parent after its child
        _, _, st = replay(g, dataclasses.replace(sub, tree_parent=bad_parent))
        assert st & (1 << binding.MLA_ERR_BAD_TREE)
        _, _, st = replay(g, sub)
        assert st == 0
    finally:
        g.close()


def test_graph_launch_host_checks():
    full = bucket_inputs()
    g = make_graph(full, 1)
    try:
        import torch
        s = torch.cuda.current_stream().cuda_stream
        assert binding.verify_graph_launch(g.handle, full.batch + 1, s) == binding.MLA_ERR_INVALID_ARG
        assert binding.verify_graph_launch(g.handle, -1, s) == binding.MLA_ERR_INVALID_ARG
        assert binding.verify_graph_launch(g.handle, 0, s) == binding.MLA_OK   # every request padded
        torch.cuda.synchronize()
        assert binding.read_status(g.workspace.data_ptr()) == 0
    finally:
        g.close()


def test_graph_auto_splits_tail_cut_matches_oracle():
    """Automatic splits on a one-round bucket: its work items are cut in two and
    merged in the kernel; smaller replays cut at most the items they have."""
    import torch
    full = I.make_inputs([1500, 900, 1200, 800], [16, 8, 32, 4], seed=31, tree_kind="uniform", stream=504)
    assert binding.num_splits(full.batch, full.total_q, full.max_tree, full.max_seq_len) == 1
    g = make_graph(full, 0)
    try:
        for k in (4, 2, 1):
            sub = I.first_requests(full, k)
            o, l, st = replay(g, sub)
            assert st == 0
            ref_o, ref_l = oracle.verify(sub)
            assert_close(o.numpy().astype(np.float64), l.numpy().astype(np.float64), ref_o, ref_l, f"batch {k}")
        eo, el = eager(full, 0)
        o, l, _ = replay(g, full)
        assert torch.equal(o, eo) and torch.equal(l, el), "same shape: replay equals eager"
    finally:
        g.close()
