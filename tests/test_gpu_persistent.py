"""GPU parity of the persistent schedule (num_splits = MLA_SPLITS_PERSISTENT,
through the C ABI) against the fp64 oracle.

A fixed grid of CTA pairs: rounds of whole work items, one per pair, then the
rest of the (work item, KV tile) positions shared out evenly; items cut between
pairs are merged in the kernel by the last of their pieces.  The cases below
cover items in one piece and in many, whole rounds followed by a shared tail,
shares that start and end inside items, requests without tree tokens and
invalid requests (their rows out = 0, lse = -inf), the sparse variant, graph
replay, the automatic choice of the schedule, and the full workload sizes on
sampled rows."""
import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import assert_close, ensure_gpu, run_gpu

pytestmark = pytest.mark.gpu
PERSISTENT = binding.SPLITS_PERSISTENT
SCALED = [(1, 1, None), (2, 4, None), (3, 16, 4), (4, 64, None), (5, 16, 16)]


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("cfg,div,cap", SCALED, ids=[f"c{c[0]}" for c in SCALED])
def test_persistent_scaled_workloads(cfg, div, cap, seed):
    inp = I.scaled_config_inputs(cfg, seed=seed, prefix_div=div, batch_cap=cap)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"persistent cfg{cfg} seed{seed}")


@pytest.mark.parametrize("prefixes,trees", [
    ([4000, 3000, 5000], [8, 4, 6]),          # 9 long items on 76 pairs: each cut into many pieces
    ([16000], [2]),                           # one item over every pair
    ([9000, 64, 1, 2500], [64, 3, 1, 33]),    # one long request, short and one-key ones
])
def test_persistent_items_cut_into_many_pieces(prefixes, trees):
    inp = I.make_inputs(prefixes, trees, tree_kind="uniform", seed=len(prefixes), stream=970)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"persistent {prefixes}")


@pytest.mark.parametrize("n_req,tree", [(10, 20), (12, 32), (40, 8)])
def test_persistent_whole_rounds_then_shared_tail(n_req, tree):
    """More items than CTA pairs: whole items round by round (snake order), then
    the last, partial round shared out and merged.  Ragged prefixes."""
    rng = np.random.default_rng(n_req)
    prefixes = [int(v) for v in rng.integers(100, 1500, size=n_req)]
    inp = I.make_inputs(prefixes, [tree] * n_req, tree_kind="uniform", seed=n_req, stream=975)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"persistent rounds {n_req} x {tree}")
    o2, l2, _ = run_gpu(inp, splits=PERSISTENT)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


@pytest.mark.parametrize("prefix", [0, 1, 63, 64, 65, 129])
@pytest.mark.parametrize("kind", ["forest", "chain"])
def test_persistent_edge_prefix_and_trees(prefix, kind):
    trees = [1, 2, 3, 7, 33, 64]
    inp = I.make_inputs([prefix] * len(trees), trees, tree_kind=kind, seed=prefix, stream=971)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"persistent prefix={prefix} kind={kind}")


def test_persistent_requests_without_tree_tokens():
    inp = I.make_inputs([100, 5000, 64, 0, 7000], [5, 0, 3, 0, 9], tree_kind="uniform", seed=8, stream=972)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, "persistent, empty trees")


def test_persistent_is_bitwise_repeatable():
    """The merge sums the pieces in piece order: the arrival order does not show."""
    inp = I.make_inputs([4000, 3000, 5000], [8, 4, 6], tree_kind="uniform", seed=3, stream=973)
    o1, l1, _ = run_gpu(inp, splits=PERSISTENT)
    for _ in range(3):
        o2, l2, _ = run_gpu(inp, splits=PERSISTENT)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_persistent_invalid_requests_zeroed():
    """A bad block id in a long request (its item cut into pieces) and a bad tree
    in a short one: status bits, their rows 0 / -inf, the others match the oracle."""
    inp = I.make_inputs([6000, 300, 5000], [4, 6, 3], tree_kind="uniform", seed=5, stream=974)
    ref_o, ref_l = oracle.verify(inp)
    inp.block_table = inp.block_table.copy()
    inp.block_table[0, 7] = inp.num_pages + 3
    inp.tree_parent = inp.tree_parent.copy()
    inp.tree_parent[4 + 2] = 4                 # request 1, node 2: parent not earlier
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status & (1 << binding.MLA_ERR_BAD_BLOCK) and status & (1 << binding.MLA_ERR_BAD_TREE)
    assert not out[:10].any() and np.isneginf(lse[:10]).all()
    assert_close(out[10:], lse[10:], ref_o[10:], ref_l[10:], "valid request next to invalid ones")


def test_persistent_invalid_request_in_a_whole_round():
    """40 requests x 8 tree tokens (160 items: two whole rounds, then a shared
    tail); request 3's block table names a page outside the cache, so its items,
    in the first whole round, carry no tiles and its rows are written as 0 / -inf."""
    rng = np.random.default_rng(77)
    prefixes = [int(v) for v in rng.integers(200, 900, size=40)]
    inp = I.make_inputs(prefixes, [8] * 40, tree_kind="uniform", seed=77, stream=977)
    rows = I.sample_rows(inp, 600, seed=77)
    ref_o, ref_l = oracle.verify_rows(inp, rows)
    inp.block_table = inp.block_table.copy()
    inp.block_table[3, 2] = inp.num_pages + 1
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status & (1 << binding.MLA_ERR_BAD_BLOCK)
    bad = slice(int(inp.q_offsets[3]), int(inp.q_offsets[4]))
    assert not out[bad].any() and np.isneginf(lse[bad]).all()
    flat_tok = rows // inp.num_heads
    keep = (flat_tok < bad.start) | (flat_tok >= bad.stop)
    assert_close(out.reshape(-1, 512)[rows[keep]], lse.reshape(-1)[rows[keep]], ref_o[keep], ref_l[keep],
                 "valid requests next to an invalid one in a whole round")


@pytest.mark.parametrize("topk", [100, 512])
def test_persistent_sparse(topk):
    inp = I.scaled_config_inputs(3, seed=1, prefix_div=16, batch_cap=4)
    idx = I.topk_indices(inp, topk, seed=topk, unused_frac=0.1, duplicates=True)
    ref_o, ref_l = oracle.verify_sparse(inp, idx)
    import torch
    ensure_gpu()
    db = binding.DeviceBatch(inp, "cuda:0")
    t = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to("cuda:0")
    out, lse, ws = binding.verify_sparse(db, t, num_splits_req=PERSISTENT)
    torch.cuda.synchronize()
    assert binding.read_status(ws.data_ptr()) == 0
    assert_close(out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_o, ref_l,
                 f"persistent sparse topk={topk}")


def test_persistent_graph_replay_matches_eager_bitwise():
    """The shares are cut on the device from the requests of each replay, over
    every CTA pair of the device, so a padded replay equals the eager call."""
    import torch
    from test_gpu_graph import bucket_inputs, eager, make_graph, replay
    full = bucket_inputs()
    g = make_graph(full, PERSISTENT)
    try:
        for k in (6, 4, 1, 6):
            sub = I.first_requests(full, k)
            o, l, st = replay(g, sub)
            assert st == 0, (k, st)
            eo, el = eager(sub, PERSISTENT)
            assert torch.equal(o, eo) and torch.equal(l, el), f"batch {k}: replay differs from eager"
        ref_o, ref_l = oracle.verify(sub)
        assert_close(o.numpy().astype(np.float64), l.numpy().astype(np.float64), ref_o, ref_l, "persistent replay")
        # a fully padded replay (no work items, no shares) is a no-op with status 0
        g.launch(0)
        torch.cuda.synchronize()
        assert binding.read_status(g.workspace.data_ptr()) == 0
    finally:
        g.close()


def test_persistent_sparse_graph_replay_matches_eager_bitwise():
    import torch
    from test_gpu_graph import bucket_inputs, eager, make_graph, replay
    full = bucket_inputs(kind="forest")
    idx = I.topk_indices(full, 100, seed=5, unused_frac=0.1, duplicates=True)
    g = make_graph(full, PERSISTENT, topk=100)
    try:
        for k in (6, 3):
            sub = I.first_requests(full, k)
            sidx = idx[:sub.total_q]
            o, l, st = replay(g, sub, sidx)
            assert st == 0
            eo, el = eager(sub, PERSISTENT, sidx)
            assert torch.equal(o, eo) and torch.equal(l, el), f"sparse batch {k}"
        ref_o, ref_l = oracle.verify_sparse(sub, sidx)
        assert_close(o.numpy().astype(np.float64), l.numpy().astype(np.float64), ref_o, ref_l,
                     "persistent sparse replay")
    finally:
        g.close()


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_persistent_full_size_sampled_rows(cfg):
    inp = I.config_inputs(cfg, seed=0)
    out, lse, status = run_gpu(inp, splits=PERSISTENT)
    assert status == 0
    rows = I.sample_rows(inp, 160, seed=cfg)
    ref_o, ref_l = oracle.verify_rows(inp, rows)
    got_o = out.reshape(-1, out.shape[-1])[rows]
    got_l = lse.reshape(-1)[rows]
    assert_close(got_o, got_l, ref_o, ref_l, f"cfg{cfg} full, persistent")
    assert np.isfinite(out).all()


def test_automatic_choice_takes_persistent_on_a_short_last_round():
    """12 requests x 16 tree tokens x 8192: 96 work items on 76 CTA pairs.  The
    per-unit grid would leave a last round of 20 items; the automatic choice
    takes the persistent schedule (split count 0), and it matches the oracle."""
    inp = I.make_inputs([8192] * 12, [16] * 12, tree_kind="uniform", seed=6, stream=976)
    ensure_gpu()
    assert binding.num_splits(inp.batch, inp.total_q, inp.max_tree, inp.max_seq_len) == 0
    out, lse, status = run_gpu(inp, splits=0)
    assert status == 0
    rows = I.sample_rows(inp, 400, seed=6)
    ref_o, ref_l = oracle.verify_rows(inp, rows)
    assert_close(out.reshape(-1, 512)[rows], lse.reshape(-1)[rows], ref_o, ref_l, "automatic persistent")
    o2, l2, _ = run_gpu(inp, splits=PERSISTENT)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)
