"""GPU parity of the paged-cache steps (mla_tree_kv_append / mla_tree_kv_accept,
through the C ABI) against the numpy oracle: the caches must match bit for bit."""
import json
import os

import numpy as np
import pytest

from oracle import kv_ops as K
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import ensure_gpu

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_kv_accept.json")


def rand_rows(n, seed):
    return np.random.default_rng(seed).integers(0, 1 << 16, size=(n, K.D_KV), dtype=np.uint16)


def random_paths(inp, seed):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(inp.n_tree)])
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


def gpu_append(inp, rows):
    import torch
    ensure_gpu()
    db = binding.DeviceBatch(inp, "cuda:0")
    t = torch.from_numpy(np.ascontiguousarray(rows).view(np.int16)).to("cuda:0")
    ws = binding.append_tree(db, t)
    torch.cuda.synchronize()
    return db.kv_cache.cpu().numpy().view(np.uint16), binding.read_status(ws.data_ptr()), db


def gpu_accept(inp, acc_len, acc_idx, db=None):
    import torch
    ensure_gpu()
    if db is None:
        db = binding.DeviceBatch(inp, "cuda:0")
    al = torch.from_numpy(acc_len).to("cuda:0")
    ai = torch.from_numpy(acc_idx).to("cuda:0")
    lens, ws = binding.accept_path(db, al, ai)
    torch.cuda.synchronize()
    return (db.kv_cache.cpu().numpy().view(np.uint16), lens.cpu().numpy(), binding.read_status(ws.data_ptr()))


CASES = [
    dict(prefixes=[70, 0, 129, 5], trees=[5, 3, 8, 1], kind="uniform"),
    dict(prefixes=[300, 64, 1000], trees=[64, 1, 33], kind="branch4"),
    dict(prefixes=[200, 260, 230, 300, 10, 700, 64, 63], trees=[4, 8, 2, 6, 0, 32, 16, 7], kind="forest",
         share_group=4),
    dict(prefixes=[1, 2, 3], trees=[64, 64, 64], kind="chain", page_size=128),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_append_matches_oracle(case):
    c = dict(CASES[case])
    inp = I.make_inputs(c.pop("prefixes"), c.pop("trees"), tree_kind=c.pop("kind"), seed=case, stream=910, **c)
    rows = rand_rows(inp.total_q, case)
    ref, ref_st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, rows, inp.page_size)
    got, st, _ = gpu_append(inp, rows)
    assert st == ref_st == 0
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_accept_matches_oracle(case, seed):
    c = dict(CASES[case])
    inp = I.make_inputs(c.pop("prefixes"), c.pop("trees"), tree_kind=c.pop("kind"), seed=case, stream=911, **c)
    acc_len, acc_idx = random_paths(inp, 100 * case + seed)
    ref, ref_lens, ref_st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree,
                                             inp.tree_parent, acc_len, acc_idx, inp.page_size)
    got, lens, st = gpu_accept(inp, acc_len, acc_idx)
    assert st == ref_st == 0
    np.testing.assert_array_equal(lens, ref_lens)
    np.testing.assert_array_equal(got, ref)


def test_golden_paths_after_append():
    g = json.load(open(GOLDEN))
    for case in g["cases"]:
        T, path = len(case["parent"]), case["path"]
        inp = I.make_inputs([67], [T], trees=[case["parent"]], seed=7, stream=912)
        rows = rand_rows(T, 3)
        _, st, db = gpu_append(inp, rows)
        assert st == 0
        acc_idx = np.full(T, -1, np.int32)
        acc_idx[:len(path)] = path
        got, lens, st = gpu_accept(inp, np.array([len(path)], np.int32), acc_idx, db=db)
        assert st == 0 and int(lens[0]) == 67 + len(path), case["name"]
        for k, node in enumerate(case["expect"]):
            t = 67 + k
            page = int(inp.block_table[0, t // inp.page_size])
            np.testing.assert_array_equal(got[page, t % inp.page_size], rows[node], err_msg=case["name"])


def test_malformed_paths_and_bad_blocks_leave_requests_untouched():
    g = json.load(open(GOLDEN))
    for case in g["invalid"]:
        T, path = len(case["parent"]), case["path"]
        inp = I.make_inputs([40, 90], [T, 3], trees=[case["parent"], [-1, 0, 1]], seed=8, stream=913)
        acc_idx = np.full(inp.total_q, -1, np.int32)
        acc_idx[:len(path)] = path
        acc_idx[T:T + 2] = [0, 1]
        acc_len = np.array([len(path), 2], np.int32)
        ref, ref_lens, ref_st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree,
                                                 inp.tree_parent, acc_len, acc_idx, inp.page_size)
        got, lens, st = gpu_accept(inp, acc_len, acc_idx)
        assert st == ref_st == K.STATUS_BAD_TREE, case["name"]
        np.testing.assert_array_equal(lens, ref_lens)
        np.testing.assert_array_equal(got, ref)
    inp = I.make_inputs([100, 50], [5, 3], tree_kind="uniform", seed=9, stream=914)
    inp.block_table[0, 104 // inp.page_size] = inp.num_pages + 3   # the tree region of request 0
    rows = rand_rows(inp.total_q, 4)
    ref, ref_st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, rows, inp.page_size)
    got, st, _ = gpu_append(inp, rows)
    assert st == ref_st == K.STATUS_BAD_BLOCK
    np.testing.assert_array_equal(got, ref)


def test_tree_counts_outside_total_q_are_rejected_without_stray_reads():
    """A negative tree count and counts that run past total_q: the GPU flags the
    malformed request, leaves it untouched and reads no row outside the arrays;
    the other requests match the oracle bit for bit."""
    for prefixes, trees, fix in (((70, 40, 100), (2, 3, 8), {0: -5}), ((70, 40), (5, 3), {1: 13})):
        inp = I.make_inputs(list(prefixes), list(trees), tree_kind="uniform", seed=15, stream=915)
        for b, v in fix.items():
            inp.n_tree[b] = v
        rows = rand_rows(inp.total_q, 16)
        ref, ref_st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, rows,
                                       inp.page_size)
        got, st, _ = gpu_append(inp, rows)
        assert st == ref_st and st & K.STATUS_BAD_TREE
        np.testing.assert_array_equal(got, ref)
        acc_len = np.ones(inp.batch, np.int32)
        acc_idx = np.zeros(inp.total_q, np.int32)
        ref2, ref_lens, ref_st2 = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree,
                                                   inp.tree_parent, acc_len, acc_idx, inp.page_size)
        got2, lens, st2 = gpu_accept(inp, acc_len, acc_idx)
        assert st2 == ref_st2 and st2 & K.STATUS_BAD_TREE
        np.testing.assert_array_equal(lens, ref_lens)
        np.testing.assert_array_equal(got2, ref2)


@pytest.mark.parametrize("cfg", [3, 5])
def test_full_size_append_then_accept(cfg):
    """Workload-sized caches (302 MB for c3; c5 with shared prefix pages), compared whole."""
    inp = I.config_inputs(cfg, seed=0)
    rows = rand_rows(inp.total_q, 20 + cfg)
    ref, st0 = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, rows, inp.page_size)
    got, st, db = gpu_append(inp, rows)
    assert st == st0 == 0
    np.testing.assert_array_equal(got, ref)
    acc_len, acc_idx = random_paths(inp, 30 + cfg)
    ref2, ref_lens, st1 = K.tree_kv_accept(ref, inp.block_table, inp.seq_lens, inp.n_tree, inp.tree_parent,
                                           acc_len, acc_idx, inp.page_size)
    got2, lens, st = gpu_accept(inp, acc_len, acc_idx, db=db)
    assert st == st1 == 0
    np.testing.assert_array_equal(lens, ref_lens)
    np.testing.assert_array_equal(got2, ref2)
