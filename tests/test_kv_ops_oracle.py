"""Pins of the paged-cache oracle (oracle/kv_ops.py): append of the draft tree's
latents and accept/compaction of the accepted path.

Checked against an independent list model of each request's logical KV
sequence, hand-worked cases (tests/golden/tree_kv_accept.json), round trips and
invariants, and the validation rules.  CPU only.
"""
import json
import os

import numpy as np
import pytest

from oracle import kv_ops as K
from mla_speculative_decoding_verify_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_kv_accept.json")


def logical_rows(cache, inp, b, length):
    """Request b's first `length` KV rows, read position by position through the block table."""
    ps = inp.page_size
    out = []
    for t in range(length):
        page = int(inp.block_table[b, t // ps])
        out.append(cache[page, t % ps].copy())
    return np.array(out).reshape(length, K.D_KV)


def small_inputs(seed, prefixes=(70, 0, 129, 5), trees=(5, 3, 8, 1), kind="uniform", share_group=None):
    kw = dict(tree_kind=kind, seed=seed, stream=900)
    if share_group:
        kw["share_group"] = share_group
    return I.make_inputs(list(prefixes), list(trees), **kw)


def random_rows(n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 16, size=(n, K.D_KV), dtype=np.uint16)


def test_append_round_trip_and_nothing_else_changes():
    inp = small_inputs(1)
    rows = random_rows(inp.total_q, 2)
    cache, st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, rows, inp.page_size)
    assert st == 0
    off = np.concatenate([[0], np.cumsum(inp.n_tree)])
    changed = np.zeros(cache.shape[:2], dtype=bool)
    for b in range(inp.batch):
        T, L = int(inp.n_tree[b]), int(inp.seq_lens[b])
        got = logical_rows(cache, inp, b, L)
        np.testing.assert_array_equal(got[L - T:], rows[off[b]:off[b] + T])
        np.testing.assert_array_equal(got[:L - T], logical_rows(inp.kv_cache, inp, b, L)[:L - T])
        for t in range(L - T, L):
            changed[int(inp.block_table[b, t // inp.page_size]), t % inp.page_size] = True
    same = (cache == inp.kv_cache) | (np.isnan(cache.view(np.float16)) & np.isnan(inp.kv_cache.view(np.float16)))
    assert np.all(same.all(axis=2) | changed)


def _apply_list_model(inp, accept_len, accept_idx):
    """Independent model: each request's logical sequence as a Python list of rows."""
    off = np.concatenate([[0], np.cumsum(inp.n_tree)])
    seqs, lens = [], []
    for b in range(inp.batch):
        T, L = int(inp.n_tree[b]), int(inp.seq_lens[b])
        P = L - T
        seq = list(logical_rows(inp.kv_cache, inp, b, L))
        prefix, tree = seq[:P], seq[P:]
        path = [int(v) for v in accept_idx[off[b]:off[b] + int(accept_len[b])]]
        kept = [tree[v] for v in path]
        # positions past the accepted path keep whatever was there before
        new_seq = prefix + kept + tree[len(kept):]
        seqs.append(np.array(new_seq).reshape(L, K.D_KV))
        lens.append(P + len(path))
    return seqs, np.array(lens, dtype=np.int32)


def _random_paths(inp, rng):
    """A random root-to-node path per request (possibly empty)."""
    off = np.concatenate([[0], np.cumsum(inp.n_tree)])
    acc_len = np.zeros(inp.batch, dtype=np.int32)
    acc_idx = np.full(inp.total_q, -1, dtype=np.int32)
    for b in range(inp.batch):
        T = int(inp.n_tree[b])
        par = inp.tree_parent[off[b]:off[b] + T]
        if T == 0:
            continue
        node = int(rng.integers(0, T))
        path = []
        while node >= 0:
            path.append(node)
            node = int(par[node])
        path = path[::-1][: int(rng.integers(0, len(path) + 1))]
        acc_len[b] = len(path)
        acc_idx[off[b]:off[b] + len(path)] = path
    return acc_len, acc_idx


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("kind", ["uniform", "chain", "forest", "branch4"])
def test_accept_matches_list_model(seed, kind):
    inp = small_inputs(seed, kind=kind, trees=(5, 3, 8, 1) if kind != "branch4" else (9, 3, 17, 2))
    acc_len, acc_idx = _random_paths(inp, np.random.default_rng(seed + 10))
    cache, lens, st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree,
                                       inp.tree_parent, acc_len, acc_idx, inp.page_size)
    assert st == 0
    seqs, want_lens = _apply_list_model(inp, acc_len, acc_idx)
    np.testing.assert_array_equal(lens, want_lens)
    for b in range(inp.batch):
        got = logical_rows(cache, inp, b, int(inp.seq_lens[b]))
        np.testing.assert_array_equal(got.view(np.uint16), seqs[b].view(np.uint16))


def test_accept_golden_cases():
    g = json.load(open(GOLDEN))
    for case in g["cases"]:
        T, path = len(case["parent"]), case["path"]
        inp = I.make_inputs([67], [T], trees=[case["parent"]], seed=7, stream=901)
        rows = random_rows(T, 3)
        cache, st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, rows,
                                     inp.page_size)
        assert st == 0
        acc_idx = np.full(T, -1, np.int32)
        acc_idx[:len(path)] = path
        cache2, lens, st = K.tree_kv_accept(cache, inp.block_table, inp.seq_lens, inp.n_tree, inp.tree_parent,
                                            np.array([len(path)], np.int32), acc_idx, inp.page_size)
        assert st == 0, case["name"]
        P = 67
        assert int(lens[0]) == P + len(case["expect"]), case["name"]
        got = logical_rows(cache2, inp, 0, P + T)
        for k, node in enumerate(case["expect"]):
            np.testing.assert_array_equal(got[P + k], rows[node], err_msg=case["name"])


def test_accept_rejects_malformed_paths_and_leaves_them_untouched():
    g = json.load(open(GOLDEN))
    for case in g["invalid"]:
        T, path = len(case["parent"]), case["path"]
        inp = I.make_inputs([40], [T], trees=[case["parent"]], seed=8, stream=902)
        acc_idx = np.full(T, -1, np.int32)
        acc_idx[:len(path)] = path
        cache, lens, st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree,
                                           inp.tree_parent, np.array([len(path)], np.int32), acc_idx,
                                           inp.page_size)
        assert st == K.STATUS_BAD_TREE, case["name"]
        assert int(lens[0]) == int(inp.seq_lens[0])
        np.testing.assert_array_equal(cache.view(np.uint16), inp.kv_cache.view(np.uint16))


def test_accept_len_out_of_range_and_bad_block():
    inp = small_inputs(4)
    acc_len = np.zeros(inp.batch, np.int32)
    acc_len[0] = int(inp.n_tree[0]) + 1
    _, lens, st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, inp.tree_parent,
                                   acc_len, np.zeros(inp.total_q, np.int32), inp.page_size)
    assert st == K.STATUS_BAD_TREE and int(lens[0]) == int(inp.seq_lens[0])
    bt = inp.block_table.copy()
    b = 2
    L, T = int(inp.seq_lens[b]), int(inp.n_tree[b])
    bt[b, (L - 1) // inp.page_size] = inp.kv_cache.shape[0] + 5
    cache, st = K.tree_kv_append(inp.kv_cache, bt, inp.seq_lens, inp.n_tree, random_rows(inp.total_q, 5),
                                 inp.page_size)
    assert st == K.STATUS_BAD_BLOCK


def test_empty_path_and_full_chain_are_identity():
    inp = small_inputs(5, kind="chain")
    off = np.concatenate([[0], np.cumsum(inp.n_tree)])
    zero = np.zeros(inp.batch, np.int32)
    c0, l0, st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, inp.tree_parent,
                                  zero, np.zeros(inp.total_q, np.int32), inp.page_size)
    assert st == 0
    np.testing.assert_array_equal(c0.view(np.uint16), inp.kv_cache.view(np.uint16))
    np.testing.assert_array_equal(l0, inp.seq_lens - inp.n_tree)
    full = np.concatenate([np.arange(int(t), dtype=np.int32) for t in inp.n_tree])
    c1, l1, st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree, inp.tree_parent,
                                  inp.n_tree.astype(np.int32), full, inp.page_size)
    assert st == 0
    np.testing.assert_array_equal(c1.view(np.uint16), inp.kv_cache.view(np.uint16))
    np.testing.assert_array_equal(l1, inp.seq_lens)


def test_shared_prefix_pages_are_not_touched():
    inp = I.make_inputs([200, 260, 230, 300], [4, 8, 2, 6], tree_kind="uniform", seed=9, stream=903,
                        share_group=4)
    cache, st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, inp.n_tree,
                                 random_rows(inp.total_q, 6), inp.page_size)
    assert st == 0
    shared = set(int(p) for p in inp.block_table[0, :200 // inp.page_size])
    for p in shared:
        np.testing.assert_array_equal(cache[p].view(np.uint16), inp.kv_cache[p].view(np.uint16))


def test_request_rows_follow_clamped_counts_and_stay_inside_total_q():
    """A negative tree count takes no rows (later requests start where it would have),
    and a request whose rows would reach past total_q is rejected untouched."""
    # negative count: request 0 is malformed; requests 1 and 2 read rows 0..2 and 3..10
    inp = small_inputs(11, prefixes=(70, 40, 100), trees=(2, 3, 8))
    n_tree = inp.n_tree.copy()
    n_tree[0] = -5
    rows = random_rows(inp.total_q, 12)
    got, st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, n_tree, rows, inp.page_size)
    assert st == K.STATUS_BAD_TREE
    np.testing.assert_array_equal(logical_rows(got, inp, 0, int(inp.seq_lens[0])),
                                  logical_rows(inp.kv_cache, inp, 0, int(inp.seq_lens[0])))
    for b, lo in ((1, 0), (2, 3)):
        T, L = int(n_tree[b]), int(inp.seq_lens[b])
        np.testing.assert_array_equal(logical_rows(got, inp, b, L)[L - T:], rows[lo:lo + T])
    # counts that reach past total_q: request 1 (rows 5 .. 17 of 8) is rejected, request 0 appended
    inp = small_inputs(13, prefixes=(70, 40), trees=(5, 3))
    n_tree = inp.n_tree.copy()
    n_tree[1] = 13
    rows = random_rows(inp.total_q, 14)
    got, st = K.tree_kv_append(inp.kv_cache, inp.block_table, inp.seq_lens, n_tree, rows, inp.page_size)
    assert st == K.STATUS_BAD_TREE
    np.testing.assert_array_equal(logical_rows(got, inp, 0, 75)[70:], rows[:5])
    np.testing.assert_array_equal(logical_rows(got, inp, 1, 43), logical_rows(inp.kv_cache, inp, 1, 43))
    acc_len = np.array([1, 1], np.int32)
    acc_idx = np.zeros(inp.total_q, np.int32)
    got, lens, st = K.tree_kv_accept(inp.kv_cache, inp.block_table, inp.seq_lens, n_tree, inp.tree_parent,
                                     acc_len, acc_idx, inp.page_size)
    assert st & K.STATUS_BAD_TREE
    assert int(lens[1]) == int(inp.seq_lens[1])
    np.testing.assert_array_equal(logical_rows(got, inp, 1, 43), logical_rows(inp.kv_cache, inp, 1, 43))
