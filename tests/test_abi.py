"""CPU checks of the C-ABI library: it loads, exports every declared entry
point, and rejects bad scalar arguments before touching the device."""
import ctypes
import os
import re

import pytest

from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla_verify.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.lib()


def test_header_declares_the_binding_surface():
    assert sorted(binding.EXPORTED) == declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_error_strings(lib):
    assert binding.version() >= 100
    for code in range(0, 9):
        assert binding.error_string(code) not in ("", "unknown status")
    assert binding.error_string(99) == "unknown status"


def _call(**over):
    args = dict(q_lat=16, q_rope=16, kv_cache=16, block_table=16, seq_lens=16, tree_parent=16,
                n_tree=16, scale=0.07, out=16, lse=16, stream=None, batch=1, total_q=1, max_tree=1,
                max_seq_len=65, num_heads=64, page_size=64, num_pages=2, max_pages_per_seq=2,
                num_splits=0, workspace=256, workspace_bytes=1 << 20)
    args.update(over)
    return binding.verify_attn(**args)


@pytest.mark.parametrize("over,code", [
    (dict(num_heads=32), binding.MLA_ERR_UNSUPPORTED),
    (dict(page_size=48), binding.MLA_ERR_UNSUPPORTED),
    (dict(page_size=0), binding.MLA_ERR_INVALID_ARG),
    (dict(max_tree=65), binding.MLA_ERR_UNSUPPORTED),
    (dict(num_splits=65), binding.MLA_ERR_UNSUPPORTED),
    (dict(batch=-1), binding.MLA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.MLA_ERR_INVALID_ARG),
    (dict(scale=0.0), binding.MLA_ERR_INVALID_ARG),        # a softmax scale is positive
    (dict(scale=-0.07), binding.MLA_ERR_INVALID_ARG),
    (dict(q_lat=None), binding.MLA_ERR_INVALID_ARG),
    (dict(out=None), binding.MLA_ERR_INVALID_ARG),
    (dict(kv_cache=24), binding.MLA_ERR_INVALID_ARG),   # not 16-byte aligned
    (dict(num_pages=0), binding.MLA_ERR_INVALID_ARG),
    (dict(batch=0, total_q=0), binding.MLA_OK),           # nothing to do
])
def test_host_argument_checks(lib, over, code):
    assert _call(**over) == code


def test_combine_argument_checks(lib):
    assert binding.split_combine(16, 16, 0, 4, 16, 16, None) == binding.MLA_ERR_INVALID_ARG
    assert binding.split_combine(16, 16, 65, 4, 16, 16, None) == binding.MLA_ERR_INVALID_ARG
    assert binding.split_combine(None, 16, 2, 4, 16, 16, None) == binding.MLA_ERR_INVALID_ARG
    assert binding.split_combine(16, 16, 2, 0, 16, 16, None) == binding.MLA_OK


def test_split_heuristic_and_workspace(lib):
    assert binding.num_splits(4, 64, 16, 4112, requested=5) == 5
    assert binding.num_splits(4, 64, 16, 4112, requested=500) == binding.MAX_SPLITS
    s = binding.num_splits(2, 128, 64, 65600)
    assert 1 <= s <= binding.MAX_SPLITS
    w1 = binding.workspace_size(16, 512, 32, 16416, splits=1)
    w4 = binding.workspace_size(16, 512, 32, 16416, splits=4)
    assert w4 - w1 >= 4 * 512 * 64 * 512 * 4
    assert binding.workspace_size(1, 1, 1, 1, num_heads=32) == 0
    # the persistent schedule: split count 0; its partial slots are sized by the CTA pairs, not the rows
    assert binding.num_splits(16, 512, 32, 16416, requested=binding.SPLITS_PERSISTENT) == 0
    assert binding.sparse_num_splits(16, 512, 32, 512, requested=binding.SPLITS_PERSISTENT) == 0
    assert binding.lib().mla_verify_num_splits(16, 512, 32, 16416, 64, -2) < 0
    wp = binding.workspace_size(16, 512, 32, 16416, splits=binding.SPLITS_PERSISTENT)
    assert wp >= 2 * 1 * 128 * 512 * 4 and wp < w4


def _kv_call(op, **over):
    args = dict(tree_kv=16, kv_cache=16, block_table=16, seq_lens=16, n_tree=16, tree_parent=16, accept_len=16,
                accept_idx=16, new_seq_lens=16, stream=None, batch=1, total_q=1, page_size=64, num_pages=2,
                max_pages_per_seq=2, workspace=256, workspace_bytes=256)
    args.update(over)
    if op == "append":
        return binding.tree_kv_append(args["tree_kv"], args["kv_cache"], args["block_table"], args["seq_lens"],
                                      args["n_tree"], args["stream"], args["batch"], args["total_q"],
                                      args["page_size"], args["num_pages"], args["max_pages_per_seq"],
                                      args["workspace"], args["workspace_bytes"])
    return binding.tree_kv_accept(args["kv_cache"], args["block_table"], args["seq_lens"], args["n_tree"],
                                  args["tree_parent"], args["accept_len"], args["accept_idx"], args["new_seq_lens"],
                                  args["stream"], args["batch"], args["total_q"], args["page_size"],
                                  args["num_pages"], args["max_pages_per_seq"], args["workspace"],
                                  args["workspace_bytes"])


@pytest.mark.parametrize("op", ["append", "accept"])
@pytest.mark.parametrize("over,code", [
    (dict(batch=-1), binding.MLA_ERR_INVALID_ARG),
    (dict(page_size=0), binding.MLA_ERR_INVALID_ARG),
    (dict(workspace=None), binding.MLA_ERR_WORKSPACE),
    (dict(workspace_bytes=2), binding.MLA_ERR_WORKSPACE),
    (dict(kv_cache=None), binding.MLA_ERR_INVALID_ARG),
    (dict(kv_cache=24), binding.MLA_ERR_INVALID_ARG),     # not 16-byte aligned
    (dict(num_pages=0), binding.MLA_ERR_INVALID_ARG),
])
def test_kv_op_host_argument_checks(lib, op, over, code):
    assert _kv_call(op, **over) == code


def test_kv_op_specific_pointer_checks(lib):
    assert _kv_call("append", tree_kv=None) in (binding.MLA_ERR_INVALID_ARG, binding.MLA_ERR_NOT_INITIALIZED)
    assert binding.tree_kv_workspace_size() >= 4


@pytest.mark.parametrize("over,code", [
    (dict(topk=0), binding.MLA_ERR_INVALID_ARG),
    (dict(topk=binding.MAX_TOPK + 1), binding.MLA_ERR_UNSUPPORTED),
    (dict(topk_idx=None), binding.MLA_ERR_INVALID_ARG),
    (dict(scale=-1.0), binding.MLA_ERR_INVALID_ARG),
    (dict(num_heads=32), binding.MLA_ERR_UNSUPPORTED),
])
def test_sparse_host_argument_checks(lib, over, code):
    args = dict(q_lat=16, q_rope=16, kv_cache=16, block_table=16, seq_lens=16, tree_parent=16, n_tree=16,
                topk_idx=16, topk=512, scale=0.07, out=16, lse=16, stream=None, batch=1, total_q=1, max_tree=1,
                max_seq_len=65, num_heads=64, page_size=64, num_pages=2, max_pages_per_seq=2, num_splits=0,
                workspace=256, workspace_bytes=1 << 20)
    args.update(over)
    assert binding.verify_sparse_attn(**args) == code


def test_sparse_split_choice_and_workspace(lib):
    assert binding.sparse_num_splits(16, 512, 32, 512) >= 1
    assert binding.sparse_num_splits(16, 512, 32, 512, requested=3) == 3
    assert binding.sparse_workspace_size(16, 512, 32, 512) > 0
    assert binding.lib().mla_verify_sparse_num_splits(1, 1, 1, 0, 64, 0) < 0


def _graph_create(**over):
    args = dict(q_lat=16, q_rope=16, kv_cache=16, block_table=16, seq_lens=16, tree_parent=16, n_tree=16,
                topk_idx=None, topk=0, scale=0.07, out=16, lse=16, max_batch=1, max_total_q=1, max_tree=1,
                max_seq_len=65, num_heads=64, page_size=64, num_pages=2, max_pages_per_seq=2, num_splits=0,
                workspace=256, workspace_bytes=1 << 20, stream=None)
    args.update(over)
    return binding.verify_graph_create(**args)


@pytest.mark.parametrize("over,code", [
    (dict(max_batch=0), binding.MLA_ERR_INVALID_ARG),
    (dict(max_total_q=0), binding.MLA_ERR_INVALID_ARG),
    (dict(n_tree=None), binding.MLA_ERR_INVALID_ARG),
    (dict(seq_lens=None), binding.MLA_ERR_INVALID_ARG),
    (dict(topk=-1), binding.MLA_ERR_INVALID_ARG),
    (dict(topk=binding.MAX_TOPK + 1), binding.MLA_ERR_UNSUPPORTED),
    (dict(topk=64), binding.MLA_ERR_INVALID_ARG),            # no slot array
])
def test_graph_create_host_checks(lib, over, code):
    got, handle = _graph_create(**over)
    assert got == code and handle is None


def test_graph_create_needs_init_and_launch_checks(lib):
    # without a GPU no device is initialised: nothing is captured
    got, handle = _graph_create()
    assert got in (binding.MLA_ERR_NOT_INITIALIZED, binding.MLA_ERR_CUDA) and handle is None
    assert lib.mla_verify_graph_create(16, 16, 16, 16, 16, 16, 16, None, 0, 0.07, 16, 16, 1, 1, 1, 65, 64, 64,
                                       2, 2, 0, 256, 1 << 20, None, None) == binding.MLA_ERR_INVALID_ARG
    assert binding.verify_graph_launch(None, 1, None) == binding.MLA_ERR_INVALID_ARG
    assert binding.verify_graph_destroy(None) == binding.MLA_OK


def test_tail_cut_workspace_only_for_automatic_single_split(lib):
    """With num_splits = 0 resolving to one split and items of >= 12 KV tiles,
    the workspace holds room for cutting the last round's items (compact
    partials of up to half the CTA pairs' row tiles); an explicit single split,
    or short items, do not."""
    # 4 requests, 24 KV tiles each: one split
    assert binding.num_splits(4, 60, 32, 1516) == 1
    auto = binding.workspace_size(4, 60, 32, 1516, splits=0)
    one = binding.workspace_size(4, 60, 32, 1516, splits=1)
    pairs = 152 // 2                      # no device here: the library assumes 152 SMs
    assert auto - one >= (pairs // 2) * 128 * 512 * 4 * 2
    # 40 requests (ragged trees) of 5 KV tiles: one split, too short to cut
    assert binding.num_splits(40, 319, 8, 264) == 1
    assert binding.workspace_size(40, 319, 8, 264, splits=0) == binding.workspace_size(40, 319, 8, 264, splits=1)
    # the sparse variant (17 tiles at top-k 512) follows the same rule
    assert binding.sparse_workspace_size(16, 512, 32, 512, splits=0) > binding.sparse_workspace_size(16, 512, 32, 512,
                                                                                                    splits=1)


def test_automatic_plan_choices(lib):
    """The plans the split model picks for the five workload shapes and for a
    uniform 96-item shape (host model only, a 152-SM device assumed when none is
    present): c1 five splits (its 4 row tiles fit many times in one wave, so the
    chain of 5 KV tiles is cut into single tiles and combined), c2 two (merged
    in the kernel), c3 one (the last round's 28 items cut in two), c4 seven,
    sparse c3 one; 12 x 8192 x 16 (96 items, whose last round of 20 the per-unit
    grid cannot cut well) the persistent schedule (0); ragged trees never take
    it.  In the one-wave regime the latency model picks three splits or more,
    never two (the merge variant's fixed cost)."""
    assert binding.num_splits(1, 8, 8, 264) == 5
    assert binding.num_splits(4, 64, 16, 4112) == 2
    assert binding.num_splits(16, 512, 32, 16416) == 1
    assert binding.num_splits(2, 128, 64, 65600) == 7
    assert binding.sparse_num_splits(16, 512, 32, 512) == 1
    assert binding.num_splits(12, 192, 16, 8208) == 0
    assert binding.num_splits(12, 191, 16, 8208) != 0          # one request with 15 tree tokens
    assert binding.num_splits(4, 32, 8, 520) == 3               # 16 row tiles of 9 KV tiles
    assert binding.num_splits(1, 8, 8, 16392) == 19             # 4 row tiles of 257 KV tiles: 19 units each
    assert binding.num_splits(16, 511, 32, 16416) == 1          # ragged: the per-unit grid
