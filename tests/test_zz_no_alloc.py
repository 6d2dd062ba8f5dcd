"""The allocation-free entry point, for callers that cannot allocate device memory.

Some callers cannot provide a device workspace (a plugin inside a serving
engine that owns all device memory through its own pool, a latency-critical
loop that must not call cudaMalloc).  mla_verify_attn_noalloc serves them from
a static 1 MiB device scratch.  Its results are compared with the workspace
entry point's and with the fp64 oracle.  This file is collected last so that a
run that stops at the first failure has already run every other test; it sets
up the library itself, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import assert_close, ensure_gpu, run_gpu

pytestmark = pytest.mark.gpu


def _noalloc(inp):
    import torch
    ensure_gpu()
    db = binding.DeviceBatch(inp, "cuda:0")
    out = torch.full((inp.total_q, inp.num_heads, 512), float("nan"), device="cuda")
    lse = torch.full((inp.total_q, inp.num_heads), float("nan"), device="cuda")
    code = binding.verify_attn_noalloc(
        db.q_lat.data_ptr(), db.q_rope.data_ptr(), db.kv_cache.data_ptr(), db.block_table.data_ptr(),
        db.seq_lens.data_ptr(), db.tree_parent.data_ptr(), db.n_tree.data_ptr(), inp.scale,
        out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream, inp.batch,
        inp.total_q, inp.max_tree, inp.max_seq_len, inp.num_heads, inp.page_size, inp.num_pages,
        inp.max_pages_per_seq)
    torch.cuda.synchronize()
    return code, out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def test_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row on different batches: each equals mla_verify_attn's result
    and the fp64 oracle's, and leaves a clean status word."""
    first = I.scaled_config_inputs(3, seed=0, prefix_div=16, batch_cap=4)
    second = I.make_inputs([700, 2500, 64], [9, 32, 1], tree_kind="forest", seed=3, stream=900)
    for inp in (first, second):
        ref_out, ref_lse, status = run_gpu(inp)
        assert status == 0
        code, out, lse = _noalloc(inp)
        assert code == binding.MLA_OK, binding.error_string(code)
        assert binding.noalloc_read_status() == 0
        assert_close(out, lse, ref_out, ref_lse, f"noalloc vs workspace path ({inp.name})")
        o_ref, l_ref = oracle.verify(inp)
        assert_close(out, lse, o_ref, l_ref, f"noalloc vs oracle ({inp.name})")


def test_noalloc_status_reports_a_bad_block():
    """A block id out of range in one request: the status word read back from the
    static scratch carries the bad-block bit; the other request matches the oracle."""
    inp = I.make_inputs([300, 200], [6, 5], tree_kind="uniform", seed=4, stream=901)
    o_ref, l_ref = oracle.verify(inp)              # on the intact block table
    inp.block_table[0, 1] = inp.num_pages + 7
    code, out, lse = _noalloc(inp)
    assert code == binding.MLA_OK
    assert binding.noalloc_read_status() & (1 << binding.MLA_ERR_BAD_BLOCK)
    rows = slice(int(inp.n_tree[0]), int(inp.total_q))
    assert_close(out[rows], lse[rows], o_ref[rows], l_ref[rows], "noalloc, request with valid pages")
    # the next call starts from a clean status word
    ok = I.make_inputs([300], [6], tree_kind="uniform", seed=5, stream=902)
    code, _, _ = _noalloc(ok)
    assert code == binding.MLA_OK and binding.noalloc_read_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ensure_gpu()
    code = binding.verify_attn_noalloc(16, 16, 16, 16, 16, 16, 16, 0.07, 16, 16, None, 4096, 200000,
                                       64, 70000, 64, 64, 10000, 2000)
    assert code == binding.MLA_ERR_WORKSPACE
