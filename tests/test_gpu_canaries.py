"""Canaries around every buffer the verify calls write: out, lse and the
workspace are carved out of larger allocations whose guard regions (before and
after) hold a fixed bit pattern, and the pattern must survive the call bit for
bit -- for one KV split, two (merged in the kernel), three (combine kernel),
the automatic choice with its cut tail items, and the sparse variant.  The
results themselves are checked against the fp64 oracle as well."""
import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import assert_close, ensure_gpu

pytestmark = pytest.mark.gpu
GUARD = 4096          # elements / bytes on each side; keeps 16-byte and 256-byte alignment
PATTERN_F32 = np.uint32(0x7FA5A5A5)     # a NaN bit pattern
PATTERN_U8 = 0xA5


def guarded(n, dtype, fill, device):
    import torch
    big = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
    if dtype == torch.float32:
        big.view(torch.int32).fill_(int(fill.view(np.int32)))
    else:
        big.fill_(fill)
    return big, big[GUARD:GUARD + n]


def check_guards(big, n, what):
    import torch
    a = big.cpu().numpy()
    if big.dtype == torch.float32:
        a = a.view(np.uint32)
        want = PATTERN_F32
    else:
        want = PATTERN_U8
    for side, seg in (("before", a[:GUARD]), ("after", a[GUARD + n:])):
        bad = np.flatnonzero(seg != want)
        assert bad.size == 0, f"{what}: {bad.size} words {side} the buffer overwritten (first at {bad[0]})"


def run_guarded(inp, splits=0, topk_idx=None):
    import torch
    ensure_gpu()
    dev = "cuda:0"
    db = binding.DeviceBatch(inp, dev)
    n_out, n_lse = inp.total_q * inp.num_heads * 512, inp.total_q * inp.num_heads
    big_o, out = guarded(n_out, torch.float32, PATTERN_F32, dev)
    big_l, lse = guarded(n_lse, torch.float32, PATTERN_F32, dev)
    if topk_idx is None:
        need = binding.workspace_size(inp.batch, inp.total_q, inp.max_tree, inp.max_seq_len, inp.num_heads, splits)
    else:
        need = binding.sparse_workspace_size(inp.batch, inp.total_q, inp.max_tree, topk_idx.shape[1],
                                             inp.num_heads, splits)
    big_w, ws = guarded(need, torch.uint8, PATTERN_U8, dev)
    out3 = out.view(inp.total_q, inp.num_heads, 512)
    lse2 = lse.view(inp.total_q, inp.num_heads)
    if topk_idx is None:
        binding.verify(db, num_splits_req=splits, out=out3, lse=lse2, workspace=ws)
    else:
        t = torch.from_numpy(np.ascontiguousarray(topk_idx, dtype=np.int32)).to(dev)
        binding.verify_sparse(db, t, num_splits_req=splits, out=out3, lse=lse2, workspace=ws)
    torch.cuda.synchronize()
    status = binding.read_status(ws.data_ptr())
    check_guards(big_o, n_out, "out")
    check_guards(big_l, n_lse, "lse")
    check_guards(big_w, need, "workspace")
    return (out3.cpu().numpy().astype(np.float64), lse2.cpu().numpy().astype(np.float64), status)


@pytest.mark.parametrize("splits", [1, 2, 3, 0, -1])
def test_dense_writes_stay_inside_their_buffers(splits):
    inp = I.make_inputs([700, 64, 2500, 5], [9, 32, 17, 1], tree_kind="forest", seed=31, stream=960)
    out, lse, status = run_guarded(inp, splits)
    assert status == 0
    ref_o, ref_l = oracle.verify(inp)
    assert_close(out, lse, ref_o, ref_l, f"dense, {splits} splits requested")


def test_tail_cut_writes_stay_inside_their_buffers():
    """Many long items on one split: the automatic choice cuts the last round's items in two."""
    inp = I.scaled_config_inputs(3, seed=1, prefix_div=4, batch_cap=None)
    out, lse, status = run_guarded(inp, 0)
    assert status == 0
    rows = np.arange(0, inp.total_q * inp.num_heads, 97)
    ref_o, ref_l = oracle.verify_rows(inp, rows)
    assert_close(out.reshape(-1, 512)[rows], lse.reshape(-1)[rows], ref_o, ref_l, "tail cut, sampled rows")


@pytest.mark.parametrize("splits", [1, 3, -1])
def test_sparse_writes_stay_inside_their_buffers(splits):
    inp = I.make_inputs([900, 300, 1500], [6, 9, 3], tree_kind="uniform", seed=32, stream=961)
    topk = I.topk_indices(inp, 100, seed=33)
    out, lse, status = run_guarded(inp, splits, topk_idx=topk)
    assert status == 0
    ref_o, ref_l = oracle.verify_sparse(inp, topk)
    assert_close(out, lse, ref_o, ref_l, f"sparse, {splits} splits")


def test_persistent_pieces_write_inside_their_buffers():
    """Few long items on the persistent schedule: most items are cut between CTA
    pairs and merged in the kernel; their partial slots live in the workspace."""
    inp = I.make_inputs([4000, 3000, 5000], [8, 4, 6], tree_kind="uniform", seed=34, stream=962)
    out, lse, status = run_guarded(inp, -1)
    assert status == 0
    ref_o, ref_l = oracle.verify(inp)
    assert_close(out, lse, ref_o, ref_l, "persistent, cut items")
