"""GPU parity of the sparse (top-k) verify variant (mla_verify_sparse_attn, through
the C ABI) against the fp64 oracle, at the tolerances of the dense path."""
import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import assert_close, ensure_gpu, errors

pytestmark = pytest.mark.gpu


def run_sparse(inp, idx, splits=0):
    import torch
    ensure_gpu()
    db = binding.DeviceBatch(inp, "cuda:0")
    t = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to("cuda:0")
    out, lse, ws = binding.verify_sparse(db, t, num_splits_req=splits)
    torch.cuda.synchronize()
    return (out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            binding.read_status(ws.data_ptr()))


@pytest.mark.parametrize("topk", [64, 100, 512])
@pytest.mark.parametrize("cfg,div,cap", [(2, 4, None), (3, 16, 4), (5, 16, 16)], ids=["c2", "c3", "c5"])
def test_sparse_parity_scaled_workloads(cfg, div, cap, topk):
    inp = I.scaled_config_inputs(cfg, seed=1, prefix_div=div, batch_cap=cap)
    idx = I.topk_indices(inp, topk, seed=topk)
    ref_o, ref_l = oracle.verify_sparse(inp, idx)
    out, lse, status = run_sparse(inp, idx)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"cfg{cfg} topk{topk}")


def test_sparse_maximum_topk():
    """topk = MLA_MAX_TOPK: 64 slot tiles per token; the shorter prefix lists
    every position once and leaves the rest of its slots unused."""
    inp = I.make_inputs([3000, 1000], [3, 2], tree_kind="forest", seed=6, stream=921)
    idx = I.topk_indices(inp, binding.MAX_TOPK, seed=7)
    assert (idx[3:] == -1).sum() == 2 * (binding.MAX_TOPK - 1000)
    ref_o, ref_l = oracle.verify_sparse(inp, idx)
    for splits in (0, 4):
        out, lse, status = run_sparse(inp, idx, splits=splits)
        assert status == 0
        assert_close(out, lse, ref_o, ref_l, f"topk=max splits={splits}")


@pytest.mark.parametrize("splits", [1, 2, 3, 5])
def test_sparse_split_counts(splits):
    inp = I.scaled_config_inputs(3, seed=2, prefix_div=16, batch_cap=3)
    idx = I.topk_indices(inp, 256, seed=3)
    ref_o, ref_l = oracle.verify_sparse(inp, idx)
    out, lse, status = run_sparse(inp, idx, splits=splits)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"splits={splits}")


@pytest.mark.parametrize("kind", ["forest", "chain", "uniform"])
def test_sparse_unused_and_repeated_slots(kind):
    trees = [1, 2, 3, 7, 33, 64]
    inp = I.make_inputs([0, 5, 70, 600, 1000, 129], trees, tree_kind=kind, seed=4, stream=920)
    idx = I.topk_indices(inp, 192, seed=5, unused_frac=0.3, duplicates=True)
    ref_o, ref_l = oracle.verify_sparse(inp, idx)
    out, lse, status = run_sparse(inp, idx)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, kind)


def test_sparse_full_list_equals_dense_path():
    """Listing every prefix position reproduces the dense kernel's output."""
    import torch
    inp = I.make_inputs([300, 64, 1000], [5, 16, 9], tree_kind="uniform", seed=6, stream=921)
    topk = int((inp.seq_lens - inp.n_tree).max())
    idx = I.topk_indices(inp, topk, seed=7)
    out_s, lse_s, st = run_sparse(inp, idx)
    assert st == 0
    db = binding.DeviceBatch(inp, "cuda:0")
    out_d, lse_d, _ = binding.verify(db)
    torch.cuda.synchronize()
    mx, mean, le = errors(out_s, lse_s, out_d.cpu().numpy().astype(np.float64), lse_d.cpu().numpy().astype(np.float64))
    assert mx < 2e-3 and le < 1e-4, (mx, le)
    ref_o, ref_l = oracle.verify(inp)
    assert_close(out_s, lse_s, ref_o, ref_l, "full list")


def test_sparse_bad_slot_reported_and_rows_zeroed():
    inp = I.make_inputs([100, 80], [4, 6], tree_kind="uniform", seed=8, stream=922)
    idx = I.topk_indices(inp, 64, seed=9)
    idx[1, 3] = 100      # request 0's prefix is 100 positions: 100 is a tree position
    out, lse, status = run_sparse(inp, idx)
    assert status & (1 << binding.MLA_ERR_BAD_INDEX)
    assert np.all(out[:4] == 0) and np.all(np.isneginf(lse[:4]))
    assert np.isfinite(out[4:]).all() and np.isfinite(lse[4:]).all()


@pytest.mark.parametrize("cfg", [3, 5])
def test_sparse_full_size_sampled_rows(cfg):
    """Workload-sized inputs with topk = 512, checked on a seeded sample of rows."""
    inp = I.config_inputs(cfg, seed=0)
    idx = I.topk_indices(inp, 512, seed=10)
    out, lse, status = run_sparse(inp, idx)
    assert status == 0
    rows = I.sample_rows(inp, 512, seed=11)
    ref_o, ref_l = oracle.verify_sparse_rows(inp, idx, rows)
    H = inp.num_heads
    got_o = out.reshape(-1, 512)[rows]
    got_l = lse.reshape(-1)[rows]
    assert_close(got_o, got_l, ref_o, ref_l, f"cfg{cfg} sampled")
