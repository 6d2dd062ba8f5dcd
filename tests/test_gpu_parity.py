"""GPU parity of the CUDA verify path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import assert_close, ensure_gpu, errors, run_gpu

pytestmark = pytest.mark.gpu

# Reduced copies of the five workloads: same tree generators, paging and value
# recipe, prefixes divided so the oracle evaluates every row in seconds while
# the kernel still walks many KV tiles and a ragged last tile.
SCALED = [(1, 1, None), (2, 4, None), (3, 16, 4), (4, 64, None), (5, 16, 16)]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("cfg,div,cap", SCALED, ids=[f"c{c[0]}" for c in SCALED])
def test_parity_scaled_workloads(cfg, div, cap, seed):
    inp = I.scaled_config_inputs(cfg, seed=seed, prefix_div=div, batch_cap=cap)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"cfg{cfg} seed{seed}")


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_parity_split_counts(splits):
    inp = I.scaled_config_inputs(3, seed=1, prefix_div=16, batch_cap=3)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=splits)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"splits={splits}")


EDGE_PREFIX = [0, 1, 63, 64, 65, 127, 129]


@pytest.mark.parametrize("prefix", EDGE_PREFIX)
@pytest.mark.parametrize("kind", ["forest", "chain", "uniform"])
def test_edge_prefix_and_trees(prefix, kind):
    trees = [1, 2, 3, 7, 33, 64]
    inp = I.make_inputs([prefix] * len(trees), trees, tree_kind=kind, seed=prefix, stream=500)
    ref_o, ref_l = oracle.verify(inp)
    for splits in (1, 2):
        out, lse, status = run_gpu(inp, splits=splits)
        assert status == 0
        assert_close(out, lse, ref_o, ref_l, f"prefix={prefix} kind={kind} splits={splits}")


@pytest.mark.parametrize("splits", [1, 3])
def test_requests_without_tree_tokens(splits):
    """Requests with no draft tokens (n_tree = 0, prefix only) sit between real
    ones: they add no rows, and the others keep their offsets and results."""
    inp = I.make_inputs([100, 500, 64, 0, 700], [5, 0, 3, 0, 9], tree_kind="uniform", seed=8, stream=507)
    assert inp.total_q == 17
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=splits)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"empty trees, splits={splits}")


@pytest.mark.parametrize("page_size", [64, 128, 192])
def test_page_sizes(page_size):
    inp = I.make_inputs([300, 64, 1000], [5, 16, 9], tree_kind="uniform", page_size=page_size,
                        seed=3, stream=501)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"page_size={page_size}")


def test_paged_layout_is_bitwise_irrelevant():
    """Same logical KV rows, contiguous vs shuffled pages: identical bits."""
    a = I.make_inputs([777, 1500], [16, 9], tree_kind="uniform", seed=5, stream=502, shuffle=False)
    b = I.make_inputs([777, 1500], [16, 9], tree_kind="uniform", seed=5, stream=502, shuffle=True)
    assert not np.array_equal(a.block_table, b.block_table)
    oa, la, _ = run_gpu(a)
    ob, lb, _ = run_gpu(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_repeatable_bitwise():
    inp = I.scaled_config_inputs(2, seed=2, prefix_div=8)
    o1, l1, _ = run_gpu(inp, splits=3)
    o2, l2, _ = run_gpu(inp, splits=3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_outlier_rows_keep_tolerance():
    """Config-2 style outliers (1% of c_kv rows x8) at full prefix 4096, all rows."""
    inp = I.config_inputs(2, seed=0)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, "4 x 4096 outliers, full")


_FULL = {}


def _full(cfg):
    if cfg not in _FULL:
        _FULL.clear()
        _FULL[cfg] = I.config_inputs(cfg, seed=0)
    return _FULL[cfg]


@pytest.mark.parametrize("cfg,splits", [(1, 0), (3, 0), (4, 16), (4, 32), (4, 0), (5, 0)])
def test_parity_full_size_sampled_rows(cfg, splits):
    """Full workload sizes in the benchmark's launch configuration; the oracle
    evaluates a seeded sample of rows (always the first and last row of each request)."""
    inp = _full(cfg)
    out, lse, status = run_gpu(inp, splits=splits)
    assert status == 0
    rows = I.sample_rows(inp, 160, seed=cfg)
    ref_o, ref_l = oracle.verify_rows(inp, rows)
    H = inp.num_heads
    got_o = out.reshape(-1, out.shape[-1])[rows]
    got_l = lse.reshape(-1)[rows]
    assert_close(got_o, got_l, ref_o, ref_l, f"cfg{cfg} full, splits={splits}")
    assert np.isfinite(out).all()


def test_split_combine_matches_oracle():
    import torch
    ensure_gpu()
    rng = np.random.default_rng(0)
    S, rows = 5, 333
    po = rng.standard_normal((S, rows, 512)).astype(np.float32)
    pl = (rng.standard_normal((S, rows)) * 3).astype(np.float32)
    pl[1, :40] = -np.inf
    pl[:, 50] = -np.inf                      # a row with no keys at all
    ref_o, ref_l = oracle.combine(po.astype(np.float64), pl.astype(np.float64))
    d_po = torch.from_numpy(po).cuda()
    d_pl = torch.from_numpy(pl).cuda()
    out = torch.empty((rows, 512), device="cuda")
    lse = torch.empty(rows, device="cuda")
    code = binding.split_combine(d_po.data_ptr(), d_pl.data_ptr(), S, rows, out.data_ptr(),
                                 lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == binding.MLA_OK
    torch.cuda.synchronize()
    o = out.cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.isneginf(l[50]) and not o[50].any()
    mx, mean, le = errors(o, l, ref_o, ref_l)
    assert mx < 1e-5 and le < 1e-5


def test_invalid_tree_reported_and_rows_zeroed():
    inp = I.make_inputs([100, 50], [4, 6], tree_kind="uniform", seed=9, stream=503)
    rows0 = np.arange(4 * inp.num_heads)
    ref_o, ref_l = oracle.verify_rows(inp, rows0)      # request 0, before corruption
    inp.tree_parent = inp.tree_parent.copy()
    inp.tree_parent[4 + 3] = 5               # parent not earlier than the node: invalid
    out, lse, status = run_gpu(inp)
    assert status & (1 << binding.MLA_ERR_BAD_TREE)
    assert not out[4:].any() and np.isneginf(lse[4:]).all()
    assert_close(out[:4].reshape(-1, 512), lse[:4].reshape(-1), ref_o, ref_l,
                 "valid request next to an invalid one")


def test_bad_block_id_reported():
    """A block id outside the cache: status bit, the request's rows written as
    out = 0, lse = -inf (the header's contract), its neighbour unaffected."""
    inp = I.make_inputs([200, 130], [3, 4], tree_kind="uniform", seed=4, stream=504)
    ref_o, ref_l = oracle.verify(inp)          # on the intact block table
    inp.block_table = inp.block_table.copy()
    inp.block_table[0, 1] = inp.num_pages + 5
    out, lse, status = run_gpu(inp)
    assert status & (1 << binding.MLA_ERR_BAD_BLOCK)
    assert not out[:3].any() and np.isneginf(lse[:3]).all()
    assert_close(out[3:], lse[3:], ref_o[3:], ref_l[3:], "valid request next to a bad block id")


def test_argument_errors_before_launch():
    ensure_gpu()
    inp = I.make_inputs([64], [2], seed=1, stream=505)
    db = binding.DeviceBatch(inp, "cuda:0")
    with pytest.raises(binding.MlaError) as e:
        binding.verify(db, num_splits_req=binding.MAX_SPLITS + 1)
    assert e.value.code == binding.MLA_ERR_UNSUPPORTED
    import torch
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.MlaError) as e:
        binding.verify(db, workspace=small)
    assert e.value.code == binding.MLA_ERR_WORKSPACE


def test_cuda_graph_capture_and_replay():
    """mla_verify_attn is capturable in a CUDA graph after mla_init: the graph
    replays prep -> verify -> combine and reads the buffers at replay time."""
    import torch
    ensure_gpu()
    kw = dict(tree_kind="uniform", stream=502)
    a = I.make_inputs([700, 130, 64], [9, 33, 4], seed=11, **kw)
    b = I.make_inputs([700, 130, 64], [9, 33, 4], seed=12, **kw)
    assert a.kv_cache.shape == b.kv_cache.shape and a.block_table.shape == b.block_table.shape
    db = binding.DeviceBatch(a, "cuda:0")
    splits = 3
    out = torch.empty((a.total_q, a.num_heads, 512), dtype=torch.float32, device="cuda:0")
    lse = torch.empty((a.total_q, a.num_heads), dtype=torch.float32, device="cuda:0")
    ws = torch.empty(binding.workspace_size(a.batch, a.total_q, a.max_tree, a.max_seq_len, a.num_heads,
                                            splits), dtype=torch.uint8, device="cuda:0")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        binding.verify(db, splits, out=out, lse=lse, workspace=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.verify(db, splits, out=out, lse=lse, workspace=ws, stream=torch.cuda.current_stream())
    for tag, inp in (("second batch", b), ("first batch", a)):
        for name in ("q_lat", "q_rope", "kv_cache", "block_table", "seq_lens", "tree_parent", "n_tree"):
            src = torch.from_numpy(np.ascontiguousarray(getattr(inp, name)).view(
                np.int32 if getattr(inp, name).dtype == np.int32 else np.int16))
            getattr(db, name).copy_(src)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert binding.read_status(ws.data_ptr()) == 0
        ref_o, ref_l = oracle.verify(inp)
        assert_close(out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                     ref_o, ref_l, f"graph replay, {tag}")
