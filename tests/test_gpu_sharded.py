"""Split-KV across ranks on the CUDA path, emulated on one GPU: each "rank"
holds only the pages of its splits (shard_inputs), computes its partials with
mla_verify_attn_split_range, and the gathered partials are merged with
mla_split_combine.  The result must match the fp64 oracle, and for three or
more ranks it must equal, bit for bit, the single-GPU call with as many splits
(the same partition, partials and merge order).  The multi-process exchange
itself is covered on the host (tests/test_sharded_gloo.py)."""
import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I
from mla_speculative_decoding_verify_gb300 import sharded as SH

from gpu_util import assert_close, ensure_gpu

pytestmark = pytest.mark.gpu


def emulate(inp, world, per_rank=1):
    import torch
    ensure_gpu()
    outs, lses = [], []
    for r in range(world):
        S, b0, k = SH.rank_splits(world, r, per_rank)
        loc = SH.shard_inputs(inp, S, b0, k)
        db = binding.DeviceBatch(loc, "cuda:0")
        po, pl, ws = binding.verify_split_range(db, S, b0, k)
        torch.cuda.synchronize()
        assert binding.read_status(ws.data_ptr()) == 0
        outs.append(po)
        lses.append(pl)
    all_o, all_l = torch.cat(outs, 0).contiguous(), torch.cat(lses, 0).contiguous()
    out = torch.empty((inp.total_q, inp.num_heads, 512), dtype=torch.float32, device="cuda:0")
    lse = torch.empty((inp.total_q, inp.num_heads), dtype=torch.float32, device="cuda:0")
    rows = inp.total_q * inp.num_heads
    binding.check(binding.split_combine(all_o.data_ptr(), all_l.data_ptr(), world * per_rank, rows, out.data_ptr(),
                                        lse.data_ptr(), torch.cuda.current_stream().cuda_stream), "combine")
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("world,per_rank", [(2, 1), (3, 1), (4, 2)])
def test_sharded_prefix_matches_oracle_and_single_gpu(world, per_rank):
    inp = I.make_inputs([9000, 3000], [33, 17], tree_kind="uniform", seed=44, stream=980)
    out, lse = emulate(inp, world, per_rank)
    ref_o, ref_l = oracle.verify(inp)
    assert_close(out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_o, ref_l,
                 f"{world} ranks x {per_rank} splits")
    S = world * per_rank
    if S >= 3:   # the single-GPU call with S equal splits runs the same partials and merge
        db = binding.DeviceBatch(inp, "cuda:0")
        o1, l1, _ = binding.verify(db, num_splits_req=S)
        import torch
        torch.cuda.synchronize()
        assert torch.equal(o1, out) and torch.equal(l1, lse)


def test_one_long_request_on_four_ranks_c4_shape():
    """One request of the long-prefix shape (prefix 65536, 64-node tree) over
    four ranks: sampled rows against the oracle."""
    inp = I.make_inputs([65536], [64], tree_kind="branch4", seed=45, stream=981)
    out, lse = emulate(inp, 4, 1)
    rows = np.arange(0, inp.total_q * inp.num_heads, 61)
    ref_o, ref_l = oracle.verify_rows(inp, rows)
    assert_close(out.reshape(-1, 512).cpu().numpy()[rows].astype(np.float64),
                 lse.reshape(-1).cpu().numpy()[rows].astype(np.float64), ref_o, ref_l, "c4-shaped, 4 ranks")


def test_split_range_argument_checks():
    ensure_gpu()
    inp = I.make_inputs([300], [4], seed=46, stream=982)
    db = binding.DeviceBatch(inp, "cuda:0")
    for S, b0, k in ((2, 2, 1), (2, -1, 1), (0, 0, 1), (3, 1, 3), (binding.SPLITS_PERSISTENT, 0, 1)):
        with pytest.raises(binding.MlaError) as e:
            binding.verify_split_range(db, S, b0, k)
        assert e.value.code == binding.MLA_ERR_INVALID_ARG
