"""Seeded randomized parity: many small batches drawn at random (batch size,
prefix and tree sizes including the edges 0, 1, 63, 64, 65, tree shapes, page
size, KV plan, outlier rows, shared prefix pages), each checked element by
element against the fp64 oracle.  The draws are fixed by the case index, so a
failing case is reproducible on its own.  Dense cases run through
mla_verify_attn with the plan drawn (automatic, 1, 2, 3 or 5 splits, or the
persistent schedule); sparse cases through mla_verify_sparse_attn with a drawn
top-k and unused / repeated slots."""
import numpy as np
import pytest

import oracle
from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import inputs as I

from gpu_util import assert_close, ensure_gpu, run_gpu

pytestmark = pytest.mark.gpu

TREE_KINDS = ["uniform", "forest", "chain", "star", "roots", "depth3", "branch2"]
PLANS = [0, 1, 2, 3, 5, binding.SPLITS_PERSISTENT]
EDGE_PREFIXES = [0, 1, 63, 64, 65, 127, 128, 129]


def draw_case(k: int):
    rng = np.random.default_rng(1000 + k)
    batch = int(rng.integers(1, 9))
    prefixes, trees = [], []
    for _ in range(batch):
        if rng.random() < 0.3:
            prefixes.append(int(rng.choice(EDGE_PREFIXES)))
        else:
            prefixes.append(int(rng.integers(0, 2500)))
        trees.append(int(rng.choice([1, 2, 3, 7, 16, 31, 32, 33, 64])) if rng.random() < 0.9 else 0)
    if sum(trees) == 0:
        trees[0] = 5
    kw = dict(tree_kind=str(rng.choice(TREE_KINDS)), page_size=int(rng.choice([64, 128, 256])),
              seed=k, stream=2000)
    if rng.random() < 0.2:
        kw["outlier_frac"] = 0.02
    if rng.random() < 0.2 and batch >= 2:
        kw["share_group"] = 2
    plan = int(rng.choice(PLANS))
    return prefixes, trees, kw, plan


@pytest.mark.parametrize("k", range(60))
def test_fuzz_dense(k):
    prefixes, trees, kw, plan = draw_case(k)
    inp = I.make_inputs(prefixes, trees, **kw)
    ref_o, ref_l = oracle.verify(inp)
    out, lse, status = run_gpu(inp, splits=plan)
    assert status == 0, (prefixes, trees, kw, plan, status)
    assert_close(out, lse, ref_o, ref_l, f"fuzz {k}: {prefixes} {trees} {kw} plan {plan}")


@pytest.mark.parametrize("k", range(30))
def test_fuzz_sparse(k):
    import torch
    prefixes, trees, kw, plan = draw_case(100 + k)
    kw.pop("share_group", None)
    rng = np.random.default_rng(3000 + k)
    topk = int(rng.choice([1, 17, 64, 100, 256, 512]))
    inp = I.make_inputs(prefixes, trees, **kw)
    idx = I.topk_indices(inp, topk, seed=k, unused_frac=float(rng.choice([0.0, 0.2])),
                         duplicates=bool(rng.random() < 0.5))
    ref_o, ref_l = oracle.verify_sparse(inp, idx)
    ensure_gpu()
    db = binding.DeviceBatch(inp, "cuda:0")
    t = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to("cuda:0")
    out, lse, ws = binding.verify_sparse(db, t, num_splits_req=plan)
    torch.cuda.synchronize()
    status = binding.read_status(ws.data_ptr())
    assert status == 0, (prefixes, trees, kw, plan, topk, status)
    assert_close(out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_o, ref_l,
                 f"sparse fuzz {k}: {prefixes} {trees} {kw} plan {plan} topk {topk}")
