"""CPU checks of the committed DRAM capture summary that bench.py reads for
roofline.traffic and per_workload[*].traffic: it is well formed, and every
launch plan the default bench run reports (the headline workload and the
per-workload sweep, each with the library's own plan choice) has an entry."""
import json
import os
import re
import sys

import pytest

from mla_speculative_decoding_verify_gb300 import binding
from mla_speculative_decoding_verify_gb300 import build as libbuild
from mla_speculative_decoding_verify_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def summary():
    with open(os.path.join(ROOT, "profiles", "verify_kernel_dram.json")) as f:
        return json.load(f)


def shape(cfg):
    """(batch, total_q, max_tree, max_seq_len) of a workload, without building its inputs."""
    prefix, trees, _ = I.config_shape(cfg)
    return len(prefix), int(sum(trees)), int(max(trees)), int(max(p + t for p, t in zip(prefix, trees)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.lib()


def test_summary_is_well_formed():
    d = summary()
    assert re.fullmatch(r"[0-9a-f]{16}", d["source_hash"])
    assert d["workloads"]
    for key, e in d["workloads"].items():
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"], key
        assert e["units"] > 0 and e["dram_read_bytes"] > 0, key
        # every capture was taken without locking the clocks, on one kernel
        assert "--clock-control none" in e["command"] and "-k regex:mla_verify_kernel" in e["command"], key
        wl, plan = key.split("/")
        topk = int(plan[len("sparse-top"):]) if plan.startswith("sparse-top") else None
        assert key == bench.plan_key(wl, e["num_splits"], topk), key


def test_source_hash_ignores_comments_and_layout():
    """The summary stays valid across comment-only and layout-only edits of the
    kernel sources, and goes stale on a code change."""
    from mla_speculative_decoding_verify_gb300 import metrics
    src = "int f(int a) {  // the sum\n    return a + 1; /* one */\n}\n"
    same = "/* header */\nint f(int a)\n{\n  return a + 1;   // changed comment\n}\n"
    other = "int f(int a) { return a + 2; }"
    assert metrics._code_only(src) == metrics._code_only(same)
    assert metrics._code_only(src) != metrics._code_only(other)
    assert re.fullmatch(r"[0-9a-f]{16}", metrics.kernel_source_hash())


def test_every_reported_plan_has_a_capture(lib):
    d = summary()
    legs = [("c3", 0, None)] + list(bench.SWEEP.values())
    for wl, req, topk in legs:
        b, tq, mt, ms = shape(bench.WORKLOADS[wl])
        splits = (binding.sparse_num_splits(b, tq, mt, topk, requested=req) if topk
                  else binding.num_splits(b, tq, mt, ms, requested=req))
        key = bench.plan_key(wl, splits, topk)
        assert key in d["workloads"], f"no DRAM capture for {key}"
