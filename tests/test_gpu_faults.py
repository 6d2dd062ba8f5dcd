"""Timeout paths of the verify kernel, tested without faulting or hanging the GPU.

A test build of the library (compiled with MLA_FAULT_INJECTION: 5 ms pipeline
waits and mla_debug_set_fault) makes one bounded wait run out on purpose: a
barrier that nothing completes in the QK issuer, a partial-score exchange that
is never sent, a two-split merge whose first unit never marks its partial
written, or (persistent schedule) pieces of cut items that never mark theirs.  Each case runs in a fresh process: the call must return, report
MLA_ERR_TIMEOUT in the status word, and leave the device usable -- the next call
in the same process, with no fault, matches the fp64 oracle.  The pages'
lesson ("The 99KB Barrier", section "What This Discovery Means": a kernel that
passes its static checks can still fail at run time) and the report-don't-crash
rule ("The Shared Memory Ceiling", section "The Guard") are what these cover.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import ctypes, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
import oracle
from mla_speculative_decoding_verify_gb300 import binding, inputs as I
from gpu_util import assert_close, run_gpu
kind, splits = {kind}, {splits}
torch.cuda.set_device(0)
binding.init(0)
lib = binding.lib()
lib.mla_debug_set_fault.argtypes = [ctypes.c_int]
inp = I.make_inputs({prefixes}, {trees}, tree_kind="uniform", seed=21, stream=950)
assert lib.mla_debug_set_fault(kind) == 0
out, lse, status = run_gpu(inp, splits=splits)
assert status & (1 << binding.MLA_ERR_TIMEOUT), ("no timeout reported", status)
assert lib.mla_debug_set_fault(0) == 0
out, lse, status = run_gpu(inp, splits=splits)
assert status == 0, status
ref_o, ref_l = oracle.verify(inp)
assert_close(out, lse, ref_o, ref_l, "first call after the timeout")
print("ok")
"""


@pytest.fixture(scope="module")
def fault_library():
    from mla_speculative_decoding_verify_gb300 import build
    return build.build_fault_injection()


SHORT = ([300, 200], [4, 3])
CUT = ([4000, 3000], [4, 2])     # persistent schedule: long items cut between CTA pairs


@pytest.mark.parametrize("kind,splits,shape", [(1, 1, SHORT), (3, 1, SHORT), (2, 2, SHORT),
                                               (1, -1, CUT), (3, -1, CUT), (4, -1, CUT)],
                         ids=["qk-wait", "exchange", "merge-poll", "persistent-qk-wait", "persistent-exchange",
                              "persistent-piece-poll"])
def test_timeout_reported_and_device_usable_after(fault_library, kind, splits, shape):
    env = dict(os.environ, MLA_VERIFY_LIBRARY=fault_library)
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"), kind=kind, splits=splits,
                         prefixes=shape[0], trees=shape[1])
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout[-2000:] + res.stderr[-3000:]
