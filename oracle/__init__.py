"""fp64 CPU oracle for MLA tree-verify attention (ctypes wrapper of mla_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg use it; the product path never imports it.  It shares no code
with the CUDA library; both sides only read the same seeded inputs.

The C file states what is computed and which passage it follows.  Parity of
every function here is pinned by the CPU tests (brute force, closed forms,
invariants, planted-mistake builds) rather than by any printed value, since
the pages print no worked example of the attention output.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS = {}

STATUS = {0: "ok", 1: "invalid argument", 6: "bad tree", 7: "bad block id", 9: "bad top-k index"}
INT64_MAX = (1 << 63) - 1


def lib_path(mutant: int = 0) -> str:
    name = "libmla_oracle.so" if mutant == 0 else f"libmla_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE double: no contraction, no fast-math)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant in _LIBS:
            return _LIBS[mutant]
        lib = ctypes.CDLL(build(mutant))
        i64, i32p, u16p, f64p, i64p = (ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_uint16),
                                       ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(ctypes.c_int64))
        lib.mla_oracle_verify_rows.restype = ctypes.c_int
        lib.mla_oracle_verify_rows.argtypes = [u16p, u16p, u16p, i32p, i32p, i32p, i32p,
                                               ctypes.c_double, i64, i64, i64, i64, i64, i64,
                                               i64, i64, i64p, i64, i64, i64, f64p, f64p,
                                               ctypes.c_int]
        lib.mla_oracle_verify_sparse_rows.restype = ctypes.c_int
        lib.mla_oracle_verify_sparse_rows.argtypes = [u16p, u16p, u16p, i32p, i32p, i32p, i32p, i32p, i64,
                                                      ctypes.c_double, i64, i64, i64, i64, i64, i64, i64,
                                                      i64, i64p, i64, f64p, f64p, ctypes.c_int]
        lib.mla_oracle_combine.restype = ctypes.c_int
        lib.mla_oracle_combine.argtypes = [f64p, f64p, i64, i64, i64, f64p, f64p]
        lib.mla_oracle_check.restype = ctypes.c_int
        lib.mla_oracle_check.argtypes = [i32p, i32p, i32p, i32p, i64, i64, i64, i64, i64]
        lib.mla_oracle_mutant.restype = ctypes.c_int
        _LIBS[mutant] = lib
        return lib


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"oracle status {status} ({STATUS.get(status, '?')})")
        self.status = status


def verify_rows(inp, rows: Optional[Sequence[int]] = None,
                key_range: Tuple[int, int] = (0, INT64_MAX), threads: int = 0,
                mutant: int = 0, d_latent: int = 512) -> Tuple[np.ndarray, np.ndarray]:
    """Output rows ``rows`` (global index q * H + h; all rows if None).

    Returns (out [n, d_latent] float64, lse [n] float64).  ``key_range``
    restricts the visible keys to positions [k0, k1) of each request's KV.
    """
    lib = load(mutant)
    H = inp.num_heads
    if rows is None:
        rows = np.arange(inp.total_q * H, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    d_rope = inp.q_rope.shape[-1]
    out = np.zeros((n, d_latent), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    arrs = [np.ascontiguousarray(a) for a in (inp.q_lat, inp.q_rope, inp.kv_cache)]
    ints = [np.ascontiguousarray(a, dtype=np.int32) for a in
            (inp.block_table, inp.seq_lens, inp.tree_parent, inp.n_tree)]
    st = lib.mla_oracle_verify_rows(
        _p(arrs[0], ctypes.c_uint16), _p(arrs[1], ctypes.c_uint16), _p(arrs[2], ctypes.c_uint16),
        _p(ints[0], ctypes.c_int32), _p(ints[1], ctypes.c_int32), _p(ints[2], ctypes.c_int32),
        _p(ints[3], ctypes.c_int32), float(inp.scale), inp.batch, inp.total_q, H, d_latent,
        d_rope, inp.page_size, inp.block_table.shape[1], inp.kv_cache.shape[0],
        _p(rows, ctypes.c_int64), n, int(key_range[0]), int(key_range[1]),
        _p(out, ctypes.c_double), _p(lse, ctypes.c_double), int(threads))
    if st != 0:
        raise OracleError(st)
    return out, lse


def verify(inp, threads: int = 0, mutant: int = 0):
    """All output rows: (out [total_q, H, 512], lse [total_q, H])."""
    out, lse = verify_rows(inp, None, threads=threads, mutant=mutant)
    return out.reshape(inp.total_q, inp.num_heads, -1), lse.reshape(inp.total_q, inp.num_heads)


def verify_sparse_rows(inp, topk_idx, rows: Optional[Sequence[int]] = None, threads: int = 0,
                       mutant: int = 0, d_latent: int = 512) -> Tuple[np.ndarray, np.ndarray]:
    """Sparse (top-k) variant: tree token g sees the prefix positions listed in
    topk_idx[g] (int32 [total_q, topk], -1 = unused slot, one key per slot) and
    its ancestor-or-self tree tokens.  Returns (out [n, d_latent], lse [n])."""
    lib = load(mutant)
    H = inp.num_heads
    if rows is None:
        rows = np.arange(inp.total_q * H, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    assert idx.ndim == 2 and idx.shape[0] == inp.total_q
    out = np.zeros((n, d_latent), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    arrs = [np.ascontiguousarray(a) for a in (inp.q_lat, inp.q_rope, inp.kv_cache)]
    ints = [np.ascontiguousarray(a, dtype=np.int32) for a in
            (inp.block_table, inp.seq_lens, inp.tree_parent, inp.n_tree)]
    st = lib.mla_oracle_verify_sparse_rows(
        _p(arrs[0], ctypes.c_uint16), _p(arrs[1], ctypes.c_uint16), _p(arrs[2], ctypes.c_uint16),
        _p(ints[0], ctypes.c_int32), _p(ints[1], ctypes.c_int32), _p(ints[2], ctypes.c_int32),
        _p(ints[3], ctypes.c_int32), _p(idx, ctypes.c_int32), idx.shape[1], float(inp.scale), inp.batch,
        inp.total_q, H, d_latent, inp.q_rope.shape[-1], inp.page_size, inp.block_table.shape[1],
        inp.kv_cache.shape[0], _p(rows, ctypes.c_int64), n, _p(out, ctypes.c_double),
        _p(lse, ctypes.c_double), int(threads))
    if st != 0:
        raise OracleError(st)
    return out, lse


def verify_sparse(inp, topk_idx, threads: int = 0, mutant: int = 0):
    """All output rows of the sparse variant: (out [total_q, H, 512], lse [total_q, H])."""
    out, lse = verify_sparse_rows(inp, topk_idx, None, threads=threads, mutant=mutant)
    return out.reshape(inp.total_q, inp.num_heads, -1), lse.reshape(inp.total_q, inp.num_heads)


def split_partials(inp, bounds: Sequence[int], rows=None, threads: int = 0, mutant: int = 0):
    """Split-KV partials over key ranges [bounds[s], bounds[s+1]).

    Returns (part_out [S, n, 512], part_lse [S, n])."""
    outs, lses = [], []
    for s in range(len(bounds) - 1):
        o, l = verify_rows(inp, rows, key_range=(bounds[s], bounds[s + 1]), threads=threads,
                           mutant=mutant)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def combine(part_out: np.ndarray, part_lse: np.ndarray, mutant: int = 0):
    """Log-sum-exp weighted merge of split partials (float64)."""
    lib = load(mutant)
    po = np.ascontiguousarray(part_out, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    S, rows, dv = po.shape
    out = np.zeros((rows, dv), dtype=np.float64)
    lse = np.zeros(rows, dtype=np.float64)
    st = lib.mla_oracle_combine(_p(po, ctypes.c_double), _p(pl, ctypes.c_double), S, rows, dv,
                                _p(out, ctypes.c_double), _p(lse, ctypes.c_double))
    if st != 0:
        raise OracleError(st)
    return out, lse


def check(inp, mutant: int = 0) -> int:
    """Validation status of the inputs: 0 ok, 1 bad argument, 6 bad tree, 7 bad block id."""
    lib = load(mutant)
    ints = [np.ascontiguousarray(a, dtype=np.int32) for a in
            (inp.block_table, inp.seq_lens, inp.tree_parent, inp.n_tree)]
    return int(lib.mla_oracle_check(_p(ints[0], ctypes.c_int32), _p(ints[1], ctypes.c_int32),
                                    _p(ints[2], ctypes.c_int32), _p(ints[3], ctypes.c_int32),
                                    inp.batch, inp.total_q, inp.page_size,
                                    inp.block_table.shape[1], inp.kv_cache.shape[0]))
