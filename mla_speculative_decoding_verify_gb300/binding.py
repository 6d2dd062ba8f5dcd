"""ctypes binding of libmla_verify.so (the C ABI in include/mla_verify.h).

Argument marshalling only: every step of the verify path runs in the CUDA
library.  torch is used for device memory and streams.  If the compiled
library is missing, every entry point raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libmla_verify.so"
# The in-tree build; MLA_VERIFY_LIBRARY names another build of the same library
# (the tests use it to load the fault-injection build in a separate process).
LIB_PATH = os.environ.get("MLA_VERIFY_LIBRARY") or os.path.join(_HERE, LIB_NAME)

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_TIMEOUT = 5
MLA_ERR_BAD_TREE = 6
MLA_ERR_BAD_BLOCK = 7
MLA_ERR_NOT_INITIALIZED = 8
MLA_ERR_BAD_INDEX = 9

NUM_HEADS = 64
D_LATENT = 512
D_ROPE = 64
MAX_TREE = 64
MAX_SPLITS = 64
SPLITS_PERSISTENT = -1   # num_splits value asking for the persistent schedule
MAX_TOPK = 2048

EXPORTED = ("mla_version", "mla_error_string", "mla_init", "mla_verify_num_splits",
            "mla_verify_workspace_size", "mla_verify_attn", "mla_split_combine",
            "mla_read_status", "mla_set_profile_events", "mla_verify_attn_noalloc",
            "mla_verify_noalloc_read_status", "mla_verify_attn_split_range",
            "mla_tree_kv_workspace_size", "mla_tree_kv_append", "mla_tree_kv_accept",
            "mla_verify_sparse_num_splits", "mla_verify_sparse_workspace_size", "mla_verify_sparse_attn",
            "mla_verify_graph_create", "mla_verify_graph_launch", "mla_verify_graph_destroy")

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class MlaError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        msg = error_string(code) if _lib is not None else str(code)
        super().__init__(f"{what}: status {code} ({msg})" if what else f"status {code} ({msg})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load the compiled library (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_NAME} is not built (expected at {LIB_PATH}); "
                               "run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.mla_version.restype = i32
        L.mla_error_string.restype = ctypes.c_char_p
        L.mla_error_string.argtypes = [i32]
        L.mla_init.restype = i32
        L.mla_init.argtypes = [i32]
        L.mla_verify_num_splits.restype = i32
        L.mla_verify_num_splits.argtypes = [i32] * 6
        L.mla_verify_workspace_size.restype = sz
        L.mla_verify_workspace_size.argtypes = [i32] * 6
        L.mla_verify_attn.restype = i32
        L.mla_verify_attn.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp,
                                      i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, sz]
        L.mla_verify_attn_noalloc.restype = i32
        L.mla_verify_attn_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp,
                                              i32, i32, i32, i32, i32, i32, i32, i32]
        L.mla_verify_attn_split_range.restype = i32
        L.mla_verify_attn_split_range.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp,
                                                  i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, sz]
        L.mla_verify_noalloc_read_status.restype = i32
        L.mla_verify_noalloc_read_status.argtypes = [vp]
        L.mla_split_combine.restype = i32
        L.mla_split_combine.argtypes = [vp, vp, i32, i32, vp, vp, vp]
        L.mla_set_profile_events.restype = i32
        L.mla_set_profile_events.argtypes = [vp, vp]
        L.mla_read_status.restype = i32
        L.mla_read_status.argtypes = [vp, ctypes.POINTER(i32)]
        L.mla_verify_sparse_num_splits.restype = i32
        L.mla_verify_sparse_num_splits.argtypes = [i32] * 6
        L.mla_verify_sparse_workspace_size.restype = sz
        L.mla_verify_sparse_workspace_size.argtypes = [i32] * 6
        L.mla_verify_sparse_attn.restype = i32
        L.mla_verify_sparse_attn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, f32, vp, vp, vp,
                                             i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, sz]
        L.mla_tree_kv_workspace_size.restype = sz
        L.mla_tree_kv_workspace_size.argtypes = []
        L.mla_tree_kv_append.restype = i32
        L.mla_tree_kv_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, sz]
        L.mla_tree_kv_accept.restype = i32
        L.mla_tree_kv_accept.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, sz]
        L.mla_verify_graph_create.restype = i32
        L.mla_verify_graph_create.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, f32, vp, vp,
                                              i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, sz, vp,
                                              ctypes.POINTER(vp)]
        L.mla_verify_graph_launch.restype = i32
        L.mla_verify_graph_launch.argtypes = [vp, i32, vp]
        L.mla_verify_graph_destroy.restype = i32
        L.mla_verify_graph_destroy.argtypes = [vp]
        _lib = L
        return L


def error_string(code: int) -> str:
    return lib().mla_error_string(int(code)).decode()


def version() -> int:
    return int(lib().mla_version())


def check(code: int, what: str = "") -> None:
    if code != MLA_OK:
        raise MlaError(code, what)


def init(device: int = 0) -> None:
    check(lib().mla_init(int(device)), "mla_init")


def num_splits(batch, total_q, max_tree, max_seq_len, num_heads=NUM_HEADS, requested=0) -> int:
    """KV splits the verify call will use; 0 means the persistent schedule."""
    s = lib().mla_verify_num_splits(batch, total_q, max_tree, max_seq_len, num_heads, requested)
    if s < 0:
        raise MlaError(-s, "mla_verify_num_splits")
    return int(s)


def workspace_size(batch, total_q, max_tree, max_seq_len, num_heads=NUM_HEADS, splits=0) -> int:
    return int(lib().mla_verify_workspace_size(batch, total_q, max_tree, max_seq_len, num_heads,
                                               splits))


def verify_attn(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale,
                out, lse, stream, batch, total_q, max_tree, max_seq_len, num_heads, page_size,
                num_pages, max_pages_per_seq, num_splits, workspace, workspace_bytes) -> int:
    """Raw call with integer pointers; returns the mla_status code."""
    return int(lib().mla_verify_attn(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent,
                                     n_tree, float(scale), out, lse, stream, batch, total_q,
                                     max_tree, max_seq_len, num_heads, page_size, num_pages,
                                     max_pages_per_seq, num_splits, workspace, workspace_bytes))


def verify_attn_split_range(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale,
                            part_out, part_lse, stream, batch, total_q, max_tree, max_seq_len, num_heads,
                            page_size, num_pages, max_pages_per_seq, num_splits, split_begin, split_count,
                            workspace, workspace_bytes) -> int:
    """Raw call: the partials of splits split_begin .. + split_count - 1 of num_splits; returns the status."""
    return int(lib().mla_verify_attn_split_range(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent,
                                                 n_tree, float(scale), part_out, part_lse, stream, batch, total_q,
                                                 max_tree, max_seq_len, num_heads, page_size, num_pages,
                                                 max_pages_per_seq, num_splits, split_begin, split_count,
                                                 workspace, workspace_bytes))


def noalloc_read_status() -> int:
    """Device status word of the last allocation-free call on the current device
    (synchronous copy; synchronise the call's stream first)."""
    v = ctypes.c_int(0)
    check(lib().mla_verify_noalloc_read_status(ctypes.byref(v)), "mla_verify_noalloc_read_status")
    return int(v.value)


def verify_attn_noalloc(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree,
                        scale, out, lse, stream, batch, total_q, max_tree, max_seq_len, num_heads,
                        page_size, num_pages, max_pages_per_seq) -> int:
    """Raw call of the allocation-free entry point (static 1 MiB device scratch,
    one KV split) for callers that cannot provide a workspace; returns the status."""
    return int(lib().mla_verify_attn_noalloc(q_lat, q_rope, kv_cache, block_table, seq_lens,
                                             tree_parent, n_tree, float(scale), out, lse, stream,
                                             batch, total_q, max_tree, max_seq_len, num_heads,
                                             page_size, num_pages, max_pages_per_seq))


def split_combine(part_out, part_lse, num_splits, rows, out, lse, stream) -> int:
    return int(lib().mla_split_combine(part_out, part_lse, num_splits, rows, out, lse, stream))


def set_profile_events(begin, end) -> None:
    """Record CUDA events (raw cudaEvent_t handles) around the fused verify kernel."""
    check(lib().mla_set_profile_events(begin, end), "mla_set_profile_events")


def sparse_num_splits(batch, total_q, max_tree, topk, num_heads=NUM_HEADS, requested=0) -> int:
    """KV splits the sparse verify call will use; 0 means the persistent schedule."""
    s = lib().mla_verify_sparse_num_splits(batch, total_q, max_tree, topk, num_heads, requested)
    if s < 0:
        raise MlaError(-s, "mla_verify_sparse_num_splits")
    return int(s)


def sparse_workspace_size(batch, total_q, max_tree, topk, num_heads=NUM_HEADS, splits=0) -> int:
    return int(lib().mla_verify_sparse_workspace_size(batch, total_q, max_tree, topk, num_heads, splits))


def verify_sparse_attn(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, topk_idx, topk,
                       scale, out, lse, stream, batch, total_q, max_tree, max_seq_len, num_heads, page_size,
                       num_pages, max_pages_per_seq, num_splits, workspace, workspace_bytes) -> int:
    """Raw call of the sparse (top-k) variant; returns the mla_status code."""
    return int(lib().mla_verify_sparse_attn(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree,
                                            topk_idx, topk, float(scale), out, lse, stream, batch, total_q,
                                            max_tree, max_seq_len, num_heads, page_size, num_pages,
                                            max_pages_per_seq, num_splits, workspace, workspace_bytes))


def tree_kv_workspace_size() -> int:
    return int(lib().mla_tree_kv_workspace_size())


def tree_kv_append(tree_kv, kv_cache, block_table, seq_lens, n_tree, stream, batch, total_q, page_size,
                   num_pages, max_pages_per_seq, workspace, workspace_bytes) -> int:
    """Raw call: write the draft tree's latents into the paged cache; returns the status."""
    return int(lib().mla_tree_kv_append(tree_kv, kv_cache, block_table, seq_lens, n_tree, stream, batch,
                                        total_q, page_size, num_pages, max_pages_per_seq, workspace,
                                        workspace_bytes))


def tree_kv_accept(kv_cache, block_table, seq_lens, n_tree, tree_parent, accept_len, accept_idx,
                   new_seq_lens, stream, batch, total_q, page_size, num_pages, max_pages_per_seq,
                   workspace, workspace_bytes) -> int:
    """Raw call: compact the accepted path of each request's tree; returns the status."""
    return int(lib().mla_tree_kv_accept(kv_cache, block_table, seq_lens, n_tree, tree_parent, accept_len,
                                        accept_idx, new_seq_lens, stream, batch, total_q, page_size,
                                        num_pages, max_pages_per_seq, workspace, workspace_bytes))


def read_status(workspace) -> int:
    v = ctypes.c_int(0)
    check(lib().mla_read_status(workspace, ctypes.byref(v)), "mla_read_status")
    return int(v.value)


# ---------------------------------------------------------------- torch glue

class DeviceBatch:
    """A batch of verify inputs resident on the GPU (torch tensors, bf16 as int16 bits)."""

    def __init__(self, inp, device="cuda", pin: bool = False):
        import numpy as np
        import torch
        self.inp = inp
        dev = torch.device(device)

        def up(a, dtype):
            t = torch.from_numpy(np.ascontiguousarray(a).view(dtype))
            return t.to(dev, non_blocking=False)
        self.q_lat = up(inp.q_lat, np.int16)
        self.q_rope = up(inp.q_rope, np.int16)
        self.kv_cache = up(inp.kv_cache, np.int16)
        self.block_table = up(inp.block_table, np.int32)
        self.seq_lens = up(inp.seq_lens, np.int32)
        self.tree_parent = up(inp.tree_parent, np.int32)
        self.n_tree = up(inp.n_tree, np.int32)
        self.device = dev


def verify(db: "DeviceBatch", num_splits_req: int = 0, out=None, lse=None, workspace=None,
           stream=None, max_tree: Optional[int] = None, max_seq_len: Optional[int] = None):
    """Run mla_verify_attn on a DeviceBatch; returns (out [total_q, 64, 512], lse [total_q, 64])."""
    import torch
    inp = db.inp
    mt = inp.max_tree if max_tree is None else max_tree
    ms = inp.max_seq_len if max_seq_len is None else max_seq_len
    if out is None:
        out = torch.empty((inp.total_q, inp.num_heads, D_LATENT), dtype=torch.float32, device=db.device)
    if lse is None:
        lse = torch.empty((inp.total_q, inp.num_heads), dtype=torch.float32, device=db.device)
    need = workspace_size(inp.batch, inp.total_q, mt, ms, inp.num_heads, num_splits_req)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=db.device)
    if stream is None:
        stream = torch.cuda.current_stream(db.device)
    code = verify_attn(db.q_lat.data_ptr(), db.q_rope.data_ptr(), db.kv_cache.data_ptr(),
                       db.block_table.data_ptr(), db.seq_lens.data_ptr(), db.tree_parent.data_ptr(),
                       db.n_tree.data_ptr(), inp.scale, out.data_ptr(), lse.data_ptr(),
                       stream.cuda_stream, inp.batch, inp.total_q, mt, ms, inp.num_heads,
                       inp.page_size, inp.num_pages, inp.max_pages_per_seq, num_splits_req,
                       workspace.data_ptr(), workspace.numel())
    check(code, "mla_verify_attn")
    return out, lse, workspace


def verify_split_range(db: "DeviceBatch", num_splits: int, split_begin: int, split_count: int,
                       part_out=None, part_lse=None, workspace=None, stream=None):
    """Partials of a range of KV splits on a DeviceBatch: returns (part_out
    [split_count, total_q, 64, 512], part_lse [split_count, total_q, 64], workspace)."""
    import torch
    inp = db.inp
    if part_out is None:
        part_out = torch.empty((split_count, inp.total_q, inp.num_heads, D_LATENT), dtype=torch.float32,
                               device=db.device)
    if part_lse is None:
        part_lse = torch.empty((split_count, inp.total_q, inp.num_heads), dtype=torch.float32, device=db.device)
    need = workspace_size(inp.batch, inp.total_q, inp.max_tree, inp.max_seq_len, inp.num_heads, 1)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=db.device)
    if stream is None:
        stream = torch.cuda.current_stream(db.device)
    check(verify_attn_split_range(db.q_lat.data_ptr(), db.q_rope.data_ptr(), db.kv_cache.data_ptr(),
                                  db.block_table.data_ptr(), db.seq_lens.data_ptr(), db.tree_parent.data_ptr(),
                                  db.n_tree.data_ptr(), inp.scale, part_out.data_ptr(), part_lse.data_ptr(),
                                  stream.cuda_stream, inp.batch, inp.total_q, inp.max_tree, inp.max_seq_len,
                                  inp.num_heads, inp.page_size, inp.num_pages, inp.max_pages_per_seq, num_splits,
                                  split_begin, split_count, workspace.data_ptr(), workspace.numel()),
          "mla_verify_attn_split_range")
    return part_out, part_lse, workspace


def append_tree(db: "DeviceBatch", tree_kv, workspace=None, stream=None):
    """Write tree_kv (torch int16 [total_q, 576] on the device) into db.kv_cache; returns the workspace."""
    import torch
    inp = db.inp
    if workspace is None:
        workspace = torch.empty(tree_kv_workspace_size(), dtype=torch.uint8, device=db.device)
    if stream is None:
        stream = torch.cuda.current_stream(db.device)
    check(tree_kv_append(tree_kv.data_ptr(), db.kv_cache.data_ptr(), db.block_table.data_ptr(),
                         db.seq_lens.data_ptr(), db.n_tree.data_ptr(), stream.cuda_stream, inp.batch,
                         inp.total_q, inp.page_size, inp.num_pages, inp.max_pages_per_seq,
                         workspace.data_ptr(), workspace.numel()), "mla_tree_kv_append")
    return workspace


def accept_path(db: "DeviceBatch", accept_len, accept_idx, new_seq_lens=None, workspace=None, stream=None):
    """Compact the accepted paths (torch int32 device tensors) in db.kv_cache; returns
    (new_seq_lens, workspace)."""
    import torch
    inp = db.inp
    if new_seq_lens is None:
        new_seq_lens = torch.empty(inp.batch, dtype=torch.int32, device=db.device)
    if workspace is None:
        workspace = torch.empty(tree_kv_workspace_size(), dtype=torch.uint8, device=db.device)
    if stream is None:
        stream = torch.cuda.current_stream(db.device)
    check(tree_kv_accept(db.kv_cache.data_ptr(), db.block_table.data_ptr(), db.seq_lens.data_ptr(),
                         db.n_tree.data_ptr(), db.tree_parent.data_ptr(), accept_len.data_ptr(),
                         accept_idx.data_ptr(), new_seq_lens.data_ptr(), stream.cuda_stream, inp.batch,
                         inp.total_q, inp.page_size, inp.num_pages, inp.max_pages_per_seq,
                         workspace.data_ptr(), workspace.numel()), "mla_tree_kv_accept")
    return new_seq_lens, workspace


def verify_sparse(db: "DeviceBatch", topk_idx, num_splits_req: int = 0, out=None, lse=None, workspace=None,
                  stream=None):
    """Run mla_verify_sparse_attn; topk_idx is a device int32 tensor [total_q, topk].
    Returns (out, lse, workspace)."""
    import torch
    inp = db.inp
    topk = int(topk_idx.shape[1])
    if out is None:
        out = torch.empty((inp.total_q, inp.num_heads, D_LATENT), dtype=torch.float32, device=db.device)
    if lse is None:
        lse = torch.empty((inp.total_q, inp.num_heads), dtype=torch.float32, device=db.device)
    need = sparse_workspace_size(inp.batch, inp.total_q, inp.max_tree, topk, inp.num_heads, num_splits_req)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=db.device)
    if stream is None:
        stream = torch.cuda.current_stream(db.device)
    check(verify_sparse_attn(db.q_lat.data_ptr(), db.q_rope.data_ptr(), db.kv_cache.data_ptr(),
                             db.block_table.data_ptr(), db.seq_lens.data_ptr(), db.tree_parent.data_ptr(),
                             db.n_tree.data_ptr(), topk_idx.data_ptr(), topk, inp.scale, out.data_ptr(),
                             lse.data_ptr(), stream.cuda_stream, inp.batch, inp.total_q, inp.max_tree,
                             inp.max_seq_len, inp.num_heads, inp.page_size, inp.num_pages, inp.max_pages_per_seq,
                             num_splits_req, workspace.data_ptr(), workspace.numel()), "mla_verify_sparse_attn")
    return out, lse, workspace



def verify_graph_create(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, topk_idx, topk,
                        scale, out, lse, max_batch, max_total_q, max_tree, max_seq_len, num_heads, page_size,
                        num_pages, max_pages_per_seq, num_splits, workspace, workspace_bytes, stream):
    """Raw call; returns (status, handle or None)."""
    h = ctypes.c_void_p()
    code = int(lib().mla_verify_graph_create(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree,
                                             topk_idx, topk, float(scale), out, lse, max_batch, max_total_q,
                                             max_tree, max_seq_len, num_heads, page_size, num_pages,
                                             max_pages_per_seq, num_splits, workspace, workspace_bytes, stream,
                                             ctypes.byref(h)))
    return code, (h.value if code == MLA_OK else None)


def verify_graph_launch(handle, batch, stream) -> int:
    return int(lib().mla_verify_graph_launch(handle, int(batch), stream))


def verify_graph_destroy(handle) -> int:
    return int(lib().mla_verify_graph_destroy(handle))


class VerifyGraph:
    """A verify step captured once for a bucket of at most `max_batch` requests
    and `max_total_q` tree tokens over one paged KV cache (mla_verify_graph_*).

    It owns the bucket's input and output buffers on the device: `load()`
    copies one step's inputs (a VerifyInputs over the same cache) into them,
    `launch()` replays the graph, padding the requests past the step's batch.
    `out` / `lse` rows past the step's tree tokens are not defined."""

    def __init__(self, kv_cache, max_batch, max_total_q, max_tree, max_seq_len, page_size, max_pages_per_seq,
                 scale, topk=0, num_splits_req=0, stream=None):
        import torch
        dev = kv_cache.device
        self.device = dev
        self.max_batch, self.max_total_q, self.topk = int(max_batch), int(max_total_q), int(topk)
        self.kv_cache = kv_cache
        self.q_lat = torch.zeros((max_total_q, NUM_HEADS, D_LATENT), dtype=torch.int16, device=dev)
        self.q_rope = torch.zeros((max_total_q, NUM_HEADS, D_ROPE), dtype=torch.int16, device=dev)
        self.block_table = torch.full((max_batch, max_pages_per_seq), -1, dtype=torch.int32, device=dev)
        self.seq_lens = torch.zeros(max_batch, dtype=torch.int32, device=dev)
        self.n_tree = torch.zeros(max_batch, dtype=torch.int32, device=dev)
        self.tree_parent = torch.full((max_total_q,), -1, dtype=torch.int32, device=dev)
        self.topk_idx = (torch.full((max_total_q, topk), -1, dtype=torch.int32, device=dev) if topk
                         else None)
        self.out = torch.empty((max_total_q, NUM_HEADS, D_LATENT), dtype=torch.float32, device=dev)
        self.lse = torch.empty((max_total_q, NUM_HEADS), dtype=torch.float32, device=dev)
        if topk:
            need = sparse_workspace_size(max_batch, max_total_q, max_tree, topk, NUM_HEADS, num_splits_req)
        else:
            need = workspace_size(max_batch, max_total_q, max_tree, max_seq_len, NUM_HEADS, num_splits_req)
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        page_rows = int(kv_cache.shape[0])
        code, self.handle = verify_graph_create(
            self.q_lat.data_ptr(), self.q_rope.data_ptr(), kv_cache.data_ptr(), self.block_table.data_ptr(),
            self.seq_lens.data_ptr(), self.tree_parent.data_ptr(), self.n_tree.data_ptr(),
            self.topk_idx.data_ptr() if topk else None, self.topk, scale, self.out.data_ptr(),
            self.lse.data_ptr(), self.max_batch, self.max_total_q, max_tree, max_seq_len, NUM_HEADS, page_size,
            page_rows, max_pages_per_seq, num_splits_req, self.workspace.data_ptr(), self.workspace.numel(),
            self.stream.cuda_stream)
        check(code, "mla_verify_graph_create")
        self.batch = 0
        self.total_q = 0

    def load(self, inp, topk_idx=None, non_blocking=False) -> None:
        """Copy one step's inputs (host VerifyInputs over the graph's cache) into the buffers."""
        import numpy as np
        import torch
        if inp.batch > self.max_batch or inp.total_q > self.max_total_q:
            raise ValueError("step exceeds the graph's bucket")
        if inp.max_pages_per_seq > self.block_table.shape[1]:
            raise ValueError("block table wider than the graph's")

        def put(dst, a, dtype):
            src = torch.from_numpy(np.ascontiguousarray(a).view(dtype))
            dst.copy_(src.reshape(dst.shape), non_blocking=non_blocking)
        nq, b = inp.total_q, inp.batch
        with torch.cuda.stream(self.stream):
            put(self.q_lat[:nq], inp.q_lat, np.int16)
            put(self.q_rope[:nq], inp.q_rope, np.int16)
            self.block_table[:b].fill_(-1)
            put(self.block_table[:b, :inp.max_pages_per_seq], inp.block_table, np.int32)
            put(self.seq_lens[:b], inp.seq_lens, np.int32)
            put(self.n_tree[:b], inp.n_tree, np.int32)
            put(self.tree_parent[:nq], inp.tree_parent, np.int32)
            if self.topk:
                put(self.topk_idx[:nq], topk_idx, np.int32)
        self.batch, self.total_q = b, nq

    def launch(self, batch=None) -> None:
        check(verify_graph_launch(self.handle, self.batch if batch is None else batch, self.stream.cuda_stream),
              "mla_verify_graph_launch")

    def close(self) -> None:
        if self.handle is not None:
            check(verify_graph_destroy(self.handle), "mla_verify_graph_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
