"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the fp64 oracle at the tolerances of the verify-attention task
(max |out err| <= 1e-2, mean |out err| <= 1e-3, max |lse err| <= 1e-3)."""
import numpy as np

TOL_OUT_MAX = 1e-2
TOL_OUT_MEAN = 1e-3
TOL_LSE_MAX = 1e-3

_ready = False


def ensure_gpu():
    global _ready
    import torch

    from mla_speculative_decoding_verify_gb300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if not _ready:
        torch.cuda.set_device(0)
        binding.init(0)
        _ready = True


def run_gpu(inp, splits=0, **kw):
    """(out [total_q, H, 512] float64, lse [total_q, H] float64, device status bits)."""
    import torch

    from mla_speculative_decoding_verify_gb300 import binding
    ensure_gpu()
    db = binding.DeviceBatch(inp, "cuda:0")
    out, lse, ws = binding.verify(db, num_splits_req=splits, **kw)
    torch.cuda.synchronize()
    status = binding.read_status(ws.data_ptr())
    return (out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), status)


def errors(out, lse, ref_out, ref_lse):
    """(max |out err|, mean |out err|, max |lse err|); -inf lse must match exactly."""
    out = np.asarray(out, dtype=np.float64).reshape(ref_out.shape)
    lse = np.asarray(lse, dtype=np.float64).reshape(ref_lse.shape)
    inf_ref = np.isneginf(ref_lse)
    assert np.array_equal(inf_ref, np.isneginf(lse)), "rows with no visible key differ"
    e_o = np.abs(out - ref_out)
    e_l = np.abs(lse[~inf_ref] - ref_lse[~inf_ref])
    return (float(e_o.max()) if e_o.size else 0.0, float(e_o.mean()) if e_o.size else 0.0,
            float(e_l.max()) if e_l.size else 0.0)


def assert_close(out, lse, ref_out, ref_lse, what=""):
    mx, mean, le = errors(out, lse, ref_out, ref_lse)
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    assert mx <= TOL_OUT_MAX and mean <= TOL_OUT_MEAN and le <= TOL_LSE_MAX, (
        f"{what}: max|out| {mx:.3e} mean|out| {mean:.3e} max|lse| {le:.3e}")
    return mx, mean, le
