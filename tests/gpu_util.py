"""Helpers for the GPU parity tests: padded device copies and the comparison rule."""
import numpy as np

from oracle import wq_oracle as O


def dev_matrix(torch, arr, ld=None, device="cuda"):
    """Copy a 2-D numpy array to the GPU inside a buffer whose row stride is
    ``ld`` elements (>= the row width); returns the [rows, cols] view."""
    arr = np.ascontiguousarray(arr)
    rows, cols = arr.shape
    ld = cols if ld is None else ld
    t = torch.from_numpy(arr)
    buf = torch.zeros((rows, ld), dtype=t.dtype, device=device)
    buf[:, :cols] = t.to(device)
    return buf[:, :cols]


def dev_empty(torch, rows, cols, dtype, ld=None, fill=None, device="cuda"):
    ld = cols if ld is None else ld
    buf = torch.empty((rows, ld), dtype=dtype, device=device)
    if fill is not None:
        buf.fill_(fill)
    return buf[:, :cols]


def assert_gemm_close(y_gpu, y_ref, dtype, rel=5e-3):
    """max|y - y_ref| <= rel * max|y_ref| + 1 ulp(dtype) at y_ref, element-wise."""
    y = y_gpu.float().cpu().numpy().astype(np.float64) if hasattr(y_gpu, "cpu") else np.asarray(y_gpu, np.float64)
    tol = O.gemm_tolerance(y_ref, dtype, rel)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert np.isfinite(y).all(), "non-finite output"
    assert not bad.any(), (f"{int(bad.sum())} / {bad.size} outside tolerance; worst err {err.max():.3e} "
                           f"vs tol {tol.reshape(-1)[np.argmax(err)]:.3e}, max|ref| {np.abs(y_ref).max():.3e}")
