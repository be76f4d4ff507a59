"""Helpers shared by the GPU parity tests: moving seeded numpy inputs to the
device and comparing the CUDA results with the oracle under the tolerances
|gpu - oracle| <= tol * S, S = the same sum over absolute values (1e-5 for
fp32 inputs, 1e-2 for bf16 inputs); where S = 0 the result must be exactly 0."""
import numpy as np

import oracle

TOL = {"f32": 1e-5, "bf16": 1e-2}


def dev(x, dtype="f32"):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    if x.dtype == np.int32:
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def host(t):
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def assert_within(gpu, ref, scale, tol, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    assert gpu.shape == ref.shape == scale.shape, (gpu.shape, ref.shape, scale.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    zero = scale == 0
    assert np.all(gpu[zero] == 0), f"{what}: nonzero output where the error scale is 0"
    err = np.abs(gpu - ref)
    bad = err > tol * scale
    if bad.any():
        idx = np.argwhere(bad)[:5]
        ratio = float(np.max(err[~zero] / scale[~zero]))
        raise AssertionError(f"{what}: {int(bad.sum())} of {gpu.size} elements exceed {tol}·S "
                             f"(worst err/S = {ratio:.3g}); first at {idx.tolist()}")


def oracle_spmm(csr, B, dtype, rows=None):
    """Oracle C and its error scale, for all rows or the selected ones."""
    vals = oracle.widen(csr.values, dtype)
    Bw = oracle.widen(B, dtype)
    ro, ci = csr.row_offsets, csr.col_indices
    if rows is not None:
        ro, ci, pos = oracle.select_rows(ro, ci, rows)
        vals = vals[pos]
    M = ro.size - 1
    C = oracle.spmm(M, csr.K, ro, ci, vals, Bw)
    S = oracle.spmm_error_scale(M, csr.K, ro, ci, vals, Bw)
    return C, S


def oracle_sddmm(csr, X, Y, dtype, rows=None):
    Xw, Yw = oracle.widen(X, dtype), oracle.widen(Y, dtype)
    ro, ci = csr.row_offsets, csr.col_indices
    pos = None
    if rows is not None:
        ro, ci, pos = oracle.select_rows(ro, ci, rows)
        Xw = Xw[np.asarray(rows)]
    M = ro.size - 1
    out = oracle.sddmm(M, csr.K, ro, ci, Xw, Yw)
    S = oracle.sddmm_error_scale(M, csr.K, ro, ci, Xw, Yw)
    return out, S, pos
