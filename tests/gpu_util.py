"""Helpers shared by the GPU parity tests: move a seeded case to the device and
compare the CUDA path's results with the fp64 oracle."""
import numpy as np
import torch

import workloads as wl

TOL = {wl.F32: 1e-4, wl.BF16: 1e-2}   # max abs error of o stated for this path
LSE_TOL = 1e-3


def dev_tensor(a: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays carry bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class DevCase:
    def __init__(self, case: wl.AttnCase):
        self.case = case
        self.q = dev_tensor(case.q)
        self.k_pool = dev_tensor(case.k_pool)
        self.v_pool = dev_tensor(case.v_pool)
        self.qo_indptr = dev_tensor(case.qo_indptr.astype(np.int32))
        self.kv_len = dev_tensor(case.kv_len.astype(np.int32))
        self.page_indptr = dev_tensor(case.table.page_indptr.astype(np.int32))
        self.page_indices = dev_tensor(case.table.page_indices.astype(np.int32))
        self.max_kv_len = int(case.kv_len.max()) if len(case.kv_len) else 0
        self.max_qo_len = int(np.diff(case.qo_indptr).max()) if len(case.kv_len) else 0
        if case.k_new is not None:
            self.k_new = dev_tensor(case.k_new)
            self.v_new = dev_tensor(case.v_new)


def compare(o_dev, lse_dev, o_ref, lse_ref, dtype, rows=None, heads=None):
    """Max abs errors of o and lse against the oracle, asserting the tolerances."""
    o = host_f64(o_dev)
    lse = lse_dev.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, lse = o[rows, heads], lse[rows, heads]
    assert np.isfinite(o).all(), "non-finite output"
    err_o = float(np.max(np.abs(o - o_ref))) if o.size else 0.0
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), finite)
    err_l = float(np.max(np.abs(lse[finite] - lse_ref[finite]))) if finite.any() else 0.0
    assert err_o <= TOL[dtype], f"max |o - oracle| = {err_o}"
    assert err_l <= LSE_TOL, f"max |lse - oracle| = {err_l}"
    return err_o, err_l
