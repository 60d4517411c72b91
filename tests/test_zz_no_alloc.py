"""GPU test of pd_attn_decode_static, the decode entry point that needs no
workspace from the caller (its scratch is a fixed array inside the library),
for callers that cannot allocate device memory themselves.

Called through the C ABI on two batches in a row: a large grouped-query batch
that runs on the tensor-core kernel, then a smaller one that runs the split-KV
kernel with its partial results in the array, so that anything the first call
left in the shared scratch array would show up in the second. Each result must
be bit-identical to pd_attn_decode with a workspace of its own (the same
kernels on the same plan) and within the stated tolerances of the fp64 oracle.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    import oracle
    from gpu_util import DevCase, compare


def _static_fn():
    lib = pd.load_library()
    fn = lib.pd_attn_decode_static
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(pd.AttnDesc), ctypes.POINTER(pd.Batch), P, P, P, P, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def _run_static(d: "DevCase", max_kv_len: int):
    desc = pd.make_attn_desc(d.q, d.k_pool)
    batch = pd.make_batch(d.kv_len, d.page_indptr, d.page_indices, d.k_pool.shape[0],
                          total_qo=d.q.shape[0], max_kv_len=max_kv_len)
    o = torch.full_like(d.q, float("nan"))
    lse = torch.full(d.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _static_fn()(ctypes.byref(desc), ctypes.byref(batch), d.q.data_ptr(), d.k_pool.data_ptr(),
                      d.v_pool.data_ptr(), o.data_ptr(), lse.data_ptr(), status.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, o, lse, int(status.item())


def _case(seed, n, kv_hi, hq=32, hkv=8):
    kv = np.random.default_rng(seed).integers(1, kv_hi + 1, size=n)
    return wl.make_attn_case(seed, [1] * n, kv, hq, hkv, 128, 16, wl.BF16)


def test_static_decode_matches_workspace_decode_twice():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    big = -(-4 * sms // 8) + 8                      # (request, KV head) pairs above 4 per SM
    cases = [(_case(901, big, 1500), "prefill_kernel"),            # tensor-core path
             (_case(902, 37, 2500, hq=16, hkv=4), "decode_kernel")]  # split-KV path
    for case, kernel in cases:              # two calls in a row, different batches and paths
        d = DevCase(case)
        ref_o, ref_lse = pd.pd_attn_decode(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices,
                                           max_kv_len=d.max_kv_len)
        torch.cuda.synchronize()
        assert pd.pd_last_kernel() == kernel
        rc, o, lse, status = _run_static(d, d.max_kv_len)
        assert rc == pd.PD_OK and status == 0
        assert pd.pd_last_kernel() == kernel
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
        o_ref, lse_ref = oracle.attention_case(case)
        compare(o, lse, o_ref, lse_ref, wl.BF16)


def test_static_decode_rejects_batch_beyond_scratch():
    # A bound of 4M tokens per request makes the split plan far larger than the fixed scratch.
    d = DevCase(_case(903, 2, 64))
    rc, _, _, _ = _run_static(d, 65536 * 64)
    assert rc == pd.PD_ERR_WORKSPACE
