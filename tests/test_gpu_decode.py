"""GPU parity of pd_attn_decode against the fp64 oracle (same seeded inputs).

Tolerances stated for this path: max |o - oracle| <= 1e-4 for fp32
inputs, <= 1e-2 for bf16 inputs (fp32 accumulation), |lse - oracle| <= 1e-3.
Unused pool pages and tail slots hold NaN, so a stray read shows up."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import DevCase, compare


def run_decode(case, o_dtype=None, status=None):
    d = DevCase(case)
    odt = None if o_dtype is None else {wl.F32: torch.float32, wl.BF16: torch.bfloat16}[o_dtype]
    o, lse = pd.pd_attn_decode(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices,
                               sm_scale=case.sm_scale, max_kv_len=d.max_kv_len, o_dtype=odt,
                               dev_status=status)
    torch.cuda.synchronize()
    return o, lse


def check(case, o_dtype=None):
    o, lse = run_decode(case, o_dtype)
    o_ref, lse_ref = oracle.attention_case(case)
    return compare(o, lse, o_ref, lse_ref, case.dtype)


def test_decode_correctness_workload_fp32():
    # 4 requests, kv_len {17, 64, 100, 255}, 8 heads, D 64, page 16, fp32, 64-page pool
    check(wl.decode_correctness())


def test_decode_batch_workload_bf16_full():
    # 128 requests, kv_len U[512, 4096], GQA 32/8, D 128, page 16, bf16: every output row
    case = wl.decode_batch()
    err_o, err_l = check(case)
    assert err_o < 1e-2 and err_l < 1e-3


@pytest.mark.parametrize("o_dtype", [wl.F32, wl.BF16])
def test_decode_output_dtypes(o_dtype):
    case = wl.make_attn_case(101, [1] * 5, [1, 16, 17, 300, 700], 16, 4, 128, 16, wl.BF16, num_pages=80)
    check(case, o_dtype)


@pytest.mark.parametrize("hq,hkv,d,p,dtype", [
    (8, 8, 64, 16, wl.F32),      # no grouping
    (8, 1, 64, 16, wl.BF16),     # group 8, eight heads per item
    (32, 4, 128, 16, wl.BF16),   # group 8, two items of four heads
    (10, 2, 128, 16, wl.BF16),   # group 5, one head per item
    (12, 2, 64, 16, wl.F32),     # group 6, two heads per item
    (4, 2, 128, 1, wl.BF16),     # one token per page
    (4, 2, 128, 3, wl.F32),      # page size not a power of two
    (4, 1, 64, 64, wl.BF16),     # large pages
    (2, 1, 128, 128, wl.F32),    # pages longer than a chunk's stage
])
def test_decode_shapes(hq, hkv, d, p, dtype):
    rng = np.random.default_rng(hq * 1000 + p)
    kv = rng.integers(1, 1500, size=7)
    kv[0], kv[1] = 1, 513
    case = wl.make_attn_case(int(hq + d + p), [1] * 7, kv, hq, hkv, d, p, dtype,
                             num_pages=int(np.sum(-(-kv // p))) + 5)
    check(case)


def test_decode_empty_and_single_key_requests():
    # causal is irrelevant for one row per request; the oracle rejects a causal row with no key
    case = wl.make_attn_case(102, [1] * 4, [0, 1, 0, 33], 4, 2, 128, 16, wl.BF16, num_pages=8, causal=False)
    o, lse = run_decode(case)
    o_ref, lse_ref = oracle.attention_case(case)
    compare(o, lse, o_ref, lse_ref, case.dtype)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_decode_custom_scale_and_long_context():
    case = wl.make_attn_case(103, [1, 1], [16384, 5000], 8, 2, 128, 16, wl.BF16, sm_scale=0.05)
    check(case)


def test_decode_bad_page_id_is_reported_not_faulted():
    case = wl.make_attn_case(104, [1, 1], [40, 40], 4, 2, 64, 16, wl.F32, num_pages=6)
    case.table.page_indices[1] = 1000          # out of range for request 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = run_decode(case, status=status)
    assert int(status.item()) == 3
    # request 1 is unaffected
    first = int(case.table.page_indptr[1])
    o_ref, lse_ref = oracle.attention([0, 1], case.kv_len[1:], [0, int(case.table.page_indptr[2]) - first],
                                      case.table.page_indices[first:], case.q[1:], case.k_pool, case.v_pool, 4, 2,
                                      case.scale)
    np.testing.assert_allclose(o[1].cpu().numpy(), o_ref[0], atol=1e-4)


def test_decode_length_above_bound_is_reported():
    case = wl.make_attn_case(105, [1, 1], [40, 20], 4, 2, 64, 16, wl.F32, num_pages=6)
    d = DevCase(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pd.pd_attn_decode(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices, max_kv_len=30,
                      dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2


def test_decode_is_deterministic():
    case = wl.make_attn_case(106, [1] * 9, [900] * 9, 32, 8, 128, 16, wl.BF16)
    a, la = run_decode(case)
    b, lb = run_decode(case)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_decode_many_requests_with_empty_ones():
    # more requests than the planner's block of threads; every 97th request has
    # no cached key (o = 0, lse = -inf) and the rest mix one- and many-chunk splits
    rng = np.random.default_rng(107)
    kv = rng.integers(1, 700, size=1300)
    kv[::97] = 0
    case = wl.make_attn_case(107, [1] * 1300, kv, 4, 2, 64, 16, wl.F32, causal=False)
    o, lse = run_decode(case)
    empty = torch.from_numpy(kv == 0).cuda()
    assert torch.all(o[empty] == 0) and torch.all(torch.isneginf(lse[empty]))
    o_ref, lse_ref = oracle.attention_case(case)
    compare(o, lse, o_ref, lse_ref, case.dtype)


def test_large_gqa_batch_runs_packed_on_tensor_cores_and_others_split():
    # the decode batch (128 requests x 8 KV heads) goes through the tensor-core
    # kernel with 4 query heads per tile; a small batch and an MHA batch keep the
    # split-KV kernel; all three match the oracle
    big = wl.decode_batch()
    check(big)
    assert pd.pd_last_kernel() == "prefill_kernel"
    small = wl.make_attn_case(108, [1] * 6, [4000, 17, 900, 2, 4096, 1000], 32, 8, 128, 16, wl.BF16)
    check(small)
    assert pd.pd_last_kernel() == "decode_kernel"
    mha = wl.make_attn_case(109, [1] * 80, np.arange(80) * 7 + 1, 40, 40, 128, 16, wl.BF16)
    check(mha)
    assert pd.pd_last_kernel() == "decode_kernel"


def test_tensor_core_decode_with_empty_and_short_requests():
    # enough (request, KV head) pairs for the tensor-core path, with requests of
    # no, one and a few keys among long ones
    rng = np.random.default_rng(110)
    kv = rng.integers(1, 3000, size=160)
    kv[::13] = 0
    kv[1::17] = 1
    case = wl.make_attn_case(110, [1] * 160, kv, 32, 8, 128, 16, wl.BF16, causal=False)
    o, lse = run_decode(case)
    assert pd.pd_last_kernel() == "prefill_kernel"
    empty = torch.from_numpy(kv == 0).cuda()
    assert torch.all(o[empty] == 0) and torch.all(torch.isneginf(lse[empty]))
    o_ref, lse_ref = oracle.attention_case(case)
    compare(o, lse, o_ref, lse_ref, case.dtype)


@pytest.mark.parametrize("big", [False, True])
def test_binding_replaces_a_workspace_that_is_too_small(big):
    # the binding passes the caller's workspace straight through; when the call
    # reports it too small, it retries with one of pd_attn_workspace_size bytes
    case = wl.decode_batch() if big else wl.make_attn_case(111, [1] * 6, [4000, 17, 900, 2, 4096, 1000],
                                                          32, 8, 128, 16, wl.BF16)
    d = DevCase(case)
    tiny = torch.empty(16, dtype=torch.uint8, device="cuda")
    o, lse = pd.pd_attn_decode(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices,
                               sm_scale=case.sm_scale, max_kv_len=d.max_kv_len, workspace=tiny)
    torch.cuda.synchronize()
    assert pd.pd_last_kernel() == ("prefill_kernel" if big else "decode_kernel")
    o_ref, lse_ref = oracle.attention_case(case)
    compare(o, lse, o_ref, lse_ref, case.dtype)
