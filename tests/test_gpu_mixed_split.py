"""GPU parity of pd_attn_mixed_split (the prefill requests of a mixed batch on
the tensor-core kernel and its decode requests on the split-KV kernel, at the
same time on disjoint SM partitions) against the fp64 oracle, and bit-identity
with the same two parts launched one after the other on the caller's stream
(the same kernels on the same plans, only on fewer SMs each)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import DevCase, LSE_TOL, host_f64


def run_split(case, num_prefill, o_dtype=torch.float32, prefill_sms=0, status=None):
    d = DevCase(case)
    o, lse = pd.pd_attn_mixed_split(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices,
                                    d.qo_indptr, num_prefill, prefill_sms=prefill_sms, causal=case.causal,
                                    max_qo_len=d.max_qo_len, max_kv_len=d.max_kv_len, o_dtype=o_dtype,
                                    dev_status=status, layout=case.layout)
    torch.cuda.synchronize()
    return d, o, lse


def check_vs_oracle(case, o, lse, o_tol=1e-2):
    o_ref, lse_ref = oracle.attention_case(case)
    err = float(np.abs(host_f64(o) - o_ref).max())
    lerr = float(np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max())
    assert err <= o_tol and lerr <= LSE_TOL, (err, lerr)


def test_mixed_split_1p63d_workload_full():
    # one prefill of 1024 tokens + 63 decodes with kv_len U[512, 576], 40 heads, D 128, bf16
    case = wl.mixed_1p_nd()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d, ob, lseb = run_split(case, 1, torch.bfloat16, status=status)  # the call the benchmark times
    assert int(status.item()) == 0
    check_vs_oracle(case, ob, lseb)
    if pd.pd_last_kernel() != "prefill_kernel+decode_kernel":
        return  # the one-launch path ran (no green contexts here, or a CUDA tool attached)
    # the two parts one after the other on the whole GPU
    pre = int(case.qo_len[0])
    o_p, lse_p = pd.pd_attn_prefill(d.q, d.k_pool, d.v_pool, d.kv_len[:1], d.page_indptr[:2], d.page_indices,
                                    d.qo_indptr[:2], max_qo_len=pre, max_kv_len=d.max_kv_len,
                                    o_dtype=torch.bfloat16)
    o_d, lse_d = pd.pd_attn_decode(d.q, d.k_pool, d.v_pool, d.kv_len[1:], d.page_indptr[1:], d.page_indices,
                                   d.qo_indptr[1:], max_kv_len=d.max_kv_len, o_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(ob[:pre], o_p[:pre]) and torch.equal(lseb[:pre], lse_p[:pre])
    assert torch.equal(ob[pre:], o_d[pre:]) and torch.equal(lseb[pre:], lse_d[pre:])


@pytest.mark.parametrize("qo,kv,hq,hkv,n_pf,sms", [
    ([300, 77, 1, 1, 1], [300, 200, 900, 5, 128], 8, 2, 2, 0),      # GQA, two prefills then decodes
    ([512, 1, 1, 1, 1, 1], [600, 4000, 129, 1, 64, 2048], 4, 4, 1, 16),  # MHA, an explicit 16-SM partition
    ([128, 1], [128, 700], 4, 1, 1, 136),                           # the largest prefill partition
    ([1, 1, 1], [1, 129, 4000], 4, 4, 0, 0),                        # no prefill: the decode part alone
    ([512, 256], [512, 600], 4, 1, 2, 0),                           # no decode: the prefill part alone
])
def test_mixed_split_shapes(qo, kv, hq, hkv, n_pf, sms):
    case = wl.make_attn_case(501 + sum(kv), qo, kv, hq, hkv, 128, 16, wl.BF16, causal=True)
    _, o, lse = run_split(case, n_pf, prefill_sms=sms)
    check_vs_oracle(case, o, lse)


@pytest.mark.parametrize("layout,causal,o_dtype,hq,hkv", [
    ("NHD", True, torch.bfloat16, 8, 2),      # NHD pools, GQA 4, bf16 output
    ("HND", False, torch.float32, 4, 4),      # a non-causal prefill part, fp32 output
    ("HND", True, torch.bfloat16, 32, 8),     # GQA 4 with the prefill tiles packing 4 heads
])
def test_mixed_split_layouts_and_outputs(layout, causal, o_dtype, hq, hkv):
    case = wl.make_attn_case(521 + hq, [640, 129, 1, 1, 1, 1], [700, 129, 900, 17, 2048, 300], hq, hkv, 128, 16,
                             wl.BF16, causal=causal)
    if layout == "NHD":
        case = wl.to_nhd(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, o, lse = run_split(case, 2, o_dtype, status=status)
    assert int(status.item()) == 0
    assert o.dtype == o_dtype
    check_vs_oracle(case, o, lse)


def test_mixed_split_reports_a_decode_with_several_rows():
    # request 2 is in the decode part but has 3 query rows
    case = wl.make_attn_case(511, [64, 1, 3, 1], [64, 300, 300, 40], 4, 4, 128, 16, wl.BF16, causal=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_split(case, 1, status=status)
    assert int(status.item()) == 4  # PD_DEV_NOT_DECODE


def test_mixed_split_orders_after_and_before_the_callers_stream():
    # inputs written on a side stream just before the call, the output read on
    # that stream right after it: the call must order its two parts after the
    # stream's earlier work and the stream's later work after both parts
    case = wl.mixed_1p_nd()
    d = DevCase(case)
    s = torch.cuda.Stream()
    q2 = torch.zeros_like(d.q)
    o = torch.empty_like(d.q)
    with torch.cuda.stream(s):
        for _ in range(3):
            q2.copy_(d.q)
            pd.pd_attn_mixed_split(q2, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices, d.qo_indptr,
                                   1, max_qo_len=d.max_qo_len, max_kv_len=d.max_kv_len, o=o, stream=s)
            o_copy = o.clone()
            q2.zero_()
    torch.cuda.synchronize()
    o_ref, _ = oracle.attention_case(case)
    assert float(np.abs(host_f64(o_copy) - o_ref).max()) <= 1e-2
