"""GPU parity of pd_attn_mixed (one fused launch over prefill and decode
requests) against the fp64 oracle, and against the same batch run as separate
launches (prefill on the prefill requests, split-KV decode on the decodes)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import DevCase, LSE_TOL, host_f64


def run_mixed(case, o_dtype=torch.float32):
    d = DevCase(case)
    o, lse = pd.pd_attn_mixed(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices, d.qo_indptr,
                              causal=case.causal, max_qo_len=d.max_qo_len, max_kv_len=d.max_kv_len, o_dtype=o_dtype)
    torch.cuda.synchronize()
    return d, o, lse


def check_vs_oracle(case, o, lse, o_tol=1e-2):
    o_ref, lse_ref = oracle.attention_case(case)
    err = float(np.abs(host_f64(o) - o_ref).max())
    lerr = float(np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max())
    assert err <= o_tol and lerr <= LSE_TOL, (err, lerr)
    return err, lerr


def test_mixed_1p63d_workload_full():
    # one prefill of 1024 tokens + 63 decodes with kv_len U[512, 576], 40 heads, D 128, bf16
    case = wl.mixed_1p_nd()
    d, ob, lseb = run_mixed(case, torch.bfloat16)   # the call the benchmark times
    check_vs_oracle(case, ob, lseb)
    d, o, lse = run_mixed(case)
    check_vs_oracle(case, o, lse)
    # the same batch as separate launches: prefill request alone, decodes alone
    qo = case.qo_len
    pre_rows = int(qo[0])
    o_p, lse_p = pd.pd_attn_prefill(d.q[:pre_rows], d.k_pool, d.v_pool, d.kv_len[:1], d.page_indptr[:2],
                                    d.page_indices, d.qo_indptr[:2], max_qo_len=pre_rows, max_kv_len=pre_rows,
                                    o_dtype=torch.float32)
    o_d, lse_d = pd.pd_attn_decode(d.q[pre_rows:], d.k_pool, d.v_pool, d.kv_len[1:], d.page_indptr[1:],
                                   d.page_indices, max_kv_len=576, o_dtype=torch.float32)
    torch.cuda.synchronize()
    sep = torch.cat([o_p, o_d])
    sep_lse = torch.cat([lse_p, lse_d])
    assert float((sep - o).abs().max()) <= 2e-2
    assert float((sep_lse - lse).abs().max()) <= 2 * LSE_TOL


@pytest.mark.parametrize("qo,kv,hq,hkv", [
    ([1, 300, 1, 1, 77], [900, 300, 5, 128, 200], 8, 2),     # GQA, decodes around prefills
    ([1, 1, 1], [1, 129, 4000], 4, 4),                       # decode-only through the mixed path
    ([512, 256], [512, 600], 4, 1),                          # prefill-only, one chunked
])
def test_mixed_shapes(qo, kv, hq, hkv):
    case = wl.make_attn_case(401 + sum(kv), qo, kv, hq, hkv, 128, 16, wl.BF16, causal=True)
    _, o, lse = run_mixed(case)
    check_vs_oracle(case, o, lse)


def test_mixed_bf16_output():
    case = wl.make_attn_case(402, [128, 1, 1, 256], [128, 700, 33, 256], 4, 2, 128, 16, wl.BF16, causal=True)
    _, o, lse = run_mixed(case, torch.bfloat16)
    assert o.dtype == torch.bfloat16
    check_vs_oracle(case, o, lse)


@pytest.mark.parametrize("qo,kv,hq,hkv", [
    ([4] * 6, [700, 64, 2049, 513, 4, 1000], 32, 8),            # draft verification, GQA 4: 32 rows x 4 heads a tile
    ([2, 8, 5, 1], [300, 900, 129, 64], 32, 2),                 # GQA 16: 8 query rows x 16 heads a tile
    ([3, 7], [40, 500], 6, 2),                                  # group 3 does not divide 128: one head a tile
])
def test_multi_token_verification_decode(qo, kv, hq, hkv):
    # a speculative step verifies qo_len draft tokens per request under the
    # bottom-right causal mask; GQA groups share each KV tile
    case = wl.make_attn_case(403 + sum(kv), qo, kv, hq, hkv, 128, 16, wl.BF16, causal=True)
    _, o, lse = run_mixed(case)
    check_vs_oracle(case, o, lse)
    d = DevCase(case)
    o2, lse2 = pd.pd_attn_prefill(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices, d.qo_indptr,
                                  max_qo_len=d.max_qo_len, max_kv_len=d.max_kv_len, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(lse2, lse)
