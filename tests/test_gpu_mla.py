"""GPU parity of pd_mla_decode (MLA decode over a paged latent cache, tcgen05
path) against the fp64 oracle on the same seeded bf16 inputs.

Tolerances as for bf16 attention: max |o - oracle| <= 1e-2 (fp32 accumulation),
|lse - oracle| <= 1e-3, on fp32 and bf16 outputs alike. Unused pool slots hold
NaN, so a stray read shows up."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import dev_tensor, host_f64, LSE_TOL


def run_mla(c, o_dtype=None, status=None, workspace=None):
    q, pool = dev_tensor(c.q), dev_tensor(c.kv_pool)
    kv = dev_tensor(c.kv_len.astype(np.int32))
    ptr, idx = dev_tensor(c.table.page_indptr), dev_tensor(c.table.page_indices)
    o, lse = pd.pd_mla_decode(q, pool, kv, ptr, idx, kv_lora_rank=c.d_c, sm_scale=c.sm_scale,
                              max_kv_len=int(c.kv_len.max()) if len(c.kv_len) else 0, o_dtype=o_dtype,
                              dev_status=status, workspace=workspace)
    torch.cuda.synchronize()
    return o, lse


def check(c, o, lse, sel=None):
    if sel is None:
        o_ref, lse_ref = oracle.mla_decode(c.kv_len, c.table.page_indptr, c.table.page_indices, c.q, c.kv_pool,
                                           c.d_c, c.sm_scale)
        got, lg = host_f64(o), lse.cpu().numpy().astype(np.float64)
    else:
        sr, sh = sel
        o_ref, lse_ref = oracle.mla_decode(c.kv_len, c.table.page_indptr, c.table.page_indices, c.q, c.kv_pool,
                                           c.d_c, c.sm_scale, sel_req=sr, sel_head=sh)
        got, lg = host_f64(o)[sr, sh], lse.cpu().numpy().astype(np.float64)[sr, sh]
    assert np.isfinite(got).all(), "non-finite output"
    diff = np.abs(got - o_ref)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    lerr = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert float(diff.max()) <= 1e-2, f"max |o - oracle| = {diff.max()}"
    assert lerr <= LSE_TOL, lerr
    return float(diff.max()), lerr


def test_mla_small_all_heads():
    # lengths around the 32- and 64-token edges, and one request split into chunks
    c = wl.mla_case(501, [1, 31, 32, 33, 63, 64, 65, 700], num_qo_heads=128, page_size=64)
    o, lse = run_mla(c)
    assert pd.pd_last_kernel() == "mla_decode_kernel"
    check(c, o, lse)


@pytest.mark.parametrize("hq,page,kv", [
    (16, 16, [0, 1, 17, 1500, 64, 513]),     # TP8 shape: 16 heads; an empty request
    (128, 16, [1025, 2, 300]),               # two boxes per column chunk
    (64, 256, [600, 255, 256, 257]),         # big pages
    (1, 32, [100, 3000]),                    # one head, padded to the 128-row tile
])
def test_mla_shapes(hq, page, kv):
    c = wl.mla_case(502, kv, num_qo_heads=hq, page_size=page)
    o, lse = run_mla(c)
    check(c, o, lse)
    empty = torch.from_numpy(c.kv_len == 0).cuda()
    assert torch.all(o[empty] == 0) and torch.all(torch.isneginf(lse[empty]))


def test_mla_fp32_output():
    c = wl.mla_case(503, [90, 1200, 7], num_qo_heads=32, page_size=64)
    o, lse = run_mla(c, o_dtype=torch.float32)
    assert o.dtype == torch.float32
    check(c, o, lse)


def test_mla_decode_batch_sampled():
    # the MLA decode batch: 128 requests, kv_len U[512, 4096], 128 heads, page 64;
    # every output is checked finite, 512 sampled (request, head) pairs against the oracle
    c = wl.mla_decode_batch()
    o, lse = run_mla(c)
    rng = np.random.default_rng(504)
    sr = rng.integers(0, c.batch_size, size=512)
    sh = rng.integers(0, c.num_qo_heads, size=512)
    sr[:128] = np.arange(128)                       # every request at least once
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    check(c, o, lse, sel=(sr, sh))


def test_mla_many_short_requests():
    # more requests than the planner's block of threads
    rng = np.random.default_rng(505)
    kv = rng.integers(0, 200, size=1100)
    c = wl.mla_case(505, kv, num_qo_heads=16, page_size=16)
    o, lse = run_mla(c)
    check(c, o, lse)
    o32, lse32 = run_mla(c, o_dtype=torch.float32)   # the computation alone, within 1e-2
    check(c, o32, lse32)


def test_mla_bad_page_id_is_reported_not_faulted():
    c = wl.mla_case(506, [40, 70], num_qo_heads=16, page_size=16)
    c.table.page_indices[1] = c.table.num_pages + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_mla(c, status=status)
    assert int(status.item()) == 3  # PD_DEV_BAD_PAGE_TABLE


def test_mla_is_deterministic():
    c = wl.mla_case(507, [3000, 100, 1800], num_qo_heads=128, page_size=64)
    o1, l1 = run_mla(c)
    o2, l2 = run_mla(c)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mla_workspace_too_small_is_replaced():
    c = wl.mla_case(508, [700, 5], num_qo_heads=16, page_size=64)
    o, lse = run_mla(c, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    check(c, o, lse)
