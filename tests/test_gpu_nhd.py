"""GPU parity of every entry point on NHD pools ([page][slot][head][dim], the
token-before-head layout of the post's figure on NHD and HND KV-cache layouts)
against the fp64 oracle reading the same NHD pools.

The pools come from the seeded HND generators with their head and slot axes
swapped (workloads.to_nhd), so each case holds the values of an HND case; the
oracle's NHD reading is pinned to its HND reading on the CPU. Tolerances as for
HND: o within 1e-4 (fp32) / 1e-2 (bf16), lse within 1e-3, copies bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import DevCase, compare, dev_tensor, host_f64, LSE_TOL


def _bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def _host_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("hq,hkv,d,p,dtype,kv", [
    (8, 8, 64, 16, wl.F32, [17, 64, 100, 255]),        # no grouping
    (32, 8, 128, 16, wl.BF16, [4000, 17, 900, 2, 1000]),  # GQA 4, split-KV (few requests)
    (8, 1, 64, 16, wl.BF16, [300, 31, 1]),             # one KV head: NHD rows are contiguous
    (12, 2, 64, 1, wl.F32, [5, 40, 1]),                # one token per page
    (16, 2, 128, 64, wl.BF16, [700, 64, 65]),          # group 8, page 64
])
def test_split_kv_decode_on_nhd_pools(hq, hkv, d, p, dtype, kv):
    case = wl.to_nhd(wl.make_attn_case(401, [1] * len(kv), kv, hq, hkv, d, p, dtype))
    dc = DevCase(case)
    o, lse = pd.pd_attn_decode(dc.q, dc.k_pool, dc.v_pool, dc.kv_len, dc.page_indptr, dc.page_indices,
                               max_kv_len=dc.max_kv_len, layout="NHD")
    torch.cuda.synchronize()
    assert pd.pd_last_kernel() == "decode_kernel"
    o_ref, lse_ref = oracle.attention_case(case)
    compare(o, lse, o_ref, lse_ref, dtype)


def test_tensor_core_decode_batch_on_nhd_pools():
    # the 128-request GQA decode batch: the packed tensor-core path, NHD tiles by TMA
    case = wl.to_nhd(wl.decode_batch())
    dc = DevCase(case)
    o, lse = pd.pd_attn_decode(dc.q, dc.k_pool, dc.v_pool, dc.kv_len, dc.page_indptr, dc.page_indices,
                               max_kv_len=4096, layout="NHD")
    torch.cuda.synchronize()
    assert pd.pd_last_kernel() == "prefill_kernel"
    o_ref, lse_ref = oracle.attention_case(case)
    err_o, err_l = compare(o, lse, o_ref, lse_ref, case.dtype)
    assert err_o < 1e-2 and err_l < 1e-3


def test_decode_results_do_not_depend_on_the_layout():
    # the same values in both layouts give bit-identical outputs on each path
    for kv in ([4000, 17, 900, 2, 1000], list(range(1, 1300, 9))):
        hnd = wl.make_attn_case(402, [1] * len(kv), kv, 32, 8, 128, 16, wl.BF16)
        outs = []
        for case in (hnd, wl.to_nhd(hnd)):
            dc = DevCase(case)
            o, lse = pd.pd_attn_decode(dc.q, dc.k_pool, dc.v_pool, dc.kv_len, dc.page_indptr, dc.page_indices,
                                       max_kv_len=dc.max_kv_len, layout=case.layout)
            torch.cuda.synchronize()
            outs.append((o.cpu(), lse.cpu(), pd.pd_last_kernel()))
        assert outs[0][2] == outs[1][2]
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


# -------------------------------------------------------- prefill and mixed

def _check_attn(case, o, lse):
    o_ref, lse_ref = oracle.attention_case(case)
    err = float(np.abs(host_f64(o) - o_ref).max())
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    lerr = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert err <= 1e-2 and lerr <= LSE_TOL, (err, lerr)


@pytest.mark.parametrize("qo,kv,hq,hkv,p,causal", [
    ([100], [100], 2, 2, 16, True),                  # one tile, MHA
    ([300, 5, 129], [300, 40, 200], 8, 2, 16, True),  # GQA 4 packed, ragged, bottom-right causal
    ([64, 1], [64, 513], 16, 1, 64, True),           # group 16, page 64
    ([77, 33], [150, 33], 6, 3, 8, False),           # group 2, page 8, not causal
])
def test_prefill_on_nhd_pools(qo, kv, hq, hkv, p, causal):
    case = wl.to_nhd(wl.make_attn_case(403, qo, kv, hq, hkv, 128, p, wl.BF16, causal=causal))
    dc = DevCase(case)
    o, lse = pd.pd_attn_prefill(dc.q, dc.k_pool, dc.v_pool, dc.kv_len, dc.page_indptr, dc.page_indices,
                                dc.qo_indptr, causal=causal, max_qo_len=dc.max_qo_len, max_kv_len=dc.max_kv_len,
                                o_dtype=torch.float32, layout="NHD")
    torch.cuda.synchronize()
    _check_attn(case, o, lse)


def test_mixed_batch_on_nhd_pools():
    # one prefill of 257 rows and 20 decodes, GQA 4, in one launch
    rng = np.random.default_rng(404)
    kv = [257] + list(rng.integers(1, 600, size=20))
    case = wl.to_nhd(wl.make_attn_case(404, [257] + [1] * 20, kv, 16, 4, 128, 16, wl.BF16))
    dc = DevCase(case)
    o, lse = pd.pd_attn_mixed(dc.q, dc.k_pool, dc.v_pool, dc.kv_len, dc.page_indptr, dc.page_indices, dc.qo_indptr,
                              max_qo_len=dc.max_qo_len, max_kv_len=dc.max_kv_len, o_dtype=torch.float32,
                              layout="NHD")
    torch.cuda.synchronize()
    _check_attn(case, o, lse)


# ---------------------------------------------------------------- copies

@pytest.mark.parametrize("args", [
    dict(seed=405, qo=[5, 1, 16, 33], kv=[9, 30, 16, 40], hkv=4, d=128, p=16, dt=wl.BF16),
    dict(seed=406, qo=[3, 7], kv=[3, 11], hkv=2, d=64, p=1, dt=wl.F32),
    dict(seed=407, qo=[20, 1, 1], kv=[70, 64, 65], hkv=3, d=64, p=64, dt=wl.BF16),
    dict(seed=409, qo=[7, 19, 1], kv=[40, 19, 33], hkv=3, d=96, p=16, dt=wl.BF16),
])
def test_append_into_nhd_pools(args):
    case = wl.to_nhd(wl.make_attn_case(args["seed"], args["qo"], args["kv"], args["hkv"], args["hkv"], args["d"],
                                       args["p"], args["dt"], with_new_tokens=True, num_pages=40))
    dc = DevCase(case)
    pd.pd_kv_append(dc.k_new, dc.v_new, dc.k_pool, dc.v_pool, dc.qo_indptr, dc.kv_len, dc.page_indptr,
                    dc.page_indices, max_kv_len=dc.max_kv_len, layout="NHD")
    k, v = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.qo_indptr, case.kv_len, case.table.page_indptr, case.table.page_indices,
                     case.k_new, case.v_new, k, v, layout=oracle.NHD)
    np.testing.assert_array_equal(_bits(dc.k_pool), _host_bits(k))
    np.testing.assert_array_equal(_bits(dc.v_pool), _host_bits(v))


@pytest.mark.parametrize("src_layout,dst_layout,head_dim", [("NHD", "NHD", 64), ("HND", "NHD", 64), ("NHD", "HND", 64),
                                                          ("NHD", "NHD", 96)])
def test_handoff_between_layouts(src_layout, dst_layout, head_dim):
    # pack from one layout, unpack into a page-64 pool of the other: the packed
    # block format does not depend on either pool's layout (head_dim 96: rows
    # of 12 sixteen-byte vectors, NHD rows found by division)
    hc = wl.kv_handoff(seed=408, batch=3, layers=3, heads=4, head_dim=head_dim, src_page=16, dst_page=64,
                       dtype=wl.BF16, kv_lens=[100, 17, 64], src_slack=5, dst_slack=2)
    src = wl.to_nhd(hc) if src_layout == "NHD" else hc
    L, H, D = hc.num_layers, hc.num_kv_heads, hc.head_dim
    kv_len = dev_tensor(hc.kv_len.astype(np.int32))
    s_ptr, s_idx = dev_tensor(hc.src_table.page_indptr), dev_tensor(hc.src_table.page_indices)
    d_ptr, d_idx = dev_tensor(hc.dst_table.page_indptr), dev_tensor(hc.dst_table.page_indices)
    offs = dev_tensor(hc.dst_offsets)
    total = wl.packed_bytes(hc.kv_len, L, H, D, 2)
    buf = torch.zeros(total, dtype=torch.uint8, device="cuda")
    pd.pd_kv_pack(dev_tensor(src.k_src), dev_tensor(src.v_src), kv_len, s_ptr, s_idx, buf, offs, max_kv_len=100,
                  layout=src_layout)
    hnd_shape = (L, hc.dst_table.num_pages, H, 64, D)
    poison = wl._poison(hnd_shape, hc.dtype)
    if dst_layout == "NHD":
        poison = wl.nhd_pool(poison)
    k_dst, v_dst = dev_tensor(poison), dev_tensor(poison)
    pd.pd_kv_unpack(buf, offs, k_dst, v_dst, kv_len, d_ptr, d_idx, max_kv_len=100, layout=dst_layout)
    torch.cuda.synchronize()
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, src.k_src, src.v_src,
                         hc.dst_offsets, total, layout=src_layout)
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
    k_ref, v_ref = poison.copy(), poison.copy()
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, ref, hc.dst_offsets,
                     k_ref, v_ref, layout=dst_layout)
    np.testing.assert_array_equal(_bits(k_dst), _host_bits(k_ref))
    np.testing.assert_array_equal(_bits(v_dst), _host_bits(v_ref))


def test_head_range_pack_from_nhd_pools():
    # heads [1, 3) of a 4-head NHD pool (a TP2 shard's half of the heads)
    hc = wl.to_nhd(wl.kv_handoff(seed=409, batch=2, layers=2, heads=4, head_dim=128, src_page=16, dst_page=64,
                                 dtype=wl.BF16, kv_lens=[90, 33]))
    L, D = hc.num_layers, hc.head_dim
    part = wl.packed_bytes(hc.kv_len, L, 2, D, 2)
    offs = np.array([0, wl.packed_bytes(hc.kv_len[:1], L, 2, D, 2)], np.int64)
    buf = torch.zeros(part, dtype=torch.uint8, device="cuda")
    pd.pd_kv_pack_heads(dev_tensor(hc.k_src), dev_tensor(hc.v_src), dev_tensor(hc.kv_len.astype(np.int32)),
                        dev_tensor(hc.src_table.page_indptr), dev_tensor(hc.src_table.page_indices), buf,
                        dev_tensor(offs), 1, 2, max_kv_len=90, layout="NHD")
    torch.cuda.synchronize()
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         offs, part, head_begin=1, head_count=2, layout=oracle.NHD)
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)


def test_layer_range_packs_from_nhd_pools():
    # layers [0, 1) then [1, 3) of a 3-layer NHD handoff into one buffer equal the
    # oracle's whole pack; ragged lengths below max_kv_len leave token units idle
    hc = wl.to_nhd(wl.kv_handoff(seed=411, batch=3, layers=3, heads=5, head_dim=64, src_page=16, dst_page=64,
                                 dtype=wl.BF16, kv_lens=[77, 16, 130]))
    L, H, D = hc.num_layers, hc.num_kv_heads, hc.head_dim
    total = wl.packed_bytes(hc.kv_len, L, H, D, 2)
    offs = np.zeros(len(hc.kv_len), np.int64)
    for r in range(1, len(hc.kv_len)):
        offs[r] = offs[r - 1] + wl.packed_bytes(hc.kv_len[r - 1:r], L, H, D, 2)
    buf = torch.zeros(total, dtype=torch.uint8, device="cuda")
    args = (dev_tensor(hc.k_src), dev_tensor(hc.v_src), dev_tensor(hc.kv_len.astype(np.int32)),
            dev_tensor(hc.src_table.page_indptr), dev_tensor(hc.src_table.page_indices), buf, dev_tensor(offs))
    pd.pd_kv_pack_layers(*args, 0, 1, max_kv_len=200, layout="NHD")
    pd.pd_kv_pack_layers(*args, 1, 2, max_kv_len=200, layout="NHD")
    torch.cuda.synchronize()
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         offs, total, layout=oracle.NHD)
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
