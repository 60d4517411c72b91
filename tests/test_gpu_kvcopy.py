"""GPU parity of pd_kv_append / pd_kv_pack / pd_kv_unpack against the oracle:
bit-exact on every logical slot; slots that hold no token stay untouched."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import DevCase, dev_tensor


def _bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def _host_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


@pytest.mark.parametrize("args", [
    dict(seed=201, qo=[5, 1, 16, 33], kv=[9, 30, 16, 40], hkv=4, d=128, p=16, dt=wl.BF16),
    dict(seed=202, qo=[3, 7], kv=[3, 11], hkv=2, d=64, p=1, dt=wl.F32),
    dict(seed=203, qo=[20, 1, 1], kv=[70, 64, 65], hkv=3, d=64, p=64, dt=wl.BF16),
    # head rows of 12 and 5 sixteen-byte vectors: the copy's head index by division
    dict(seed=207, qo=[7, 19, 1], kv=[40, 19, 33], hkv=3, d=96, p=16, dt=wl.BF16),
    dict(seed=208, qo=[33, 2], kv=[50, 9], hkv=5, d=40, p=8, dt=wl.BF16),
])
def test_append_small(args):
    case = wl.make_attn_case(args["seed"], args["qo"], args["kv"], args["hkv"], args["hkv"], args["d"], args["p"],
                             args["dt"], with_new_tokens=True, num_pages=40)
    d = DevCase(case)
    pd.pd_kv_append(d.k_new, d.v_new, d.k_pool, d.v_pool, d.qo_indptr, d.kv_len, d.page_indptr, d.page_indices,
                    max_kv_len=d.max_kv_len)
    k, v = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.qo_indptr, case.kv_len, case.table.page_indptr, case.table.page_indices,
                     case.k_new, case.v_new, k, v)
    np.testing.assert_array_equal(_bits(d.k_pool), _host_bits(k))
    np.testing.assert_array_equal(_bits(d.v_pool), _host_bits(v))


def test_append_causal_prefill_workload_full():
    # 8 x 512 new tokens, 40 kv heads, D 128, page 16, bf16 -> 256 pages
    case = wl.causal_prefill()
    d = DevCase(case)
    pd.pd_kv_append(d.k_new, d.v_new, d.k_pool, d.v_pool, d.qo_indptr, d.kv_len, d.page_indptr, d.page_indices,
                    max_kv_len=512)
    k, v = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.qo_indptr, case.kv_len, case.table.page_indptr, case.table.page_indices,
                     case.k_new, case.v_new, k, v)
    np.testing.assert_array_equal(_bits(d.k_pool), _host_bits(k))
    np.testing.assert_array_equal(_bits(d.v_pool), _host_bits(v))


def _append_with(case, page_indices):
    """The GPU append of a case with the given page table; returns (pools, status)."""
    d = DevCase(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pd.pd_kv_append(d.k_new, d.v_new, d.k_pool, d.v_pool, d.qo_indptr, d.kv_len, d.page_indptr,
                    dev_tensor(page_indices.astype(np.int32)), max_kv_len=d.max_kv_len, dev_status=status)
    torch.cuda.synchronize()
    return d.k_pool, d.v_pool, int(status.item())


def _oracle_append(case):
    k, v = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.qo_indptr, case.kv_len, case.table.page_indptr, case.table.page_indices,
                     case.k_new, case.v_new, k, v)
    return k, v


def test_append_reports_a_bad_page_id_and_writes_the_rest():
    case = wl.make_attn_case(210, [9, 20, 5], [30, 20, 40], 2, 2, 64, 16, wl.BF16, with_new_tokens=True,
                             num_pages=40)
    bad_at = int(case.table.page_indptr[1]) + 1  # request 1's second page
    bad_page = int(case.table.page_indices[bad_at])
    idx = case.table.page_indices.copy()
    idx[bad_at] = 1000  # past the 40-page pool
    k_dev, v_dev, status = _append_with(case, idx)
    assert status == 3  # bad page table
    k, v = _oracle_append(case)
    # every slot matches the oracle's append except those of the page it could not reach
    k[bad_page], v[bad_page] = case.k_pool[bad_page], case.v_pool[bad_page]
    np.testing.assert_array_equal(_bits(k_dev), _host_bits(k))
    np.testing.assert_array_equal(_bits(v_dev), _host_bits(v))


def test_append_reports_bad_lengths_and_writes_the_rest():
    case = wl.make_attn_case(211, [9, 20, 5], [30, 20, 40], 2, 2, 64, 16, wl.BF16, with_new_tokens=True,
                             num_pages=40)
    d = DevCase(case)
    kv = case.kv_len.astype(np.int32).copy()
    kv[1] = 12  # request 1 brings 20 new tokens but claims 12 cached
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pd.pd_kv_append(d.k_new, d.v_new, d.k_pool, d.v_pool, d.qo_indptr, dev_tensor(kv), d.page_indptr,
                    d.page_indices, max_kv_len=d.max_kv_len, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2  # bad length
    k, v = _oracle_append(case)
    for pg in case.table.page_indices[case.table.page_indptr[1]:case.table.page_indptr[2]]:
        k[pg], v[pg] = case.k_pool[pg], case.v_pool[pg]  # request 1 left unwritten
    np.testing.assert_array_equal(_bits(d.k_pool), _host_bits(k))
    np.testing.assert_array_equal(_bits(d.v_pool), _host_bits(v))


def _handoff_roundtrip(hc: wl.HandoffCase, check_oracle_layers=None):
    es = wl.element_size(hc.dtype)
    L, H, D = hc.num_layers, hc.num_kv_heads, hc.head_dim
    k_src, v_src = dev_tensor(hc.k_src), dev_tensor(hc.v_src)
    kv_len = dev_tensor(hc.kv_len.astype(np.int32))
    s_ptr, s_idx = dev_tensor(hc.src_table.page_indptr), dev_tensor(hc.src_table.page_indices)
    d_ptr, d_idx = dev_tensor(hc.dst_table.page_indptr), dev_tensor(hc.dst_table.page_indices)
    offs = dev_tensor(hc.dst_offsets)
    total = wl.packed_bytes(hc.kv_len, L, H, D, es)
    buf = torch.empty(total, dtype=torch.uint8, device="cuda")
    max_kv = int(hc.kv_len.max())
    pd.pd_kv_pack(k_src, v_src, kv_len, s_ptr, s_idx, buf, offs, max_kv_len=max_kv)
    shape = (L, hc.dst_table.num_pages, H, hc.dst_page_size, D)
    poison = wl._poison(shape, hc.dtype)
    k_dst, v_dst = dev_tensor(poison), dev_tensor(poison)
    pd.pd_kv_unpack(buf, offs, k_dst, v_dst, kv_len, d_ptr, d_idx, max_kv_len=max_kv)
    again = torch.empty_like(buf)
    pd.pd_kv_pack(k_dst, v_dst, kv_len, d_ptr, d_idx, again, offs, max_kv_len=max_kv)
    torch.cuda.synchronize()
    assert torch.equal(buf, again), "pack(unpack(pack(x))) != pack(x)"
    return buf, k_dst, v_dst


def test_pack_unpack_small_against_oracle():
    hc = wl.kv_handoff(seed=204, batch=3, layers=3, heads=4, head_dim=64, src_page=16, dst_page=64,
                       dtype=wl.BF16, kv_lens=[100, 17, 64], src_slack=5, dst_slack=2)
    buf, k_dst, v_dst = _handoff_roundtrip(hc)
    total = buf.numel()
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         hc.dst_offsets, total)
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
    shape = (3, hc.dst_table.num_pages, 4, 64, 64)
    k_ref, v_ref = wl._poison(shape, hc.dtype), wl._poison(shape, hc.dtype)
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, ref, hc.dst_offsets,
                     k_ref, v_ref)
    np.testing.assert_array_equal(_bits(k_dst), _host_bits(k_ref))
    np.testing.assert_array_equal(_bits(v_dst), _host_bits(v_ref))


def test_pack_unpack_head_dim_not_a_power_of_two():
    # head rows of 12 sixteen-byte vectors (head_dim 96, bf16)
    hc = wl.kv_handoff(seed=209, batch=2, layers=2, heads=3, head_dim=96, src_page=16, dst_page=64,
                       dtype=wl.BF16, kv_lens=[70, 33], src_slack=3, dst_slack=1)
    buf, k_dst, v_dst = _handoff_roundtrip(hc)
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         hc.dst_offsets, buf.numel())
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)
    shape = (2, hc.dst_table.num_pages, 3, 64, 96)
    k_ref, v_ref = wl._poison(shape, hc.dtype), wl._poison(shape, hc.dtype)
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, ref, hc.dst_offsets,
                     k_ref, v_ref)
    np.testing.assert_array_equal(_bits(k_dst), _host_bits(k_ref))
    np.testing.assert_array_equal(_bits(v_dst), _host_bits(v_ref))


def test_pack_unpack_fp32_odd_pages():
    hc = wl.kv_handoff(seed=205, batch=2, layers=2, heads=2, head_dim=64, src_page=3, dst_page=5,
                       dtype=wl.F32, kv_lens=[13, 1])
    buf, k_dst, v_dst = _handoff_roundtrip(hc)
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         hc.dst_offsets, buf.numel())
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)


def test_handoff_workload_full():
    # 8 requests x 512 tokens x 40 layers x 40 heads x 128, bf16; pages 16 -> 64.
    # The packed buffer and both destination pools are compared with the
    # oracle's pack and unpack in full. The destination pool has three pages
    # per layer that no request owns: they must keep their poison.
    hc = wl.kv_handoff(dst_slack=3)
    buf, k_dst, v_dst = _handoff_roundtrip(hc)
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         hc.dst_offsets, buf.numel())
    assert np.array_equal(buf.cpu().numpy(), ref)
    shape = tuple(k_dst.shape)
    k_ref, v_ref = wl._poison(shape, hc.dtype), wl._poison(shape, hc.dtype)
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, ref, hc.dst_offsets,
                     k_ref, v_ref)
    used = np.zeros(hc.dst_table.num_pages, dtype=bool)
    used[hc.dst_table.page_indices] = True
    assert not used.all()
    assert np.all(_host_bits(k_ref)[:, ~used] == wl.BF16_NAN)
    assert np.array_equal(_bits(k_dst), _host_bits(k_ref))
    assert np.array_equal(_bits(v_dst), _host_bits(v_ref))


def test_pack_bad_offset_is_reported():
    hc = wl.kv_handoff(seed=206, batch=2, layers=1, heads=2, head_dim=64, src_page=16, dst_page=16,
                       dtype=wl.BF16, kv_lens=[16, 16])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf = torch.zeros(4 * 16 * 64 * 2 * 2 + 64, dtype=torch.uint8, device="cuda")
    offs = dev_tensor(np.array([0, 8], dtype=np.int64))
    pd.pd_kv_pack(dev_tensor(hc.k_src), dev_tensor(hc.v_src), dev_tensor(hc.kv_len), dev_tensor(hc.src_table.page_indptr),
                  dev_tensor(hc.src_table.page_indices), buf, offs, max_kv_len=16, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6


def test_sharded_handoff_tp2_to_tp1_and_back():
    # two prefiller shards hold kv heads [0, 4) and [4, 8); each packs its own
    # pool and the decoder (all 8 heads, page 64) unpacks both blocks at head
    # offsets 0 and 4; then head ranges of the decoder pool are packed again
    hc = wl.kv_handoff(seed=206, batch=3, layers=3, heads=8, head_dim=128, src_page=16, dst_page=64,
                       dtype=wl.BF16, kv_lens=[100, 17, 64], src_slack=3, dst_slack=2)
    L, H, D, half = 3, 8, 128, 4
    kv_len = dev_tensor(hc.kv_len.astype(np.int32))
    s_ptr, s_idx = dev_tensor(hc.src_table.page_indptr), dev_tensor(hc.src_table.page_indices)
    d_ptr, d_idx = dev_tensor(hc.dst_table.page_indptr), dev_tensor(hc.dst_table.page_indices)
    half_bytes = wl.packed_bytes(hc.kv_len, L, half, D, 2)
    half_offs_h = (hc.dst_offsets // 2).astype(np.int64)
    half_offs = dev_tensor(half_offs_h)
    shape = (L, hc.dst_table.num_pages, H, 64, D)
    k1, v1 = dev_tensor(wl._poison(shape, hc.dtype)), dev_tensor(wl._poison(shape, hc.dtype))
    for s in range(2):
        ks = dev_tensor(np.ascontiguousarray(hc.k_src[:, :, s * half:(s + 1) * half]))
        vs = dev_tensor(np.ascontiguousarray(hc.v_src[:, :, s * half:(s + 1) * half]))
        buf = torch.empty(half_bytes, dtype=torch.uint8, device="cuda")
        pd.pd_kv_pack(ks, vs, kv_len, s_ptr, s_idx, buf, half_offs, max_kv_len=100)
        pd.pd_kv_unpack_heads(buf, half_offs, k1, v1, kv_len, d_ptr, d_idx, s * half, half, max_kv_len=100)
    whole = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                           hc.dst_offsets, wl.packed_bytes(hc.kv_len, L, H, D, 2))
    k_ref, v_ref = wl._poison(shape, hc.dtype), wl._poison(shape, hc.dtype)
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, whole, hc.dst_offsets,
                     k_ref, v_ref)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(k1), _host_bits(k_ref))
    np.testing.assert_array_equal(_bits(v1), _host_bits(v_ref))
    for s in range(2):
        buf = torch.empty(half_bytes, dtype=torch.uint8, device="cuda")
        pd.pd_kv_pack_heads(k1, v1, kv_len, d_ptr, d_idx, buf, half_offs, s * half, half, max_kv_len=100)
        ref = oracle.kv_pack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, k_ref, v_ref,
                             half_offs_h, half_bytes, head_begin=s * half, head_count=half)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(buf.cpu().numpy(), ref)
