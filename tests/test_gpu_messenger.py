"""GPU: the layer-streamed handoff. A model stream writes one layer at a time
and signals a counter after each; the messenger's host thread packs every layer
as soon as the counter passes it, on its own stream. The packed blocks must be
bit-identical to the oracle's pack of the finished pools (a layer packed before
its data arrived would show the NaN poison the pools start with)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import dev_tensor


def test_streamed_layer_pack_equals_the_full_pack():
    hc = wl.kv_handoff(seed=208, batch=3, layers=6, heads=4, head_dim=128, src_page=16, dst_page=64,
                       dtype=wl.BF16, kv_lens=[100, 17, 64], src_slack=2)
    L = hc.num_layers
    truth_k, truth_v = dev_tensor(hc.k_src), dev_tensor(hc.v_src)
    poison = wl._poison(hc.k_src.shape, hc.dtype)
    k_pool, v_pool = dev_tensor(poison), dev_tensor(poison)
    kv_len = dev_tensor(hc.kv_len.astype(np.int32))
    s_ptr, s_idx = dev_tensor(hc.src_table.page_indptr), dev_tensor(hc.src_table.page_indices)
    offs = dev_tensor(hc.dst_offsets)
    total = wl.packed_bytes(hc.kv_len, L, hc.num_kv_heads, hc.head_dim, 2)
    buf = torch.zeros(total, dtype=torch.uint8, device="cuda")
    host_w, dev_w = pd.pd_counter_alloc()
    model, messenger = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        h = pd.pd_messenger_start_pack(host_w, k_pool, v_pool, kv_len, s_ptr, s_idx, buf, offs, timeout_ms=5000,
                                       max_kv_len=100, stream=messenger)
        with torch.cuda.stream(model):
            for layer in range(L):
                torch.cuda._sleep(200000)  # layers become ready one at a time
                k_pool[layer].copy_(truth_k[layer])
                v_pool[layer].copy_(truth_v[layer])
                pd.pd_layer_signal(dev_w, layer + 1, stream=model)
        assert pd.pd_messenger_join(h) == L
        model.synchronize()
        messenger.synchronize()
        assert pd.counter_value(host_w) == L
    finally:
        torch.cuda.synchronize()
        pd.pd_counter_free(host_w)
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         hc.dst_offsets, total)
    np.testing.assert_array_equal(buf.cpu().numpy(), ref)


def test_layer_range_pack_fills_its_slice_of_the_blocks():
    hc = wl.kv_handoff(seed=209, batch=2, layers=4, heads=2, head_dim=64, src_page=16, dst_page=64,
                       dtype=wl.BF16, kv_lens=[40, 7])
    L, H, D = hc.num_layers, hc.num_kv_heads, hc.head_dim
    total = wl.packed_bytes(hc.kv_len, L, H, D, 2)
    buf = torch.zeros(total, dtype=torch.uint8, device="cuda")
    pd.pd_kv_pack_layers(dev_tensor(hc.k_src), dev_tensor(hc.v_src), dev_tensor(hc.kv_len.astype(np.int32)),
                         dev_tensor(hc.src_table.page_indptr), dev_tensor(hc.src_table.page_indices), buf,
                         dev_tensor(hc.dst_offsets), 1, 2, max_kv_len=40)
    torch.cuda.synchronize()
    got = buf.cpu().numpy()
    ref = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                         hc.dst_offsets, total)
    for r, n in enumerate(hc.kv_len):
        blk = slice(int(hc.dst_offsets[r]), int(hc.dst_offsets[r]) + L * 2 * H * int(n) * D * 2)
        g, w = got[blk].reshape(L, -1), ref[blk].reshape(L, -1)
        np.testing.assert_array_equal(g[1:3], w[1:3])         # layers 1 and 2 written
        assert not g[0].any() and not g[3].any()              # layers 0 and 3 untouched


def test_messenger_timeout_without_signal():
    hc = wl.kv_handoff(seed=210, batch=1, layers=2, heads=2, head_dim=64, src_page=16, dst_page=64,
                       dtype=wl.BF16, kv_lens=[20])
    total = wl.packed_bytes(hc.kv_len, 2, 2, 64, 2)
    buf = torch.zeros(total, dtype=torch.uint8, device="cuda")
    host_w, _ = pd.pd_counter_alloc()
    try:
        h = pd.pd_messenger_start_pack(host_w, dev_tensor(hc.k_src), dev_tensor(hc.v_src),
                                       dev_tensor(hc.kv_len.astype(np.int32)), dev_tensor(hc.src_table.page_indptr),
                                       dev_tensor(hc.src_table.page_indices), buf, dev_tensor(hc.dst_offsets),
                                       timeout_ms=100, max_kv_len=20)
        with pytest.raises(pd.PdError) as e:
            pd.pd_messenger_join(h)
        assert e.value.code == pd.PD_ERR_TIMEOUT
    finally:
        torch.cuda.synchronize()
        pd.pd_counter_free(host_w)
