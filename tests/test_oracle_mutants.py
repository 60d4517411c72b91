"""Each planted mistake in the oracle (built with -DORACLE_MUTANT=n) must fail
at least one of the pins, so that a plausible slip in the oracle (a dropped
scale, a wrong head or slot index, the wrong causal alignment, the wrong log
base, an operand mix-up, a wrong packed order) cannot go unnoticed.

All cases here use even page sizes so every mutant stays inside its buffers.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from test_oracle_pins import brute_force, _two_key_case, _golden, _nhd_golden_pools, mla_brute_force

MUTANTS = {
    1: "scale dropped",
    2: "interleaved GQA head mapping",
    3: "causal bound off by one",
    4: "top-left causal alignment",
    5: "neighbouring page slots swapped",
    6: "base-2 log-sum-exp",
    7: "values read from the key pool",
    8: "packed block token-major",
    9: "unpack writes K into the V pool",
    10: "append writes new tokens in reverse order",
    11: "head range packed from the pool's first heads",
    12: "NHD pools read as HND",
    13: "MLA scores without the rope part",
}


def _attention_pins_hold(mutant):
    cases = [
        wl.make_attn_case(71, [1, 4, 1], [9, 12, 33], 4, 2, 8, 4, wl.F32, causal=True, num_pages=20),
        wl.make_attn_case(72, [6, 2], [6, 11], 4, 2, 16, 2, wl.BF16, causal=True, num_pages=20),
    ]
    cases.append(wl.to_nhd(cases[0]))
    for case in cases:
        o, lse = oracle.attention_case(case, mutant=mutant)
        o_ref, lse_ref = brute_force(case)
        if not (np.allclose(o, o_ref, atol=1e-12, rtol=0) and np.allclose(lse, lse_ref, atol=1e-12, rtol=0)):
            return False
    mla = wl.mla_case(35, [9, 30, 2], num_qo_heads=4, d_c=16, d_r=8, page_size=4, dtype=wl.F32)
    o, lse = oracle.mla_decode(mla.kv_len, mla.table.page_indptr, mla.table.page_indices, mla.q, mla.kv_pool,
                               mla.d_c, mla.sm_scale, mutant=mutant)
    o_ref, lse_ref = mla_brute_force(mla)
    if not (np.allclose(o, o_ref, atol=1e-12, rtol=0) and np.allclose(lse, lse_ref, atol=1e-12, rtol=0)):
        return False
    case, g = _two_key_case(2)
    o, lse = oracle.attention_case(case, mutant=mutant)
    if not (np.allclose(o[1, 0], g["row1_o"], atol=1e-15) and np.isclose(lse[1, 0], g["row1_lse"][0], atol=1e-15)):
        return False
    return True


def _copy_pins_hold(mutant):
    g = _golden("pack_small.txt")
    k = np.zeros((1, 3, 2, 2, 2), np.float32)
    for page in range(3):
        for h in range(2):
            for s in range(2):
                for d in range(2):
                    k[0, page, h, s, d] = 1000 * page + 100 * h + 10 * s + d
    v = k + np.float32(0.5)
    packed = oracle.kv_pack([3], [0, 2], [2, 0], k, v, [0], 96, mutant=mutant)
    if not np.array_equal(packed.view(np.float32), np.array(g["expected"], np.float32)):
        return False
    kn, vn = _nhd_golden_pools()
    packed = oracle.kv_pack([3], [0, 2], [2, 0], kn, vn, [0], 96, mutant=mutant, layout=oracle.NHD)
    if not np.array_equal(packed.view(np.float32), np.array(g["expected"], np.float32)):
        return False
    hc = wl.kv_handoff(seed=81, batch=2, layers=2, heads=2, head_dim=4, src_page=4, dst_page=8,
                       dtype=wl.F32, kv_lens=[13, 8])
    total = wl.packed_bytes(hc.kv_len, 2, 2, 4, 4)
    buf = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices,
                         hc.k_src, hc.v_src, hc.dst_offsets, total, mutant=mutant)
    shape = (2, hc.dst_table.num_pages, 2, 8, 4)
    kd, vd = np.full(shape, np.nan, np.float32), np.full(shape, np.nan, np.float32)
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, buf,
                     hc.dst_offsets, kd, vd, mutant=mutant)
    again = oracle.kv_pack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices,
                           kd, vd, hc.dst_offsets, total, mutant=0)
    if not np.array_equal(buf, again):
        return False
    # a head range is the head slice of the full block
    part_total = wl.packed_bytes(hc.kv_len, 2, 1, 4, 4)
    part_off = np.array([0, wl.packed_bytes(hc.kv_len[:1], 2, 1, 4, 4)], np.int64)
    part = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices,
                          hc.k_src, hc.v_src, part_off, part_total, mutant=mutant, head_begin=1, head_count=1)
    for r, n in enumerate(hc.kv_len):
        full_r = buf[hc.dst_offsets[r]:hc.dst_offsets[r] + wl.packed_bytes([n], 2, 2, 4, 4)]
        want = full_r.reshape(2, 2, 2, n, 16)[:, :, 1:2]
        got = part[part_off[r]:part_off[r] + want.size].reshape(want.shape)
        if not np.array_equal(got, want):
            return False
    pre = wl.make_attn_case(82, [5, 3], [9, 12], 2, 2, 4, 4, wl.F32, with_new_tokens=True, num_pages=8)
    full = wl.make_attn_case(82, [5, 3], [9, 12], 2, 2, 4, 4, wl.F32, with_new_tokens=False, num_pages=8)
    k2, v2 = pre.k_pool.copy(), pre.v_pool.copy()
    oracle.kv_append(pre.qo_indptr, pre.kv_len, pre.table.page_indptr, pre.table.page_indices,
                     pre.k_new, pre.v_new, k2, v2, mutant=mutant)
    return np.array_equal(k2.view(np.uint32), full.k_pool.view(np.uint32)) and \
        np.array_equal(v2.view(np.uint32), full.v_pool.view(np.uint32))


def test_unmutated_oracle_passes_the_battery():
    assert _attention_pins_hold(0) and _copy_pins_hold(0)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant):
    assert oracle.build(mutant)
    assert not (_attention_pins_hold(mutant) and _copy_pins_hold(mutant)), MUTANTS[mutant]
