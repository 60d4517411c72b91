"""Pins for the fp64 oracle, on the CPU.

The oracle is checked against things other than itself: numpy brute force on
tiny inputs (written here, independently), torch's fp64 scaled_dot_product_attention
on densely gathered tensors, closed forms, hand-worked golden examples and
invariants that the definition implies (Perplexity, "Disaggregated prefill and
decode", sections "Prefill vs Decode performance", "Sharded KV cache
transfers", "Speculative decoding").
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = [float(v) for v in vals]
    return rows


def _values(arr):
    return wl.bf16_to_f32(arr).astype(np.float64) if arr.dtype == np.uint16 else arr.astype(np.float64)


# ---------------------------------------------------------------------------
# independent references
# ---------------------------------------------------------------------------

def brute_force(case):
    """Dense softmax(Q K^T * scale + mask) V per request, numpy fp64, token-wise gather."""
    q = _values(case.q)
    kp, vp = _values(case.k_pool), _values(case.v_pool)
    G = case.num_qo_heads // case.num_kv_heads
    P = case.page_size
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for r in range(case.batch_size):
        n = int(case.kv_len[r])
        qo = int(case.qo_indptr[r + 1] - case.qo_indptr[r])
        pages = case.table.page_indices[case.table.page_indptr[r]:case.table.page_indptr[r + 1]]
        if case.layout == "NHD":   # page [P][Hkv][D]: slot first
            at = lambda pool, t: pool[pages[t // P], t % P, :, :]
        else:                      # page [Hkv][P][D]: head first
            at = lambda pool, t: pool[pages[t // P], :, t % P, :]
        K = np.stack([at(kp, t) for t in range(n)], axis=1) if n else np.zeros((case.num_kv_heads, 0, q.shape[2]))
        V = np.stack([at(vp, t) for t in range(n)], axis=1) if n else np.zeros((case.num_kv_heads, 0, q.shape[2]))
        K = np.repeat(K, G, axis=0)            # [Hq][n][D]
        V = np.repeat(V, G, axis=0)
        Q = q[case.qo_indptr[r]:case.qo_indptr[r + 1]].transpose(1, 0, 2)  # [Hq][qo][D]
        S = np.einsum("hid,hjd->hij", Q, K) * case.scale
        if case.causal:
            i = np.arange(qo)[:, None]
            j = np.arange(n)[None, :]
            S = np.where(j <= n - qo + i, S, -np.inf)
        m = S.max(axis=2, keepdims=True) if n else np.full(S.shape[:2] + (1,), -np.inf)
        with np.errstate(invalid="ignore"):
            E = np.exp(S - m)
        E = np.nan_to_num(E)
        l = E.sum(axis=2, keepdims=True)
        O = np.einsum("hij,hjd->hid", E, V) / np.where(l > 0, l, 1)
        o[case.qo_indptr[r]:case.qo_indptr[r + 1]] = O.transpose(1, 0, 2)
        with np.errstate(divide="ignore"):
            lse[case.qo_indptr[r]:case.qo_indptr[r + 1]] = (m[..., 0] + np.log(l[..., 0])).T
    return o, lse


def sdpa_reference(case, r):
    """torch fp64 SDPA for request r, KV gathered page by page (a different gather)."""
    n = int(case.kv_len[r])
    qo = int(case.qo_indptr[r + 1] - case.qo_indptr[r])
    pages = case.table.page_indices[case.table.page_indptr[r]:case.table.page_indptr[r + 1]]
    G = case.num_qo_heads // case.num_kv_heads

    def dense(pool):
        x = torch.from_numpy(_values(pool)[pages])              # [np][Hkv][P][D]
        x = x.permute(1, 0, 2, 3).reshape(case.num_kv_heads, -1, x.shape[-1])[:, :n]
        return x.repeat_interleave(G, dim=0)[None]               # [1][Hq][n][D]

    Q = torch.from_numpy(_values(case.q)[case.qo_indptr[r]:case.qo_indptr[r + 1]]).permute(1, 0, 2)[None]
    causal = case.causal and qo > 1
    assert not causal or qo == n, "SDPA's causal mask is top-left aligned; use it only when qo == kv"
    O = torch.nn.functional.scaled_dot_product_attention(Q, dense(case.k_pool), dense(case.v_pool),
                                                         is_causal=causal, scale=case.scale)
    return O[0].permute(1, 0, 2).numpy()


def run_oracle(case, mutant=0):
    return oracle.attention_case(case, mutant=mutant)


def small_cases():
    yield wl.make_attn_case(11, [1, 1, 1], [1, 7, 33], 4, 2, 8, 4, wl.F32, causal=True, num_pages=20)
    yield wl.make_attn_case(12, [3, 5, 1], [3, 9, 16], 6, 3, 16, 2, wl.BF16, causal=True, num_pages=20)
    yield wl.make_attn_case(13, [4, 2], [10, 2], 2, 2, 8, 1, wl.F32, causal=False, num_pages=15)
    yield wl.make_attn_case(14, [8, 1, 6], [8, 40, 13], 8, 2, 32, 16, wl.BF16, causal=True, num_pages=8)


# ---------------------------------------------------------------------------
# brute force and library pins
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("idx", range(4))
def test_brute_force(idx):
    case = list(small_cases())[idx]
    o, lse = run_oracle(case)
    o_ref, lse_ref = brute_force(case)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_sdpa_library_decode_and_square_prefill():
    cases = [
        wl.make_attn_case(21, [1, 1, 1, 1], [5, 16, 17, 64], 8, 2, 64, 16, wl.BF16, causal=True),
        wl.make_attn_case(22, [24, 17], [24, 17], 4, 4, 32, 4, wl.F32, causal=True),
        wl.make_attn_case(23, [5, 9], [12, 30], 4, 1, 16, 8, wl.F32, causal=False),
    ]
    for case in cases:
        o, _ = run_oracle(case)
        for r in range(case.batch_size):
            ref = sdpa_reference(case, r)
            np.testing.assert_allclose(o[case.qo_indptr[r]:case.qo_indptr[r + 1]], ref, rtol=0, atol=1e-12)


def test_rows_entry_matches_full():
    case = list(small_cases())[3]
    o, lse = run_oracle(case)
    rows = np.array([0, 3, 7, 8, 9, 14], dtype=np.int32)
    heads = np.array([0, 7, 3, 5, 1, 2], dtype=np.int32)
    o2, lse2 = oracle.attention_rows(case.qo_indptr, case.kv_len, case.table.page_indptr,
                                     case.table.page_indices, case.q, case.k_pool, case.v_pool,
                                     case.num_qo_heads, case.num_kv_heads, case.scale, rows, heads,
                                     causal=case.causal)
    np.testing.assert_array_equal(o2, o[rows, heads])
    np.testing.assert_array_equal(lse2, lse[rows, heads])


# ---------------------------------------------------------------------------
# closed forms and golden examples
# ---------------------------------------------------------------------------

def _two_key_case(qo_len):
    g = _golden("two_key_attention.txt")
    P, D = 2, 2
    k_pool = np.full((2, 1, P, D), np.nan, dtype=np.float32)
    v_pool = np.full((2, 1, P, D), np.nan, dtype=np.float32)
    k_pool[1, 0, 0], k_pool[1, 0, 1] = g["k0"], g["k1"]
    v_pool[1, 0, 0], v_pool[1, 0, 1] = g["v0"], g["v1"]
    q = np.array(g["q"], dtype=np.float32).reshape(2, 1, D)[2 - qo_len:]
    table = wl.PageTable(np.array([0, 1], np.int32), np.array([1], np.int32), 2)
    case = wl.AttnCase(wl.F32, 1, 1, D, P, np.array([0, qo_len], np.int32), np.array([2], np.int32),
                       table, q, k_pool, v_pool, causal=True, sm_scale=1.0)
    return case, g


def test_golden_two_key_prefill_and_decode():
    case, g = _two_key_case(2)
    o, lse = run_oracle(case)
    np.testing.assert_allclose(o[0, 0], g["row0_o"], atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], g["row0_lse"][0], atol=1e-15)
    np.testing.assert_allclose(o[1, 0], g["row1_o"], atol=1e-15)
    np.testing.assert_allclose(lse[1, 0], g["row1_lse"][0], atol=1e-15)
    case, g = _two_key_case(1)
    o, lse = run_oracle(case)
    np.testing.assert_allclose(o[0, 0], g["row1_o"], atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], g["row1_lse"][0], atol=1e-15)


def test_single_key_returns_its_value():
    case = wl.make_attn_case(31, [1, 1], [1, 1], 4, 2, 16, 4, wl.BF16, num_pages=6)
    o, lse = run_oracle(case)
    kp, vp, q = _values(case.k_pool), _values(case.v_pool), _values(case.q)
    for r in range(2):
        page = case.table.page_indices[case.table.page_indptr[r]]
        for h in range(4):
            g = h // 2
            np.testing.assert_array_equal(o[r, h], vp[page, g, 0])
            np.testing.assert_allclose(lse[r, h], case.scale * np.dot(q[r, h], kp[page, g, 0]), atol=1e-14)


def test_identical_keys_give_mean_value():
    case = wl.make_attn_case(32, [1], [37], 2, 1, 8, 4, wl.F32)
    pages = case.table.page_indices
    key = np.random.default_rng(0).standard_normal(8).astype(np.float32)
    case.k_pool[pages] = key                       # every slot of the request's pages
    o, lse = run_oracle(case)
    n = 37
    vals = np.stack([_values(case.v_pool)[pages[t // 4], 0, t % 4] for t in range(n)])
    for h in range(2):
        np.testing.assert_allclose(o[0, h], vals.mean(axis=0), atol=1e-13)
        s = case.scale * np.dot(_values(case.q)[0, h], key.astype(np.float64))
        np.testing.assert_allclose(lse[0, h], s + np.log(n), atol=1e-12)


def test_softmax_rows_sum_to_one_via_constant_values():
    # With every value equal to 1, o = sum_j p_j must be exactly 1 per row.
    case = wl.make_attn_case(33, [6, 1, 3], [6, 50, 20], 4, 2, 16, 8, wl.BF16, causal=True)
    case.v_pool[:] = wl.bf16_from_f32(np.ones(1, np.float32))[0]
    o, _ = run_oracle(case)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


def test_dominant_key_selects_its_value():
    case = wl.make_attn_case(34, [1], [40], 1, 1, 4, 4, wl.F32, sm_scale=1.0)
    pages = case.table.page_indices
    case.q[0, 0] = [1, 0, 0, 0]
    case.k_pool[pages, 0, :, 0] = 0.0
    t = 29
    case.k_pool[pages[t // 4], 0, t % 4, 0] = 60.0   # exp(-60) relative weight for the rest
    o, lse = run_oracle(case)
    np.testing.assert_allclose(o[0, 0], case.v_pool[pages[t // 4], 0, t % 4], atol=1e-20 + 1e-24)
    np.testing.assert_allclose(lse[0, 0], 60.0, atol=1e-20)


def test_empty_request_gives_zero_and_minus_inf():
    case = wl.make_attn_case(35, [1, 1], [0, 5], 2, 2, 8, 4, wl.F32, causal=False, num_pages=4)
    o, lse = run_oracle(case)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(o[1]))


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_physical_page_permutation_invariance():
    case = wl.make_attn_case(41, [1, 4, 1], [30, 22, 9], 4, 2, 16, 4, wl.BF16, num_pages=25)
    o, lse = run_oracle(case)
    rng = np.random.default_rng(7)
    perm = rng.permutation(case.table.num_pages)           # new physical id of each page
    k2 = np.empty_like(case.k_pool)
    v2 = np.empty_like(case.v_pool)
    k2[perm] = case.k_pool
    v2[perm] = case.v_pool
    o2, lse2 = oracle.attention(case.qo_indptr, case.kv_len, case.table.page_indptr,
                                perm[case.table.page_indices], case.q, k2, v2, 4, 2, case.scale)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_prefill_equals_successive_decodes():
    # Speculative-decoding section: the last prompt token is run as a decode step
    # with no change of result; generally, causal row i of a prefill equals a
    # decode over the first kv_len - qo_len + i + 1 keys.
    L = 21
    pre = wl.make_attn_case(42, [L], [L], 4, 2, 16, 4, wl.BF16, causal=True)
    o, lse = run_oracle(pre)
    for i in range(L):
        dec_q = pre.q[i:i + 1]
        od, ld = oracle.attention([0, 1], [i + 1], pre.table.page_indptr, pre.table.page_indices,
                                  dec_q, pre.k_pool, pre.v_pool, 4, 2, pre.scale, causal=True)
        np.testing.assert_allclose(od[0], o[i], atol=1e-14)
        np.testing.assert_allclose(ld[0], lse[i], atol=1e-14)


def test_lse_merge_of_two_key_halves_equals_whole():
    # Splitting the key axis (the blog's "Split-K" parallelism over kv_len) and
    # merging by log-sum-exp must give the whole: o = sum_c exp(lse_c - lse) o_c.
    P = 4
    case = wl.make_attn_case(43, [1], [36], 4, 2, 16, P, wl.F32, causal=False)
    o, lse = run_oracle(case)
    pages = case.table.page_indices
    first = dict(kv_len=[16], page_indptr=[0, 4], page_indices=pages[:4])
    second = dict(kv_len=[20], page_indptr=[0, 5], page_indices=pages[4:])
    parts = []
    for part in (first, second):
        parts.append(oracle.attention([0, 1], part["kv_len"], part["page_indptr"], part["page_indices"],
                                      case.q, case.k_pool, case.v_pool, 4, 2, case.scale, causal=False))
    lse_m = np.logaddexp(parts[0][1], parts[1][1])
    o_m = (np.exp(parts[0][1] - lse_m)[..., None] * parts[0][0]
           + np.exp(parts[1][1] - lse_m)[..., None] * parts[1][0])
    np.testing.assert_allclose(lse_m, lse, atol=1e-13)
    np.testing.assert_allclose(o_m, o, atol=1e-13)


# ---------------------------------------------------------------------------
# append / pack / unpack
# ---------------------------------------------------------------------------

def test_golden_pack_small():
    g = _golden("pack_small.txt")
    L, Hkv, D, P = 1, 2, 2, 2
    k = np.full((L, 3, Hkv, P, D), np.nan, np.float32)
    for page in range(3):
        for h in range(Hkv):
            for s in range(P):
                for d in range(D):
                    k[0, page, h, s, d] = 1000 * page + 100 * h + 10 * s + d
    v = k + np.float32(0.5)
    packed = oracle.kv_pack([3], [0, 2], [2, 0], k, v, [0], 2 * Hkv * 3 * D * 4)
    np.testing.assert_array_equal(packed.view(np.float32), np.array(g["expected"], np.float32))


def test_pack_unpack_roundtrip_and_page_size_change():
    hc = wl.kv_handoff(seed=51, batch=3, layers=2, heads=3, head_dim=8, src_page=4, dst_page=16,
                       dtype=wl.BF16, kv_lens=[13, 32, 1], src_slack=3, dst_slack=2)
    es = 2
    total = wl.packed_bytes(hc.kv_len, 2, 3, 8, es)
    packed = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices,
                            hc.k_src, hc.v_src, hc.dst_offsets, total)
    # decoder pool with page size 16
    shape = (2, hc.dst_table.num_pages, 3, 16, 8)
    k_dst = np.full(shape, wl.BF16_NAN, np.uint16)
    v_dst = np.full(shape, wl.BF16_NAN, np.uint16)
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, packed,
                     hc.dst_offsets, k_dst, v_dst)
    # every logical token is identical, byte for byte, on both sides
    for layer in range(2):
        for r, n in enumerate(hc.kv_len):
            sp = hc.src_table.page_indices[hc.src_table.page_indptr[r]:hc.src_table.page_indptr[r + 1]]
            dp = hc.dst_table.page_indices[hc.dst_table.page_indptr[r]:hc.dst_table.page_indptr[r + 1]]
            for t in range(n):
                np.testing.assert_array_equal(hc.k_src[layer, sp[t // 4], :, t % 4], k_dst[layer, dp[t // 16], :, t % 16])
                np.testing.assert_array_equal(hc.v_src[layer, sp[t // 4], :, t % 4], v_dst[layer, dp[t // 16], :, t % 16])
    # re-packing the decoder pool reproduces the same bytes
    again = oracle.kv_pack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices,
                           k_dst, v_dst, hc.dst_offsets, total)
    np.testing.assert_array_equal(packed, again)
    # slots that hold no token stay untouched (still poison)
    used = np.zeros((hc.dst_table.num_pages, 16), bool)
    for r, n in enumerate(hc.kv_len):
        dp = hc.dst_table.page_indices[hc.dst_table.page_indptr[r]:hc.dst_table.page_indptr[r + 1]]
        for t in range(n):
            used[dp[t // 16], t % 16] = True
    kd = k_dst.transpose(0, 1, 3, 2, 4)                     # [L][page][slot][Hkv][D]
    assert np.all(kd[:, ~used] == wl.BF16_NAN)
    assert np.all(kd[:, used] != wl.BF16_NAN)


def test_append_then_attention_matches_direct_fill():
    pre = wl.make_attn_case(61, [5, 1, 16], [9, 30, 16], 4, 2, 16, 4, wl.BF16, causal=True,
                            with_new_tokens=True, num_pages=20)
    full = wl.make_attn_case(61, [5, 1, 16], [9, 30, 16], 4, 2, 16, 4, wl.BF16, causal=True,
                             with_new_tokens=False, num_pages=20)
    k, v = pre.k_pool.copy(), pre.v_pool.copy()
    oracle.kv_append(pre.qo_indptr, pre.kv_len, pre.table.page_indptr, pre.table.page_indices,
                     pre.k_new, pre.v_new, k, v)
    np.testing.assert_array_equal(k.view(np.uint16), full.k_pool.view(np.uint16))
    np.testing.assert_array_equal(v.view(np.uint16), full.v_pool.view(np.uint16))


def test_transfer_estimate_bookkeeping():
    g = _golden("kv_transfer_estimate.txt")
    per_token = wl.packed_bytes([1], int(g["layers"][0]), int(g["kv_heads"][0]),
                                int(g["head_dim"][0]), int(g["elem_bytes"][0]))
    assert per_token == g["bytes_per_token"][0] == 4.5 * 2 ** 20
    total = wl.packed_bytes([int(g["tokens"][0])], int(g["layers"][0]), int(g["kv_heads"][0]),
                            int(g["head_dim"][0]), int(g["elem_bytes"][0]))
    ms = total / (g["links"][0] * g["link_gib_s"][0] * 2 ** 30) * 1e3
    assert ms == pytest.approx(g["transfer_ms"][0], abs=1e-9)
    assert round(ms, 1) == g["printed_ms"][0]


def _block_heads(buf, off, n, layers, heads, row_bytes):
    """One request's packed block as [layer][K,V][head][token][row bytes]."""
    size = layers * 2 * heads * n * row_bytes
    return buf[off:off + size].reshape(layers, 2, heads, n, row_bytes)


def test_head_range_pack_is_the_head_slice_of_the_full_pack():
    # Perplexity, "Disaggregated prefill and decode" (2025), "Sharded KV cache
    # transfers": a shard's heads are a slice of the whole, so packing heads
    # [h0, h0 + hc) must give exactly that slice of the full block.
    hc = wl.kv_handoff(seed=91, batch=3, layers=2, heads=4, head_dim=8, src_page=4, dst_page=8,
                       dtype=wl.BF16, kv_lens=[9, 16, 5])
    row = 8 * 2
    full = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                          hc.dst_offsets, wl.packed_bytes(hc.kv_len, 2, 4, 8, 2))
    for h0, cnt in [(0, 4), (1, 2), (3, 1)]:
        per = np.asarray(hc.kv_len, np.int64) * 2 * 2 * cnt * row
        offs = np.concatenate([[0], np.cumsum(per)[:-1]]).astype(np.int64)
        part = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src,
                              hc.v_src, offs, int(per.sum()), head_begin=h0, head_count=cnt)
        for r, n in enumerate(hc.kv_len):
            want = _block_heads(full, hc.dst_offsets[r], n, 2, 4, row)[:, :, h0:h0 + cnt]
            assert np.array_equal(_block_heads(part, offs[r], n, 2, cnt, row), want)


def test_tp2_prefiller_to_tp1_decoder_and_back():
    # Two prefiller shards hold heads [0, 2) and [2, 4) of the same logical pool;
    # each packs its own pool and the decoder unpacks both into one 4-head pool
    # at head offsets 0 and 2: the result equals unpacking the whole at once.
    # Back the other way, head ranges of the decoder pool unpacked into 2-head
    # pools give the head slices of the whole.
    hc = wl.kv_handoff(seed=92, batch=2, layers=2, heads=4, head_dim=8, src_page=4, dst_page=8,
                       dtype=wl.BF16, kv_lens=[11, 20])
    full_bytes = wl.packed_bytes(hc.kv_len, 2, 4, 8, 2)
    half_bytes = wl.packed_bytes(hc.kv_len, 2, 2, 8, 2)
    half_offs = (hc.dst_offsets // 2).astype(np.int64)
    dshape = (2, hc.dst_table.num_pages, 4, 8, 8)
    ref_k, ref_v = np.full(dshape, 0xFFFF, np.uint16), np.full(dshape, 0xFFFF, np.uint16)
    whole = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                           hc.dst_offsets, full_bytes)
    oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, whole, hc.dst_offsets,
                     ref_k, ref_v)
    k1, v1 = np.full(dshape, 0xFFFF, np.uint16), np.full(dshape, 0xFFFF, np.uint16)
    for s in range(2):
        ks = np.ascontiguousarray(hc.k_src[:, :, 2 * s:2 * s + 2])
        vs = np.ascontiguousarray(hc.v_src[:, :, 2 * s:2 * s + 2])
        buf = oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, ks, vs,
                             half_offs, half_bytes)
        oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, buf, half_offs,
                         k1, v1, head_begin=2 * s, head_count=2)
    assert np.array_equal(k1, ref_k) and np.array_equal(v1, ref_v)
    for s in range(2):
        buf = oracle.kv_pack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, ref_k, ref_v,
                             half_offs, half_bytes, head_begin=2 * s, head_count=2)
        hshape = (2, hc.dst_table.num_pages, 2, 8, 8)
        k2, v2 = np.full(hshape, 0xFFFF, np.uint16), np.full(hshape, 0xFFFF, np.uint16)
        oracle.kv_unpack(hc.kv_len, hc.dst_table.page_indptr, hc.dst_table.page_indices, buf, half_offs, k2, v2)
        assert np.array_equal(k2, ref_k[:, :, 2 * s:2 * s + 2]) and np.array_equal(v2, ref_v[:, :, 2 * s:2 * s + 2])


def test_head_range_outside_the_pool_is_rejected():
    hc = wl.kv_handoff(seed=93, batch=1, layers=1, heads=2, head_dim=8, src_page=4, dst_page=8,
                       dtype=wl.BF16, kv_lens=[5])
    for h0, cnt in [(1, 2), (-1, 1), (0, 0)]:
        with pytest.raises(ValueError):
            oracle.kv_pack(hc.kv_len, hc.src_table.page_indptr, hc.src_table.page_indices, hc.k_src, hc.v_src,
                           [0], 1024, head_begin=h0, head_count=cnt)


# ---------------------------------------------------------------------------
# NHD pools (post, "Sharded KV cache transfers": the figure contrasts NHD,
# token before head, with HND, head before token)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("idx", range(4))
def test_nhd_pools_match_brute_force_and_the_hnd_result(idx):
    case = list(small_cases())[idx]
    nhd = wl.to_nhd(case)
    o, lse = oracle.attention_case(nhd)
    o_bf, lse_bf = brute_force(nhd)
    np.testing.assert_allclose(o, o_bf, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse_bf, atol=1e-12, rtol=0)
    o_h, lse_h = oracle.attention_case(case)
    assert np.array_equal(o, o_h) and np.array_equal(lse, lse_h)  # same values, same order of sums


def _nhd_golden_pools():
    """The pack_small.txt pools written in the NHD layout: element (page, head h,
    slot s, dim d) = 1000 page + 100 h + 10 s + d, stored at [page][s][h][d]."""
    k = np.zeros((1, 3, 2, 2, 2), np.float32)
    for page in range(3):
        for s in range(2):
            for h in range(2):
                for d in range(2):
                    k[0, page, s, h, d] = 1000 * page + 100 * h + 10 * s + d
    return k, k + np.float32(0.5)


def test_golden_pack_small_from_nhd_pools():
    g = _golden("pack_small.txt")
    k, v = _nhd_golden_pools()
    packed = oracle.kv_pack([3], [0, 2], [2, 0], k, v, [0], 96, layout=oracle.NHD)
    np.testing.assert_array_equal(packed.view(np.float32), np.array(g["expected"], np.float32))


def test_nhd_append_pack_unpack_agree_with_hnd():
    hc = wl.kv_handoff(seed=91, batch=3, layers=2, heads=3, head_dim=4, src_page=4, dst_page=8,
                       dtype=wl.F32, kv_lens=[13, 1, 8], src_slack=2, dst_slack=1)
    nhd = wl.to_nhd(hc)
    total = wl.packed_bytes(hc.kv_len, 2, 3, 4, 4)
    t = hc.src_table
    a = oracle.kv_pack(hc.kv_len, t.page_indptr, t.page_indices, hc.k_src, hc.v_src, hc.dst_offsets, total)
    b = oracle.kv_pack(hc.kv_len, t.page_indptr, t.page_indices, nhd.k_src, nhd.v_src, hc.dst_offsets, total,
                       layout=oracle.NHD)
    assert np.array_equal(a, b)
    # unpack into page-8 pools of both layouts (NaN where no token lands)
    dshape = (2, hc.dst_table.num_pages, 3, 8, 4)
    kh, vh = np.full(dshape, np.nan, np.float32), np.full(dshape, np.nan, np.float32)
    kn, vn = wl.nhd_pool(kh), wl.nhd_pool(vh)
    d = hc.dst_table
    oracle.kv_unpack(hc.kv_len, d.page_indptr, d.page_indices, a, hc.dst_offsets, kh, vh)
    oracle.kv_unpack(hc.kv_len, d.page_indptr, d.page_indices, a, hc.dst_offsets, kn, vn, layout=oracle.NHD)
    np.testing.assert_array_equal(wl.nhd_pool(kh), kn)
    np.testing.assert_array_equal(wl.nhd_pool(vh), vn)
    # append the last two tokens of every request into both layouts
    case = wl.make_attn_case(92, [2, 1, 2], [13, 1, 8], 6, 3, 4, 4, wl.F32, with_new_tokens=True, num_pages=9)
    ckn, cvn = wl.nhd_pool(case.k_pool), wl.nhd_pool(case.v_pool)
    tt = case.table
    oracle.kv_append(case.qo_indptr, case.kv_len, tt.page_indptr, tt.page_indices, case.k_new, case.v_new,
                     case.k_pool, case.v_pool)
    oracle.kv_append(case.qo_indptr, case.kv_len, tt.page_indptr, tt.page_indices, case.k_new, case.v_new,
                     ckn, cvn, layout=oracle.NHD)
    np.testing.assert_array_equal(wl.nhd_pool(case.k_pool), ckn)
    np.testing.assert_array_equal(wl.nhd_pool(case.v_pool), cvn)
    # and the appended NHD pools attend like the brute force over them
    nhd_case = wl.to_nhd(case)
    nhd_case.k_pool, nhd_case.v_pool = ckn, cvn
    o, lse = oracle.attention_case(nhd_case)
    o_bf, lse_bf = brute_force(nhd_case)
    np.testing.assert_allclose(o, o_bf, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse_bf, atol=1e-12, rtol=0)


def test_unknown_layout_is_rejected():
    case = next(small_cases())
    with pytest.raises(ValueError):
        oracle.attention_case(case.__class__(**{**case.__dict__, "layout": "HDN"}))


# ---------------------------------------------------------------------------
# MLA decode over a paged latent cache (post, "Disaggregated Deployments",
# "DeepSeek-R1": one latent vector per token shared by every head)
# ---------------------------------------------------------------------------

def _mla_small(seed=31, dtype=wl.F32):
    return wl.mla_case(seed, [5, 0, 17, 1, 40], num_qo_heads=6, d_c=32, d_r=8, page_size=4, dtype=dtype,
                       num_pages=40)


def _mla_oracle(c, mutant=0):
    return oracle.mla_decode(c.kv_len, c.table.page_indptr, c.table.page_indices, c.q, c.kv_pool, c.d_c,
                             c.sm_scale, mutant=mutant)


def mla_brute_force(c):
    """numpy fp64: gather each request's latent rows token by token, dense softmax."""
    q, pool = _values(c.q), _values(c.kv_pool)
    B, H, W = q.shape
    o, lse = np.zeros((B, H, c.d_c)), np.full((B, H), -np.inf)
    for r in range(B):
        n = int(c.kv_len[r])
        if n == 0:
            continue
        pages = c.table.page_indices[c.table.page_indptr[r]:c.table.page_indptr[r + 1]]
        C = np.stack([pool[pages[t // c.page_size], t % c.page_size] for t in range(n)])  # [n][W]
        S = q[r] @ C.T * c.sm_scale                                                        # [H][n]
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        o[r] = (E @ C[:, :c.d_c]) / E.sum(axis=1, keepdims=True)
        lse[r] = m[:, 0] + np.log(E.sum(axis=1))
    return o, lse


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_mla_matches_brute_force(dtype):
    c = _mla_small(dtype=dtype)
    o, lse = _mla_oracle(c)
    o_bf, lse_bf = mla_brute_force(c)
    np.testing.assert_allclose(o, o_bf, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse_bf, atol=1e-12, rtol=0)


def test_mla_is_attention_with_one_shared_head_and_zeroed_rope_values():
    # the pinned attention oracle with Hkv = 1, head_dim d_c + d_r: keys are the
    # whole latent row, values the same row with its rope part zeroed
    c = _mla_small()
    B, H, W = c.q.shape
    k_pool = c.kv_pool[:, None, :, :].copy()           # [pages][1][P][W] (HND, one head)
    v_pool = k_pool.copy()
    v_pool[..., c.d_c:] = 0
    qo_indptr = np.arange(B + 1, dtype=np.int32)
    o_a, lse_a = oracle.attention(qo_indptr, c.kv_len, c.table.page_indptr, c.table.page_indices, c.q, k_pool,
                                  v_pool, H, 1, c.sm_scale, causal=False)
    o, lse = _mla_oracle(c)
    np.testing.assert_allclose(o, o_a[:, :, :c.d_c], atol=1e-13, rtol=0)
    assert np.all(o_a[:, :, c.d_c:] == 0)
    np.testing.assert_allclose(lse, lse_a, atol=1e-13, rtol=0)


def test_mla_matches_torch_sdpa_with_a_narrower_value():
    c = _mla_small(seed=32)
    o, lse = _mla_oracle(c)
    q, pool = torch.from_numpy(_values(c.q)), torch.from_numpy(_values(c.kv_pool))
    for r in range(c.batch_size):
        n = int(c.kv_len[r])
        if n == 0:
            continue
        pages = torch.from_numpy(c.table.page_indices[c.table.page_indptr[r]:c.table.page_indptr[r + 1]].astype(np.int64))
        C = pool[pages].reshape(-1, pool.shape[-1])[:n]          # [n][W], pages in order
        ref = torch.nn.functional.scaled_dot_product_attention(q[r][None, :, None, :], C[None, None],
                                                               C[None, None, :, :c.d_c], scale=c.sm_scale)
        np.testing.assert_allclose(o[r], ref[0, :, 0].numpy(), atol=1e-12, rtol=0)


def test_mla_single_key_returns_its_latent_part():
    c = wl.mla_case(33, [1, 1], num_qo_heads=3, d_c=16, d_r=8, page_size=2, dtype=wl.F32)
    o, lse = _mla_oracle(c)
    for r in range(2):
        page = c.table.page_indices[c.table.page_indptr[r]]
        row = c.kv_pool[page, 0].astype(np.float64)
        np.testing.assert_array_equal(o[r], np.broadcast_to(row[:16], (3, 16)))
        np.testing.assert_allclose(lse[r], c.sm_scale * (c.q[r].astype(np.float64) @ row), atol=1e-12)


def test_mla_selected_pairs_equal_the_full_result():
    c = _mla_small(seed=34)
    o, lse = _mla_oracle(c)
    sel_r, sel_h = np.array([4, 0, 2, 4]), np.array([5, 0, 3, 1])
    o_s, lse_s = oracle.mla_decode(c.kv_len, c.table.page_indptr, c.table.page_indices, c.q, c.kv_pool, c.d_c,
                                   c.sm_scale, sel_req=sel_r, sel_head=sel_h)
    np.testing.assert_array_equal(o_s, o[sel_r, sel_h])
    np.testing.assert_array_equal(lse_s, lse[sel_r, sel_h])
