"""Seeded random batches for every attention entry point (and MLA decode), against the fp64
oracle on the same inputs.

Each case draws its shape from its own seed: batch size, query and KV lengths
(empty requests, single keys, lengths just past a page or a 128-key tile),
grouped-query head counts, page size, pool layout and output dtype. Calls with
many query rows per request and decode-like calls run different shapes of the
tensor-core kernel, and small batches run short persistent grids; all of them
must meet the same bars as the fixed cases: |o - oracle| <= 1e-2 for bf16
inputs (fp32 or bf16 outputs alike), 1e-4 for fp32 inputs, |lse - oracle| <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import decode_ragged_paged_gb300 as pd
    from gpu_util import DevCase, dev_tensor, host_f64, LSE_TOL


def _length(rng, lo, hi):
    """A length in [lo, hi], often at a page or tile edge."""
    edges = [v for v in (lo, lo + 1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, hi) if lo <= v <= hi]
    return int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(lo, hi + 1))


def _case(seed, kind):
    rng = np.random.default_rng(seed)
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 3, 4, 8]))
    page = int(rng.choice([8, 16, 32, 64, 128]))
    b = int(rng.integers(1, 7))
    dtype = wl.BF16
    d = 128
    if kind == "decode":
        d = int(rng.choice([64, 128]))
        if rng.random() < 0.3:
            dtype = wl.F32
        qo = [1] * b
        kv = [_length(rng, 0 if rng.random() < 0.1 else 1, 2500) for _ in range(b)]
    elif kind == "prefill":
        qo = [_length(rng, 1, 300) for _ in range(b)]
        kv = [q + _length(rng, 0, 400) for q in qo]
    else:  # mixed: some prefill rows, some decodes, some multi-token verifications
        qo, kv = [], []
        for _ in range(b):
            r = rng.random()
            q = 1 if r < 0.5 else (int(rng.integers(2, 6)) if r < 0.7 else _length(rng, 1, 300))
            qo.append(q)
            kv.append(q + _length(rng, 0, 600))
    # decode rows see every cached key (the bottom-right mask is a no-op for one
    # row); the oracle takes them unmasked, so that an empty request is valid
    case = wl.make_attn_case(seed, qo, kv, hkv * g, hkv, d, page, dtype, causal=kind != "decode")
    if rng.random() < 0.3:
        case = wl.to_nhd(case)
    o_dtype = torch.float32 if (dtype == wl.F32 or rng.random() < 0.5) else torch.bfloat16
    return case, o_dtype


@pytest.mark.parametrize("kind", ["decode", "prefill", "mixed"])
@pytest.mark.parametrize("seed", list(range(700, 708)))
def test_random_batches(kind, seed):
    case, o_dtype = _case(seed + {"decode": 0, "prefill": 100, "mixed": 200}[kind], kind)
    d = DevCase(case)
    layout = getattr(case, "layout", "HND")
    if kind == "decode":
        o, lse = pd.pd_attn_decode(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices,
                                   max_kv_len=d.max_kv_len, o_dtype=o_dtype, layout=layout)
    else:
        fn = pd.pd_attn_prefill if kind == "prefill" else pd.pd_attn_mixed
        o, lse = fn(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices, d.qo_indptr,
                    max_qo_len=d.max_qo_len, max_kv_len=d.max_kv_len, o_dtype=o_dtype, layout=layout)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention_case(case)
    got = host_f64(o)
    assert np.isfinite(got).all(), "non-finite output"
    tol = 1e-4 if case.dtype == wl.F32 else 1e-2
    err = np.abs(got - o_ref)
    assert float(err.max()) <= tol, f"{kind} seed {seed}: max |o - oracle| = {err.max()}"
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    if fin.any():
        assert float(np.abs(lg[fin] - lse_ref[fin]).max()) <= LSE_TOL


@pytest.mark.parametrize("seed", list(range(1000, 1004)))
def test_random_mla_batches(seed):
    # MLA decode: head count, page size and lengths drawn per seed (empty
    # requests and single keys included); a long request is split into chunks
    rng = np.random.default_rng(seed)
    hq = int(rng.choice([1, 8, 16, 64, 128]))
    page = int(rng.choice([16, 32, 64, 128, 256]))
    kv = [_length(rng, 0, 3000) for _ in range(int(rng.integers(1, 9)))]
    c = wl.mla_case(seed, kv, num_qo_heads=hq, page_size=page)
    o_dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    o, lse = pd.pd_mla_decode(dev_tensor(c.q), dev_tensor(c.kv_pool), dev_tensor(c.kv_len.astype(np.int32)),
                              dev_tensor(c.table.page_indptr), dev_tensor(c.table.page_indices), kv_lora_rank=c.d_c,
                              sm_scale=c.sm_scale, max_kv_len=int(c.kv_len.max()), o_dtype=o_dtype)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.mla_decode(c.kv_len, c.table.page_indptr, c.table.page_indices, c.q, c.kv_pool, c.d_c,
                                       c.sm_scale)
    got = host_f64(o)
    assert np.isfinite(got).all()
    assert float(np.abs(got - o_ref).max()) <= 1e-2, f"seed {seed}: max |o - oracle| = {np.abs(got - o_ref).max()}"
    lg = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    if fin.any():
        assert float(np.abs(lg[fin] - lse_ref[fin]).max()) <= LSE_TOL


@pytest.mark.parametrize("seed", list(range(1100, 1108)))
def test_random_split_mixed_batches(seed):
    # pd_attn_mixed_split: 1-3 prefill requests first, then 1-6 decodes, with
    # a drawn partition size (0: the call's own choice); GQA, page size,
    # layout and output dtype drawn as above
    rng = np.random.default_rng(seed)
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8]))
    page = int(rng.choice([8, 16, 32, 64, 128]))
    n_pf, n_dec = int(rng.integers(1, 4)), int(rng.integers(1, 7))
    qo = [_length(rng, 1, 300) for _ in range(n_pf)] + [1] * n_dec
    kv = [q + _length(rng, 0, 400) for q in qo[:n_pf]] + [1 + _length(rng, 0, 2500) for _ in range(n_dec)]
    case = wl.make_attn_case(seed, qo, kv, hkv * g, hkv, 128, page, wl.BF16, causal=True)
    if rng.random() < 0.3:
        case = wl.to_nhd(case)
    o_dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    sms = int(rng.choice([0, 8, 16, 24, 48]))
    d = DevCase(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = pd.pd_attn_mixed_split(d.q, d.k_pool, d.v_pool, d.kv_len, d.page_indptr, d.page_indices, d.qo_indptr,
                                    n_pf, prefill_sms=sms, max_qo_len=d.max_qo_len, max_kv_len=d.max_kv_len,
                                    o_dtype=o_dtype, layout=case.layout, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, lse_ref = oracle.attention_case(case)
    got = host_f64(o)
    assert np.isfinite(got).all(), "non-finite output"
    assert float(np.abs(got - o_ref).max()) <= 1e-2, f"seed {seed}: max |o - oracle| = {np.abs(got - o_ref).max()}"
    lg = lse.cpu().numpy().astype(np.float64)
    assert float(np.abs(lg - lse_ref).max()) <= LSE_TOL
