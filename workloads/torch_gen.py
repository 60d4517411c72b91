"""Seeded synthetic inputs drawn directly on the GPU with torch, for timing.

Same shapes, lengths and value distributions as the numpy generators in
``workloads`` (request lengths are drawn with the same numpy seeds), but the
tensor values come from torch's CUDA generator so that multi-GB workloads are
ready in milliseconds. Holds none of the method's arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _csr(lengths, page: int, device):
    need = -(-np.asarray(lengths, dtype=np.int64) // page)
    indptr = np.zeros(len(need) + 1, dtype=np.int32)
    indptr[1:] = np.cumsum(need)
    return torch.from_numpy(indptr).to(device), int(indptr[-1])


def paged_batch(seed: int, qo_lens, kv_lens, hq: int, hkv: int, d: int, page: int,
                dtype=torch.bfloat16, device="cuda", new_tokens: bool = False) -> dict:
    """q, HND pools and page table of a ragged batch; pages are a seeded random
    permutation of the pool. With ``new_tokens`` also k_new / v_new rows for an
    append of each request's last qo_len tokens."""
    g = _gen(seed, device)
    qo = np.asarray(qo_lens, dtype=np.int64)
    kv = np.asarray(kv_lens, dtype=np.int64)
    page_indptr, npages = _csr(kv, page, device)
    qo_indptr = torch.from_numpy(np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)).to(device)
    out = dict(
        qo_indptr=qo_indptr,
        kv_len=torch.from_numpy(kv.astype(np.int32)).to(device),
        page_indptr=page_indptr,
        page_indices=torch.randperm(npages, generator=g, device=device, dtype=torch.int32),
        k_pool=torch.randn((npages, hkv, page, d), generator=g, device=device, dtype=dtype),
        v_pool=torch.randn((npages, hkv, page, d), generator=g, device=device, dtype=dtype),
        q=torch.randn((int(qo.sum()), hq, d), generator=g, device=device, dtype=dtype),
        kv_len_host=kv, qo_len_host=qo, hq=hq, hkv=hkv, d=d, page=page,
    )
    if new_tokens:
        out["k_new"] = torch.randn((int(qo.sum()), hkv, d), generator=g, device=device, dtype=dtype)
        out["v_new"] = torch.randn((int(qo.sum()), hkv, d), generator=g, device=device, dtype=dtype)
    return out


def decode_batch(seed: int = 2, batch: int = 128, kv_lo: int = 512, kv_hi: int = 4096, device="cuda") -> dict:
    """128 decode requests, kv_len U[512, 4096], GQA 32/8, D 128, page 16, bf16."""
    kv = np.random.default_rng(seed + 1000).integers(kv_lo, kv_hi + 1, size=batch)
    return paged_batch(seed, np.ones(batch, dtype=np.int64), kv, 32, 8, 128, 16, device=device, new_tokens=True)


def causal_prefill(seed: int = 3, batch: int = 8, length: int = 512, heads: int = 40, device="cuda") -> dict:
    """8 x 512-token causal prefill, 40 = 40 heads, D 128, page 16, bf16."""
    return paged_batch(seed, [length] * batch, [length] * batch, heads, heads, 128, 16, device=device,
                       new_tokens=True)


def mixed_1p_nd(seed: int = 4, prefill_len: int = 1024, n_decode: int = 63, kv_lo: int = 512,
                kv_hi: int = 576, heads: int = 40, device="cuda") -> dict:
    """One 1024-token prefill plus 63 decodes with kv_len U[512, 576]; 40 heads, D 128."""
    dec = np.random.default_rng(seed + 1000).integers(kv_lo, kv_hi + 1, size=n_decode)
    qo = np.concatenate([[prefill_len], np.ones(n_decode, dtype=np.int64)])
    kv = np.concatenate([[prefill_len], dec])
    return paged_batch(seed, qo, kv, heads, heads, 128, 16, device=device)


def kv_handoff(seed: int = 5, batch: int = 8, length: int = 512, layers: int = 40, heads: int = 40,
               head_dim: int = 128, src_page: int = 16, dst_page: int = 64, device="cuda") -> dict:
    """Layered source pools (page 16) and an empty destination pool (page 64),
    each with its own seeded random page table; contiguous handoff buffer."""
    g = _gen(seed, device)
    kv = np.full(batch, length, dtype=np.int64)
    s_indptr, s_pages = _csr(kv, src_page, device)
    d_indptr, d_pages = _csr(kv, dst_page, device)
    per = layers * 2 * heads * length * head_dim * 2
    return dict(
        kv_len=torch.from_numpy(kv.astype(np.int32)).to(device),
        src_indptr=s_indptr,
        src_indices=torch.randperm(s_pages, generator=g, device=device, dtype=torch.int32),
        dst_indptr=d_indptr,
        dst_indices=torch.randperm(d_pages, generator=g, device=device, dtype=torch.int32),
        k_src=torch.randn((layers, s_pages, heads, src_page, head_dim), generator=g, device=device,
                          dtype=torch.bfloat16),
        v_src=torch.randn((layers, s_pages, heads, src_page, head_dim), generator=g, device=device,
                          dtype=torch.bfloat16),
        k_dst=torch.empty((layers, d_pages, heads, dst_page, head_dim), device=device, dtype=torch.bfloat16),
        v_dst=torch.empty((layers, d_pages, heads, dst_page, head_dim), device=device, dtype=torch.bfloat16),
        offsets=torch.arange(batch, dtype=torch.int64, device=device) * per,
        buffer=torch.empty(per * batch, dtype=torch.uint8, device=device),
        kv_len_host=kv, layers=layers, heads=heads, head_dim=head_dim,
    )


def mla_decode_batch(seed: int = 7, batch: int = 128, kv_lo: int = 512, kv_hi: int = 4096, heads: int = 128,
                     d_c: int = 512, d_r: int = 64, page: int = 64, device="cuda") -> dict:
    """MLA decode: 128 requests, kv_len U[512, 4096], 128 query heads over one
    512 + 64 latent row per token, page 64, bf16; pages a seeded permutation."""
    g = _gen(seed, device)
    kv = np.random.default_rng(seed + 1000).integers(kv_lo, kv_hi + 1, size=batch)
    page_indptr, npages = _csr(kv, page, device)
    return dict(
        kv_len=torch.from_numpy(kv.astype(np.int32)).to(device),
        page_indptr=page_indptr,
        page_indices=torch.randperm(npages, generator=g, device=device, dtype=torch.int32),
        kv_pool=torch.randn((npages, page, d_c + d_r), generator=g, device=device, dtype=torch.bfloat16),
        q=torch.randn((batch, heads, d_c + d_r), generator=g, device=device, dtype=torch.bfloat16),
        kv_len_host=kv, heads=heads, d_c=d_c, d_r=d_r, page=page,
    )
