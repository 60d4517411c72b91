"""Seeded synthetic inputs for the paged-attention and KV-handoff hot path.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests. It draws random numbers and lays them out, and holds none of
the attention arithmetic (no dot products, no softmax, no merge). To place a
request's tokens and poison the slots that hold none, ``logical_slots`` does
use the paged cache's token -> (page, slot) map (page t // P of the request's
page list, slot t % P). The oracle and the CUDA path each compute that map
themselves, and no test takes an expected value from this module: copies and
attention outputs are compared with the oracle's results.

Layouts produced here (all C-contiguous numpy arrays):

* ``q``            [total_qo][Hq][D]            rows of all requests, packed
* ``k_pool``       [num_pages][Hkv][P][D]       HND pages ("head before token")
* ``v_pool``       same as ``k_pool``
  (``to_nhd`` turns a case's pools into [num_pages][P][Hkv][D], the NHD
  layout, "token before head", by swapping the two axes; nothing else changes)
* ``qo_indptr``    int32 [B+1]
* ``kv_len``       int32 [B]
* ``page_indptr``  int32 [B+1]
* ``page_indices`` int32 [nnz] physical page ids

bf16 data is carried as raw ``uint16`` bit patterns. A draw is made in fp32
from N(0, 1) and rounded once to bf16 (round to nearest, ties to even); both
the GPU path and the oracle then consume exactly those bf16 values.

Unused pool pages and the unused tail slots of each request's last page are
filled with NaN ("poison"), so that any read of a slot that holds no token
shows up as NaN in the result.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"

BF16_NAN = np.uint16(0x7FC0)


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1).view(np.uint32)
    out = np.empty(flat.shape, dtype=np.uint16)
    step = 1 << 22
    tmp = np.empty(step, dtype=np.uint32)
    for s in range(0, flat.size, step):
        u = flat[s:s + step]
        t = tmp[:u.size]
        np.right_shift(u, 16, out=t)
        np.bitwise_and(t, 1, out=t)
        t += 0x7FFF
        t += u                      # cannot wrap for finite inputs
        np.right_shift(t, 16, out=t)
        out[s:s + step] = t
    bad = ~np.isfinite(x.reshape(-1))
    if bad.any():
        out[bad] = (flat[bad] >> 16).astype(np.uint16)
        out[np.isnan(x.reshape(-1))] = BF16_NAN
    return out.reshape(x.shape)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _draw(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == BF16:
        return bf16_from_f32(x)
    if dtype == F32:
        return x
    raise ValueError(f"unknown dtype {dtype!r}")


def _poison(shape, dtype: str) -> np.ndarray:
    if dtype == BF16:
        return np.full(shape, BF16_NAN, dtype=np.uint16)
    return np.full(shape, np.nan, dtype=np.float32)


def element_size(dtype: str) -> int:
    return 2 if dtype == BF16 else 4


@dataclass
class PageTable:
    """CSR page table: request r owns pages page_indices[page_indptr[r]:page_indptr[r+1]]."""

    page_indptr: np.ndarray
    page_indices: np.ndarray
    num_pages: int


def random_page_table(rng: np.random.Generator, kv_len, page_size: int,
                      num_pages: int | None = None) -> PageTable:
    """Give each request ceil(kv_len / page_size) pages, drawn as a seeded random
    permutation of the pool (the first pages of the permutation are used)."""
    kv_len = np.asarray(kv_len, dtype=np.int64)
    need = -(-kv_len // page_size)
    total = int(need.sum())
    if num_pages is None:
        num_pages = total
    if num_pages < total:
        raise ValueError("pool too small")
    perm = rng.permutation(num_pages).astype(np.int32)
    indptr = np.zeros(len(kv_len) + 1, dtype=np.int32)
    indptr[1:] = np.cumsum(need)
    return PageTable(indptr, perm[:total].copy(), num_pages)


@dataclass
class AttnCase:
    """One ragged batch: q rows, paged K/V pools and the page table."""

    dtype: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    qo_indptr: np.ndarray
    kv_len: np.ndarray
    table: PageTable
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    causal: bool = True
    sm_scale: float | None = None
    # rows of the new tokens for an append (packed [total_new][Hkv][D]); optional
    k_new: np.ndarray | None = None
    v_new: np.ndarray | None = None
    meta: dict = field(default_factory=dict)
    layout: str = "HND"        # "HND": pools [pages][Hkv][P][D]; "NHD": [pages][P][Hkv][D]

    @property
    def batch_size(self) -> int:
        return len(self.kv_len)

    @property
    def qo_len(self) -> np.ndarray:
        return np.diff(self.qo_indptr)

    @property
    def total_qo(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def scale(self) -> float:
        return float(self.sm_scale) if self.sm_scale else 1.0 / float(np.sqrt(self.head_dim))


def logical_slots(table: PageTable, kv_len, page_size: int):
    """(page, slot) of every logical token, request-major then token order."""
    kv_len = np.asarray(kv_len, dtype=np.int64)
    pages, slots, req, tok = [], [], [], []
    for r, n in enumerate(kv_len):
        n = int(n)
        t = np.arange(n, dtype=np.int64)
        own = table.page_indices[table.page_indptr[r]:table.page_indptr[r + 1]]
        pages.append(own[t // page_size].astype(np.int64))
        slots.append(t % page_size)
        req.append(np.full(n, r, dtype=np.int64))
        tok.append(t)
    cat = lambda a: np.concatenate(a) if a else np.zeros(0, dtype=np.int64)
    return cat(pages), cat(slots), cat(req), cat(tok)


def make_attn_case(seed: int, qo_lens, kv_lens, num_qo_heads: int, num_kv_heads: int,
                   head_dim: int, page_size: int, dtype: str, causal: bool = True,
                   num_pages: int | None = None, sm_scale: float | None = None,
                   with_new_tokens: bool = False) -> AttnCase:
    """Generic seeded ragged batch.

    Draw order from one ``numpy.random.default_rng(seed)`` stream: the page
    permutation, then the whole K pool, the whole V pool, then q. Slots that hold
    no logical token are then poisoned. With ``with_new_tokens`` the K/V rows of
    each request's last ``qo_len`` tokens are moved into ``k_new``/``v_new``
    (packed like q, [total_qo][Hkv][D]) and their pool slots poisoned, so that
    an append has to write them."""
    rng = np.random.default_rng(seed)
    qo_lens = np.asarray(qo_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    B = len(kv_lens)
    assert len(qo_lens) == B
    table = random_page_table(rng, kv_lens, page_size, num_pages)
    shape = (table.num_pages, num_kv_heads, page_size, head_dim)
    k_all = _draw(rng, shape, dtype)
    v_all = _draw(rng, shape, dtype)
    qo_indptr = np.zeros(B + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    total_qo = int(qo_indptr[-1])
    q = _draw(rng, (total_qo, num_qo_heads, head_dim), dtype)

    pg, sl, req, tok = logical_slots(table, kv_lens, page_size)
    used = np.zeros((table.num_pages, page_size), dtype=bool)
    used[pg, sl] = True
    k_new = v_new = None
    if with_new_tokens:
        first_new = kv_lens[req] - qo_lens[req]
        is_new = tok >= first_new
        rows = qo_indptr[req[is_new]] + (tok[is_new] - first_new[is_new])
        k_new = _poison((total_qo, num_kv_heads, head_dim), dtype)
        v_new = _poison((total_qo, num_kv_heads, head_dim), dtype)
        k_new[rows] = k_all[pg[is_new], :, sl[is_new], :]
        v_new[rows] = v_all[pg[is_new], :, sl[is_new], :]
        used[pg[is_new], sl[is_new]] = False
    mask = used[:, None, :, None]
    k_pool = np.where(mask, k_all, _poison((), dtype))
    v_pool = np.where(mask, v_all, _poison((), dtype))
    return AttnCase(dtype, num_qo_heads, num_kv_heads, head_dim, page_size,
                    qo_indptr, kv_lens.astype(np.int32), table, q, k_pool, v_pool,
                    causal=causal, sm_scale=sm_scale, k_new=k_new, v_new=v_new)


# ---------------------------------------------------------------------------
# The five workloads of the hot path. Shapes follow the blog's decode/prefill
# description (qo_len = 1 for decode, large qo_len for prefill, GQA for the
# Qwen3-Coder deployment) and the 13B model of the overview article (40 heads
# of 128, input 512).
# ---------------------------------------------------------------------------

def decode_correctness(seed: int = 1) -> AttnCase:
    """4 decode requests, kv_len {17, 64, 100, 255}, 8 q = 8 kv heads, D 64,
    page 16, fp32, pages drawn from a 64-page pool."""
    return make_attn_case(seed, [1, 1, 1, 1], [17, 64, 100, 255], 8, 8, 64, 16, F32,
                          causal=True, num_pages=64)


def decode_batch(seed: int = 2, batch: int = 128, kv_lo: int = 512, kv_hi: int = 4096) -> AttnCase:
    """128 decode requests, kv_len uniform integers in [512, 4096], GQA 32/8, D 128,
    page 16, bf16."""
    rng = np.random.default_rng(seed + 1000)
    kv = rng.integers(kv_lo, kv_hi + 1, size=batch)
    return make_attn_case(seed, np.ones(batch, dtype=np.int64), kv, 32, 8, 128, 16, BF16,
                          causal=True)


def causal_prefill(seed: int = 3, batch: int = 8, length: int = 512, heads: int = 40) -> AttnCase:
    """8 requests with qo_len = kv_len = 512, 40 = 40 heads, D 128, page 16, bf16.
    The K/V of all tokens are new (written by an append before attention)."""
    return make_attn_case(seed, [length] * batch, [length] * batch, heads, heads, 128, 16, BF16,
                          causal=True, with_new_tokens=True)


def mixed_1p_nd(seed: int = 4, prefill_len: int = 1024, n_decode: int = 63,
                kv_lo: int = 512, kv_hi: int = 576, heads: int = 40) -> AttnCase:
    """One prefill request (qo = kv = 1024) followed by 63 decode requests with
    kv_len uniform in [512, 576]; 40 heads, D 128, page 16, bf16."""
    rng = np.random.default_rng(seed + 1000)
    dec = rng.integers(kv_lo, kv_hi + 1, size=n_decode)
    qo = np.concatenate([[prefill_len], np.ones(n_decode, dtype=np.int64)])
    kv = np.concatenate([[prefill_len], dec])
    return make_attn_case(seed, qo, kv, heads, heads, 128, 16, BF16, causal=True)


@dataclass
class HandoffCase:
    """Layered KV pools of a prefill node and the page table of a decode node."""

    dtype: str
    num_layers: int
    num_kv_heads: int
    head_dim: int
    kv_len: np.ndarray
    src_page_size: int
    src_table: PageTable
    k_src: np.ndarray          # [L][num_pages][Hkv][P][D]
    v_src: np.ndarray
    dst_page_size: int
    dst_table: PageTable
    dst_offsets: np.ndarray    # int64 [B], byte offset of each request's packed block
    layout: str = "HND"        # of k_src / v_src: "NHD" holds [L][num_pages][P][Hkv][D]


def kv_handoff(seed: int = 5, batch: int = 8, length: int = 512, layers: int = 40,
               heads: int = 40, head_dim: int = 128, src_page: int = 16,
               dst_page: int = 64, dtype: str = BF16, kv_lens=None,
               src_slack: int = 0, dst_slack: int = 0) -> HandoffCase:
    """KV handoff between a prefill pool (page 16) and a decode pool (page 64), each
    with its own seeded random page table. Values ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    if kv_lens is None:
        kv_lens = [length] * batch
    kv = np.asarray(kv_lens, dtype=np.int64)
    need_src = int((-(-kv // src_page)).sum())
    need_dst = int((-(-kv // dst_page)).sum())
    src = random_page_table(rng, kv, src_page, need_src + src_slack)
    dst = random_page_table(rng, kv, dst_page, need_dst + dst_slack)
    shape = (layers, src.num_pages, heads, src_page, head_dim)
    k_src = _draw(rng, shape, dtype)
    v_src = _draw(rng, shape, dtype)
    pg, sl, _, _ = logical_slots(src, kv, src_page)
    used = np.zeros((src.num_pages, src_page), dtype=bool)
    used[pg, sl] = True
    if not used.all():
        mask = used[None, :, None, :, None]
        k_src = np.where(mask, k_src, _poison((), dtype))
        v_src = np.where(mask, v_src, _poison((), dtype))
    es = element_size(dtype)
    per_req = kv * layers * 2 * heads * head_dim * es
    offs = np.zeros(len(kv), dtype=np.int64)
    offs[1:] = np.cumsum(per_req)[:-1]
    return HandoffCase(dtype, layers, heads, head_dim, kv.astype(np.int32), src_page, src,
                       k_src, v_src, dst_page, dst, offs)


def packed_bytes(kv_len, num_layers: int, num_kv_heads: int, head_dim: int, elem_size: int) -> int:
    """Bytes of K and V that a handoff moves: every logical token of every layer,
    head and dimension, for both K and V."""
    return int(np.sum(np.asarray(kv_len, dtype=np.int64))) * 2 * num_layers * num_kv_heads * head_dim * elem_size


def nhd_pool(pool: np.ndarray) -> np.ndarray:
    """An HND pool ([..][num_pages][Hkv][P][D]) with its head and slot axes swapped:
    the same values in the NHD layout ([..][num_pages][P][Hkv][D])."""
    return np.ascontiguousarray(np.swapaxes(pool, -3, -2))


def to_nhd(case):
    """A copy of an AttnCase or HandoffCase whose pools hold the same values in
    the NHD layout. Page tables, lengths, q and new-token rows are shared."""
    import dataclasses
    if isinstance(case, AttnCase):
        assert case.layout == "HND"
        return dataclasses.replace(case, k_pool=nhd_pool(case.k_pool), v_pool=nhd_pool(case.v_pool),
                                   layout="NHD")
    assert case.layout == "HND"
    return dataclasses.replace(case, k_src=nhd_pool(case.k_src), v_src=nhd_pool(case.v_src), layout="NHD")


@dataclass
class MlaCase:
    """A decode batch over a paged latent cache (one row per token shared by all
    query heads): q [B][Hq][d_c + d_r], kv_pool [num_pages][P][d_c + d_r]."""

    dtype: str
    num_qo_heads: int
    d_c: int                   # latent (value) width
    d_r: int                   # decoupled rope width, scores only
    page_size: int
    kv_len: np.ndarray
    table: PageTable
    q: np.ndarray
    kv_pool: np.ndarray
    sm_scale: float

    @property
    def batch_size(self) -> int:
        return len(self.kv_len)


def mla_case(seed: int, kv_lens, num_qo_heads: int = 128, d_c: int = 512, d_r: int = 64, page_size: int = 64,
             dtype: str = BF16, num_pages: int | None = None, sm_scale: float = 192 ** -0.5) -> MlaCase:
    """Seeded MLA decode batch. Draw order from one default_rng(seed) stream: the
    page permutation, the latent pool, then q; slots holding no token are then
    poisoned. The default scale is 1/sqrt(192), DeepSeek-V3's query-key head size
    (128 + 64) before its up-projections are folded into q."""
    rng = np.random.default_rng(seed)
    kv = np.asarray(kv_lens, dtype=np.int64)
    table = random_page_table(rng, kv, page_size, num_pages)
    w = d_c + d_r
    pool = _draw(rng, (table.num_pages, page_size, w), dtype)
    q = _draw(rng, (len(kv), num_qo_heads, w), dtype)
    pg, sl, _, _ = logical_slots(table, kv, page_size)
    used = np.zeros((table.num_pages, page_size), dtype=bool)
    used[pg, sl] = True
    pool[~used] = _poison((), dtype)
    return MlaCase(dtype, num_qo_heads, d_c, d_r, page_size, kv.astype(np.int32), table, q, pool, float(sm_scale))


def mla_decode_batch(seed: int = 7, batch: int = 128, kv_lo: int = 512, kv_hi: int = 4096) -> MlaCase:
    """128 decode requests, kv_len U[512, 4096], 128 query heads over a 512 + 64
    latent row (DeepSeek-V3/R1 shapes with data-parallel attention: every head
    on one GPU), page 64, bf16."""
    kv = np.random.default_rng(seed + 1000).integers(kv_lo, kv_hi + 1, size=batch)
    return mla_case(seed, kv)
