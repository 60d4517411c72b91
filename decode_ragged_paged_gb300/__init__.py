"""Paged ragged attention and KV handoff for NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI in ``include/pd.h`` (``libpd.so``, built
in-tree by ``decode_ragged_paged_gb300.build``). The functions carry the C
names and only marshal arguments: torch tensors give device pointers, shapes
and the current CUDA stream; every step of the computation runs in the
library's CUDA kernels. There is no CPU path: if ``libpd.so`` is missing or a
call fails, an exception is raised.

Tensor layouts (see ``include/pd.h``):
    q, o            [total_qo][Hq][D]        fp32 or bf16
    k_pool, v_pool  [num_pages][Hkv][P][D]   HND pages (layout="HND", the default)
                    [num_pages][P][Hkv][D]   NHD pages (layout="NHD")
    qo_indptr       int32 [B+1]; kv_len int32 [B]; page_indptr int32 [B+1];
    page_indices    int32 [nnz]
    lse             fp32 [total_qo][Hq], natural log
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpd.so")

PD_OK, PD_ERR_INVALID_ARG, PD_ERR_UNSUPPORTED, PD_ERR_WORKSPACE, PD_ERR_CUDA, PD_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
PD_F32, PD_BF16 = 0, 1
PD_LAYOUT_HND, PD_LAYOUT_NHD = 0, 1
PD_KIND_DECODE, PD_KIND_PREFILL, PD_KIND_MIXED, PD_KIND_MIXED_SPLIT = 0, 1, 2, 3
DEVICE_STATUS = {0: "ok", 1: "bad indptr", 2: "bad length", 3: "bad page table", 4: "not a decode",
                 5: "timeout", 6: "bad offset"}

# Every symbol include/pd.h declares.
EXPORTS = ("pd_attn_workspace_size", "pd_attn_decode", "pd_attn_decode_static", "pd_attn_prefill",
           "pd_attn_mixed", "pd_attn_mixed_split", "pd_mla_workspace_size", "pd_mla_decode",
           "pd_kv_append", "pd_kv_pack", "pd_kv_unpack", "pd_kv_pack_heads", "pd_kv_unpack_heads",
           "pd_kv_pack_layers", "pd_counter_alloc", "pd_counter_free", "pd_layer_signal",
           "pd_messenger_start_pack", "pd_messenger_join",
           "pd_profile_events", "pd_last_kernel", "pd_status_string",
           "pd_device_status_string", "pd_version")


class PdError(RuntimeError):
    def __init__(self, msg: str, code: int = 0):
        super().__init__(msg)
        self.code = code


class AttnDesc(ctypes.Structure):
    _fields_ = [("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("o_dtype", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("causal", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


class Batch(ctypes.Structure):
    _fields_ = [("batch_size", ctypes.c_int32), ("qo_indptr", ctypes.c_void_p),
                ("kv_len", ctypes.c_void_p), ("page_indptr", ctypes.c_void_p),
                ("page_indices", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("total_qo", ctypes.c_int32), ("max_qo_len", ctypes.c_int32),
                ("max_kv_len", ctypes.c_int32)]


class KvDesc(ctypes.Structure):
    _fields_ = [("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("num_layers", ctypes.c_int32), ("layer_stride_bytes", ctypes.c_int64)]


class MlaDesc(ctypes.Structure):
    _fields_ = [("num_qo_heads", ctypes.c_int32), ("kv_lora_rank", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("kv_dtype", ctypes.c_int32), ("o_dtype", ctypes.c_int32),
                ("sm_scale", ctypes.c_float)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpd.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise PdError(f"{path} not found: build it with `python -m decode_ragged_paged_gb300.build`")
            lib = ctypes.CDLL(path)
            P, S, I32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
            attn = [ctypes.POINTER(AttnDesc), ctypes.POINTER(Batch), P, P, P, P, P, P, S, P, P]
            for name in ("pd_attn_decode", "pd_attn_prefill", "pd_attn_mixed"):
                getattr(lib, name).argtypes = attn
                getattr(lib, name).restype = ctypes.c_int
            lib.pd_attn_mixed_split.argtypes = attn[:2] + [I32, I32] + attn[2:]
            lib.pd_attn_mixed_split.restype = ctypes.c_int
            lib.pd_attn_workspace_size.argtypes = [ctypes.POINTER(AttnDesc), ctypes.POINTER(Batch), I32]
            lib.pd_attn_workspace_size.restype = S
            lib.pd_mla_workspace_size.argtypes = [ctypes.POINTER(MlaDesc), ctypes.POINTER(Batch)]
            lib.pd_mla_workspace_size.restype = S
            lib.pd_mla_decode.argtypes = [ctypes.POINTER(MlaDesc), ctypes.POINTER(Batch), P, P, P, P, P, S, P, P]
            lib.pd_mla_decode.restype = ctypes.c_int
            lib.pd_kv_append.argtypes = [ctypes.POINTER(KvDesc), ctypes.POINTER(Batch), P, P, P, P, P, P]
            lib.pd_kv_pack.argtypes = [ctypes.POINTER(KvDesc), ctypes.POINTER(Batch), P, P, P, S, P, P, P]
            lib.pd_kv_unpack.argtypes = [ctypes.POINTER(KvDesc), ctypes.POINTER(Batch), P, S, P, P, P, P, P]
            lib.pd_kv_pack_heads.argtypes = [ctypes.POINTER(KvDesc), ctypes.POINTER(Batch), I32, I32, P, P, P, S, P,
                                             P, P]
            lib.pd_kv_unpack_heads.argtypes = [ctypes.POINTER(KvDesc), ctypes.POINTER(Batch), I32, I32, P, S, P, P,
                                               P, P, P]
            lib.pd_kv_pack_layers.argtypes = lib.pd_kv_pack_heads.argtypes
            for name in ("pd_kv_append", "pd_kv_pack", "pd_kv_unpack", "pd_kv_pack_heads", "pd_kv_unpack_heads",
                         "pd_kv_pack_layers"):
                getattr(lib, name).restype = ctypes.c_int
            PP = ctypes.POINTER(ctypes.c_void_p)
            lib.pd_counter_alloc.argtypes = [PP, PP]
            lib.pd_counter_free.argtypes = [P]
            lib.pd_layer_signal.argtypes = [P, ctypes.c_uint32, P]
            lib.pd_messenger_start_pack.argtypes = [PP, P, ctypes.POINTER(KvDesc), ctypes.POINTER(Batch), P, P, P,
                                                    S, P, P, P, I32]
            lib.pd_messenger_join.argtypes = [P, ctypes.POINTER(I32)]
            for name in ("pd_counter_alloc", "pd_counter_free", "pd_layer_signal", "pd_messenger_start_pack",
                         "pd_messenger_join"):
                getattr(lib, name).restype = ctypes.c_int
            lib.pd_status_string.argtypes = [I32]
            lib.pd_status_string.restype = ctypes.c_char_p
            lib.pd_device_status_string.argtypes = [I32]
            lib.pd_device_status_string.restype = ctypes.c_char_p
            lib.pd_version.restype = I32
            lib.pd_last_kernel.restype = ctypes.c_char_p
            lib.pd_profile_events.argtypes = [P, P]
            lib.pd_profile_events.restype = ctypes.c_int
            _lib = lib
        return _lib


def _check(rc: int, what: str) -> None:
    if rc != PD_OK:
        msg = load_library().pd_status_string(rc).decode()
        raise PdError(f"{what} failed: {msg} ({rc})", rc)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return PD_F32
    if dt == torch.bfloat16:
        return PD_BF16
    raise PdError(f"unsupported dtype {dt}")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device: int | None = None) -> int | None:
    if stream is None:
        if _raw_stream is not None and device is not None and device >= 0:
            return _raw_stream(device)  # the current stream's handle, without building a Stream object
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _i32(t, name):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise PdError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


def _layout_code(layout) -> int:
    codes = {"HND": PD_LAYOUT_HND, "NHD": PD_LAYOUT_NHD, PD_LAYOUT_HND: PD_LAYOUT_HND, PD_LAYOUT_NHD: PD_LAYOUT_NHD}
    if layout not in codes:
        raise PdError(f"unknown pool layout {layout!r}")
    return codes[layout]


def _pool_dims(pool, layout):
    """(num_pages, Hkv, P, D) of a pool in `layout` ([..][pages][Hkv][P][D] or [..][pages][P][Hkv][D])."""
    n, a, b, d = pool.shape[-4:]
    return (n, a, b, d) if _layout_code(layout) == PD_LAYOUT_HND else (n, b, a, d)


def make_attn_desc(q, k_pool, *, causal=True, sm_scale=None, o_dtype=None, layout="HND") -> AttnDesc:
    num_pages, hkv, page, d = _pool_dims(k_pool, layout)
    return AttnDesc(q.shape[1], hkv, d, page, _dtype_code(q.dtype),
                    _dtype_code(o_dtype if o_dtype is not None else q.dtype), _layout_code(layout),
                    int(bool(causal)), float(sm_scale) if sm_scale else 0.0)


def make_batch(kv_len, page_indptr, page_indices, num_pages, *, qo_indptr=None, total_qo=0,
               max_qo_len=1, max_kv_len=None) -> Batch:
    _i32(kv_len, "kv_len"), _i32(page_indptr, "page_indptr"), _i32(page_indices, "page_indices")
    _i32(qo_indptr, "qo_indptr")
    if max_kv_len is None:  # convenience path: reads the lengths back (synchronises)
        max_kv_len = int(kv_len.max().item()) if kv_len.numel() else 0
    return Batch(kv_len.numel(), _ptr(qo_indptr), _ptr(kv_len), _ptr(page_indptr), _ptr(page_indices),
                 int(num_pages), int(total_qo), int(max_qo_len), int(max_kv_len))


def pd_attn_workspace_size(desc: AttnDesc, batch: Batch, kind: int) -> int:
    return int(load_library().pd_attn_workspace_size(ctypes.byref(desc), ctypes.byref(batch), kind))


def _attn(name, kind, q, k_pool, v_pool, kv_len, page_indptr, page_indices, qo_indptr, *, causal,
          sm_scale, max_qo_len, max_kv_len, o, lse, o_dtype, workspace, dev_status, stream, layout):
    lib = load_library()
    for t, n in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        if not t.is_cuda or not t.is_contiguous():
            raise PdError(f"{n} must be a contiguous CUDA tensor")
    desc = make_attn_desc(q, k_pool, causal=causal, sm_scale=sm_scale, o_dtype=o_dtype, layout=layout)
    batch = make_batch(kv_len, page_indptr, page_indices, k_pool.shape[0], qo_indptr=qo_indptr,
                       total_qo=q.shape[0], max_qo_len=max_qo_len, max_kv_len=max_kv_len)
    if o is None:
        o = torch.empty(q.shape, dtype=o_dtype if o_dtype is not None else q.dtype, device=q.device)
    if lse is True:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    fn, dref, bref = getattr(lib, name), ctypes.byref(desc), ctypes.byref(batch)
    ptrs = (_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(o), _ptr(lse))
    status, strm = _ptr(dev_status), _stream(stream, q.get_device())
    if workspace is None:
        workspace = torch.empty(max(pd_attn_workspace_size(desc, batch, kind), 16), dtype=torch.uint8,
                                device=q.device)
    rc = fn(dref, bref, *ptrs, _ptr(workspace), workspace.numel(), status, strm)
    if rc == PD_ERR_WORKSPACE:  # the caller's workspace is too small for this batch: use one that fits
        workspace = torch.empty(max(pd_attn_workspace_size(desc, batch, kind), 16), dtype=torch.uint8,
                                device=q.device)
        rc = fn(dref, bref, *ptrs, _ptr(workspace), workspace.numel(), status, strm)
    _check(rc, name)
    return o, lse


def pd_attn_decode(q, k_pool, v_pool, kv_len, page_indptr, page_indices, qo_indptr=None, *, sm_scale=None,
                   max_kv_len=None, o=None, lse=True, o_dtype=None, workspace=None, dev_status=None,
                   stream=None, layout="HND"):
    """Decode attention: one query row per request. Returns (o, lse)."""
    return _attn("pd_attn_decode", PD_KIND_DECODE, q, k_pool, v_pool, kv_len, page_indptr, page_indices,
                 qo_indptr, causal=True, sm_scale=sm_scale, max_qo_len=1, max_kv_len=max_kv_len, o=o,
                 lse=lse, o_dtype=o_dtype, workspace=workspace, dev_status=dev_status, stream=stream,
                 layout=layout)


def pd_attn_prefill(q, k_pool, v_pool, kv_len, page_indptr, page_indices, qo_indptr, *, causal=True,
                    sm_scale=None, max_qo_len=None, max_kv_len=None, o=None, lse=True, o_dtype=None,
                    workspace=None, dev_status=None, stream=None, layout="HND"):
    """Prefill attention over ragged query rows (qo_len <= kv_len). Returns (o, lse)."""
    if max_qo_len is None:
        max_qo_len = int((qo_indptr[1:] - qo_indptr[:-1]).max().item()) if qo_indptr.numel() > 1 else 0
    return _attn("pd_attn_prefill", PD_KIND_PREFILL, q, k_pool, v_pool, kv_len, page_indptr, page_indices,
                 qo_indptr, causal=causal, sm_scale=sm_scale, max_qo_len=max_qo_len, max_kv_len=max_kv_len,
                 o=o, lse=lse, o_dtype=o_dtype, workspace=workspace, dev_status=dev_status, stream=stream,
                 layout=layout)


def pd_attn_mixed(q, k_pool, v_pool, kv_len, page_indptr, page_indices, qo_indptr, *, causal=True,
                  sm_scale=None, max_qo_len=None, max_kv_len=None, o=None, lse=True, o_dtype=None,
                  workspace=None, dev_status=None, stream=None, layout="HND"):
    """Mixed prefill + decode batch in one launch. Returns (o, lse)."""
    if max_qo_len is None:
        max_qo_len = int((qo_indptr[1:] - qo_indptr[:-1]).max().item()) if qo_indptr.numel() > 1 else 0
    return _attn("pd_attn_mixed", PD_KIND_MIXED, q, k_pool, v_pool, kv_len, page_indptr, page_indices,
                 qo_indptr, causal=causal, sm_scale=sm_scale, max_qo_len=max_qo_len, max_kv_len=max_kv_len,
                 o=o, lse=lse, o_dtype=o_dtype, workspace=workspace, dev_status=dev_status, stream=stream,
                 layout=layout)


def pd_attn_mixed_split(q, k_pool, v_pool, kv_len, page_indptr, page_indices, qo_indptr, num_prefill, *,
                        prefill_sms=0, causal=True, sm_scale=None, max_qo_len=None, max_kv_len=None, o=None,
                        lse=True, o_dtype=None, workspace=None, dev_status=None, stream=None, layout="HND"):
    """Mixed batch with requests [0, num_prefill) prefill and the rest decode (qo_len 1),
    the two parts run at the same time on disjoint SM partitions. Returns (o, lse)."""
    lib = load_library()
    for t, n in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        if not t.is_cuda or not t.is_contiguous():
            raise PdError(f"{n} must be a contiguous CUDA tensor")
    if max_qo_len is None:
        max_qo_len = int((qo_indptr[1:] - qo_indptr[:-1]).max().item()) if qo_indptr.numel() > 1 else 0
    desc = make_attn_desc(q, k_pool, causal=causal, sm_scale=sm_scale, o_dtype=o_dtype, layout=layout)
    batch = make_batch(kv_len, page_indptr, page_indices, k_pool.shape[0], qo_indptr=qo_indptr,
                       total_qo=q.shape[0], max_qo_len=max_qo_len, max_kv_len=max_kv_len)
    if o is None:
        o = torch.empty(q.shape, dtype=o_dtype if o_dtype is not None else q.dtype, device=q.device)
    if lse is True:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    dref, bref = ctypes.byref(desc), ctypes.byref(batch)
    if workspace is None or workspace.numel() < pd_attn_workspace_size(desc, batch, PD_KIND_MIXED_SPLIT):
        workspace = torch.empty(max(pd_attn_workspace_size(desc, batch, PD_KIND_MIXED_SPLIT), 16), dtype=torch.uint8,
                                device=q.device)
    rc = lib.pd_attn_mixed_split(dref, bref, int(num_prefill), int(prefill_sms), _ptr(q), _ptr(k_pool),
                                 _ptr(v_pool), _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                                 _ptr(dev_status), _stream(stream, q.get_device()))
    _check(rc, "pd_attn_mixed_split")
    return o, lse


def pd_mla_decode(q, kv_pool, kv_len, page_indptr, page_indices, *, kv_lora_rank=512, sm_scale=None,
                  max_kv_len=None, o=None, lse=True, o_dtype=None, workspace=None, dev_status=None, stream=None):
    """MLA decode over a paged latent cache: q [B][Hq][kv_lora_rank + rope_dim], kv_pool
    [num_pages][P][kv_lora_rank + rope_dim]; scores over the whole row, values its first
    kv_lora_rank entries. Returns (o [B][Hq][kv_lora_rank], lse [B][Hq])."""
    lib = load_library()
    for t, n in ((q, "q"), (kv_pool, "kv_pool")):
        if not t.is_cuda or not t.is_contiguous():
            raise PdError(f"{n} must be a contiguous CUDA tensor")
    B, hq, w = q.shape
    num_pages, page, w2 = kv_pool.shape
    if w2 != w:
        raise PdError("q and kv_pool rows differ in width")
    desc = MlaDesc(hq, int(kv_lora_rank), w - int(kv_lora_rank), page, _dtype_code(q.dtype),
                   _dtype_code(o_dtype if o_dtype is not None else q.dtype), float(sm_scale) if sm_scale else 0.0)
    batch = make_batch(kv_len, page_indptr, page_indices, num_pages, total_qo=B, max_kv_len=max_kv_len)
    if o is None:
        o = torch.empty((B, hq, int(kv_lora_rank)), dtype=o_dtype if o_dtype is not None else q.dtype,
                        device=q.device)
    if lse is True:
        lse = torch.empty((B, hq), dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    dref, bref = ctypes.byref(desc), ctypes.byref(batch)
    args = (_ptr(q), _ptr(kv_pool), _ptr(o), _ptr(lse))
    status, strm = _ptr(dev_status), _stream(stream, q.get_device())
    if workspace is None:
        workspace = torch.empty(max(int(lib.pd_mla_workspace_size(dref, bref)), 16), dtype=torch.uint8,
                                device=q.device)
    rc = lib.pd_mla_decode(dref, bref, *args, _ptr(workspace), workspace.numel(), status, strm)
    if rc == PD_ERR_WORKSPACE:  # the caller's workspace is too small for this batch: use one that fits
        workspace = torch.empty(max(int(lib.pd_mla_workspace_size(dref, bref)), 16), dtype=torch.uint8,
                                device=q.device)
        rc = lib.pd_mla_decode(dref, bref, *args, _ptr(workspace), workspace.numel(), status, strm)
    _check(rc, "pd_mla_decode")
    return o, lse


def _kv_desc(pool, num_layers=1, layer_stride_bytes=0, layout="HND") -> KvDesc:
    """pool: [num_pages][Hkv][P][D] or [L][num_pages][Hkv][P][D] (HND); P and Hkv swapped for NHD."""
    _, hkv, page, d = _pool_dims(pool, layout)
    return KvDesc(hkv, d, page, _dtype_code(pool.dtype), _layout_code(layout), int(num_layers),
                  int(layer_stride_bytes))


def pd_kv_append(k_new, v_new, k_pool, v_pool, new_indptr, kv_len, page_indptr, page_indices, *,
                 max_kv_len=None, dev_status=None, stream=None, layout="HND"):
    """Write new tokens' K/V rows ([total_new][Hkv][D]) into their page slots, in place."""
    lib = load_library()
    desc = _kv_desc(k_pool, layout=layout)
    batch = make_batch(kv_len, page_indptr, page_indices, k_pool.shape[0], qo_indptr=_i32(new_indptr, "new_indptr"),
                       total_qo=k_new.shape[0], max_kv_len=max_kv_len)
    rc = lib.pd_kv_append(ctypes.byref(desc), ctypes.byref(batch), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                          _ptr(v_pool), _ptr(dev_status), _stream(stream))
    _check(rc, "pd_kv_append")


def _layers(pools):
    if pools.dim() == 5:
        return pools.shape[0], pools[0].numel() * pools.element_size(), pools.shape[1]
    return 1, 0, pools.shape[0]


def pd_kv_pack(k_pools, v_pools, kv_len, page_indptr, page_indices, dst, dst_offsets, *, max_kv_len=None,
               dev_status=None, stream=None, layout="HND"):
    """Gather every request's KV of all layers into dst (uint8) at dst_offsets (int64 bytes)."""
    lib = load_library()
    L, stride, num_pages = _layers(k_pools)
    desc = _kv_desc(k_pools, L, stride, layout)
    batch = make_batch(kv_len, page_indptr, page_indices, num_pages, max_kv_len=max_kv_len)
    rc = lib.pd_kv_pack(ctypes.byref(desc), ctypes.byref(batch), _ptr(k_pools), _ptr(v_pools), _ptr(dst),
                        dst.numel() * dst.element_size(), _ptr(dst_offsets), _ptr(dev_status), _stream(stream))
    _check(rc, "pd_kv_pack")


def pd_kv_unpack(src, src_offsets, k_pools, v_pools, kv_len, page_indptr, page_indices, *, max_kv_len=None,
                 dev_status=None, stream=None, layout="HND"):
    """Scatter packed per-request KV blocks into [L][num_pages][Hkv][P][D] pools, in place."""
    lib = load_library()
    L, stride, num_pages = _layers(k_pools)
    desc = _kv_desc(k_pools, L, stride, layout)
    batch = make_batch(kv_len, page_indptr, page_indices, num_pages, max_kv_len=max_kv_len)
    rc = lib.pd_kv_unpack(ctypes.byref(desc), ctypes.byref(batch), _ptr(src), src.numel() * src.element_size(),
                          _ptr(src_offsets), _ptr(k_pools), _ptr(v_pools), _ptr(dev_status), _stream(stream))
    _check(rc, "pd_kv_unpack")


def pd_kv_pack_heads(k_pools, v_pools, kv_len, page_indptr, page_indices, dst, dst_offsets, head_begin, head_count,
                     *, max_kv_len=None, dev_status=None, stream=None, layout="HND"):
    """pd_kv_pack of pool heads [head_begin, head_begin + head_count) only; blocks hold head_count heads."""
    lib = load_library()
    L, stride, num_pages = _layers(k_pools)
    desc = _kv_desc(k_pools, L, stride, layout)
    batch = make_batch(kv_len, page_indptr, page_indices, num_pages, max_kv_len=max_kv_len)
    rc = lib.pd_kv_pack_heads(ctypes.byref(desc), ctypes.byref(batch), int(head_begin), int(head_count),
                              _ptr(k_pools), _ptr(v_pools), _ptr(dst), dst.numel() * dst.element_size(),
                              _ptr(dst_offsets), _ptr(dev_status), _stream(stream))
    _check(rc, "pd_kv_pack_heads")


def pd_kv_unpack_heads(src, src_offsets, k_pools, v_pools, kv_len, page_indptr, page_indices, head_begin, head_count,
                       *, max_kv_len=None, dev_status=None, stream=None, layout="HND"):
    """pd_kv_unpack of blocks holding head_count heads into pool heads [head_begin, head_begin + head_count)."""
    lib = load_library()
    L, stride, num_pages = _layers(k_pools)
    desc = _kv_desc(k_pools, L, stride, layout)
    batch = make_batch(kv_len, page_indptr, page_indices, num_pages, max_kv_len=max_kv_len)
    rc = lib.pd_kv_unpack_heads(ctypes.byref(desc), ctypes.byref(batch), int(head_begin), int(head_count),
                                _ptr(src), src.numel() * src.element_size(), _ptr(src_offsets), _ptr(k_pools),
                                _ptr(v_pools), _ptr(dev_status), _stream(stream))
    _check(rc, "pd_kv_unpack_heads")


def pd_kv_pack_layers(k_pools, v_pools, kv_len, page_indptr, page_indices, dst, dst_offsets, layer_begin,
                      layer_count, *, max_kv_len=None, dev_status=None, stream=None, layout="HND"):
    """pd_kv_pack of layers [layer_begin, layer_begin + layer_count) into their places of the full blocks."""
    lib = load_library()
    L, stride, num_pages = _layers(k_pools)
    desc = _kv_desc(k_pools, L, stride, layout)
    batch = make_batch(kv_len, page_indptr, page_indices, num_pages, max_kv_len=max_kv_len)
    rc = lib.pd_kv_pack_layers(ctypes.byref(desc), ctypes.byref(batch), int(layer_begin), int(layer_count),
                               _ptr(k_pools), _ptr(v_pools), _ptr(dst), dst.numel() * dst.element_size(),
                               _ptr(dst_offsets), _ptr(dev_status), _stream(stream))
    _check(rc, "pd_kv_pack_layers")


def pd_counter_alloc():
    """One mapped pinned 32-bit word set to 0: returns (host address, device address)."""
    h, d = ctypes.c_void_p(), ctypes.c_void_p()
    _check(load_library().pd_counter_alloc(ctypes.byref(h), ctypes.byref(d)), "pd_counter_alloc")
    return h.value, d.value


def pd_counter_free(host_word) -> None:
    _check(load_library().pd_counter_free(host_word), "pd_counter_free")


def counter_value(host_word) -> int:
    """Current value of a counter from pd_counter_alloc (read on the host)."""
    return ctypes.c_uint32.from_address(host_word).value


def pd_layer_signal(device_word, value: int, stream=None) -> None:
    """Enqueue the write of `value` to the counter once earlier work on the stream has completed."""
    _check(load_library().pd_layer_signal(device_word, int(value), _stream(stream)), "pd_layer_signal")


def pd_messenger_start_pack(host_word, k_pools, v_pools, kv_len, page_indptr, page_indices, dst, dst_offsets, *,
                            timeout_ms=1000, max_kv_len=None, dev_status=None, stream=None,
                            layout="HND"):
    """Start the host thread that packs each layer once the counter passes it; returns its handle."""
    lib = load_library()
    L, stride, num_pages = _layers(k_pools)
    desc = _kv_desc(k_pools, L, stride, layout)
    batch = make_batch(kv_len, page_indptr, page_indices, num_pages, max_kv_len=max_kv_len)
    handle = ctypes.c_void_p()
    rc = lib.pd_messenger_start_pack(ctypes.byref(handle), host_word, ctypes.byref(desc), ctypes.byref(batch),
                                     _ptr(k_pools), _ptr(v_pools), _ptr(dst), dst.numel() * dst.element_size(),
                                     _ptr(dst_offsets), _ptr(dev_status), _stream(stream), int(timeout_ms))
    _check(rc, "pd_messenger_start_pack")
    return handle.value


def pd_messenger_join(handle) -> int:
    """Wait for the messenger thread; returns the number of layers enqueued, raises PdError on failure."""
    sent = ctypes.c_int32(0)
    rc = load_library().pd_messenger_join(handle, ctypes.byref(sent))
    if rc != PD_OK:
        msg = load_library().pd_status_string(rc).decode()
        raise PdError(f"pd_messenger_join: {msg} ({rc}) after {sent.value} layers", rc)
    return sent.value


def pd_last_kernel() -> str:
    """Name of the main kernel the last call of this thread launched."""
    return load_library().pd_last_kernel().decode()


def pd_profile_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event `start` / `stop` around the main kernel of every
    following call of this thread (None, None to stop). The events must have
    been recorded once already so that their CUDA handles exist."""
    h = (lambda e: None if e is None else e.cuda_event)
    _check(load_library().pd_profile_events(h(start), h(stop)), "pd_profile_events")


def packed_bytes(kv_len_host, num_layers, num_kv_heads, head_dim, elem_size) -> int:
    """Bytes of the packed handoff buffer for the given per-request lengths."""
    return int(sum(int(n) for n in kv_len_host)) * 2 * num_layers * num_kv_heads * head_dim * elem_size
