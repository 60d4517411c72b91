"""fp64 CPU oracle for ragged paged attention and the KV append / pack / unpack.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline may use this package; the library never does. It shares no code with
the CUDA path. The arithmetic lives in ``pd_oracle.c`` (plain loops in fp64);
this module compiles it with gcc on first use and marshals numpy arrays.

Pins (see ``tests/test_oracle_pins.py``): numpy brute-force dense attention on
tiny inputs, torch's fp64 ``scaled_dot_product_attention`` on gathered dense
tensors, closed forms (one key, identical keys, constant values, a two-key
example worked by hand), page-permutation invariance, prefill = successive
decodes, the log-sum-exp merge of two key halves, pack/unpack identities and
hand-written golden buffers. Each planted mistake (``-DORACLE_MUTANT=n``) fails
at least one of them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pd_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

F32, BF16 = 0, 1
HND, NHD = "HND", "NHD"
_LAYOUT = {HND: 0, NHD: 1}


def lib_path(mutant: int = 0) -> str:
    name = "libpd_oracle.so" if mutant == 0 else f"libpd_oracle_m{mutant}.so"
    return os.path.join(_HERE, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (gcc, fp64, OpenMP). Returns the shared-object path."""
    out = lib_path(mutant)
    import platform
    stamp = out + ".host"
    same_host = os.path.exists(stamp) and open(stamp).read() == platform.machine()
    if not force and same_host and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    with open(stamp, "w") as f:
        f.write(platform.machine())
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant not in _LIBS:
            lib = ctypes.CDLL(build(mutant))
            P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_attention.argtypes = [I32, P, P, P, P, I32, I32, I32, I32, I32, D, I32, I32,
                                             P, P, P, P, P, I32]
            lib.oracle_attention_rows.argtypes = [I32, P, P, P, P, I32, I32, I32, I32, I32, D, I32, I32,
                                                  P, P, P, I64, P, P, P, P, I32]
            lib.oracle_kv_append.argtypes = [I32, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P, P, P]
            lib.oracle_kv_pack.argtypes = [I32, P, P, P, I32, I32, I64, I32, I32, I32, I32, I32, I32, I32,
                                           P, P, P, P]
            lib.oracle_kv_unpack.argtypes = [I32, P, P, P, I32, I32, I64, I32, I32, I32, I32, I32, I32, I32,
                                             P, P, P, P]
            lib.oracle_mla_decode.argtypes = [I32, P, P, P, I32, I32, I32, I32, I32, D, P, P, I64, P, P, P, P,
                                              I32]
            lib.oracle_num_threads.argtypes = [I32]
            for f in ("oracle_attention", "oracle_attention_rows", "oracle_kv_append",
                      "oracle_kv_pack", "oracle_kv_unpack", "oracle_mla_decode", "oracle_num_threads",
                      "oracle_mutant"):
                getattr(lib, f).restype = ctypes.c_int
            _LIBS[mutant] = lib
        return _LIBS[mutant]


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float32:
        return F32
    raise TypeError(f"oracle takes fp32 arrays or bf16 bit patterns (uint16), got {arr.dtype}")


def num_threads(nthreads: int = 0) -> int:
    return _load().oracle_num_threads(nthreads)


def _pool_dims(pool: np.ndarray, layout: str):
    """(num_pages, Hkv, P, D) of one pool: [pages][Hkv][P][D] (HND) or [pages][P][Hkv][D] (NHD)."""
    if layout not in _LAYOUT:
        raise ValueError(f"unknown layout {layout!r}")
    n, a, b, d = pool.shape[-4:]
    return (n, a, b, d) if layout == HND else (n, b, a, d)


def attention(qo_indptr, kv_len, page_indptr, page_indices, q, k_pool, v_pool,
              num_qo_heads, num_kv_heads, scale, causal=True, nthreads=0, mutant=0, layout=HND):
    """All rows. q [total_qo][Hq][D]; pools [num_pages][Hkv][P][D] (HND) or
    [num_pages][P][Hkv][D] (NHD).
    Returns (o fp64 [total_qo][Hq][D], lse fp64 [total_qo][Hq])."""
    qo_indptr, kv_len = _i32(qo_indptr), _i32(kv_len)
    page_indptr, page_indices = _i32(page_indptr), _i32(page_indices)
    q, k_pool, v_pool = (np.ascontiguousarray(x) for x in (q, k_pool, v_pool))
    dt = _dtype_code(q)
    assert _dtype_code(k_pool) == dt and _dtype_code(v_pool) == dt
    total_qo, hq, d = q.shape
    _, hkv, p, _ = _pool_dims(k_pool, layout)
    assert hkv == num_kv_heads
    o = np.zeros((total_qo, hq, d), dtype=np.float64)
    lse = np.zeros((total_qo, hq), dtype=np.float64)
    rc = _load(mutant).oracle_attention(len(kv_len), _ptr(qo_indptr), _ptr(kv_len), _ptr(page_indptr),
                                        _ptr(page_indices), hq, num_kv_heads, d, p, dt, float(scale),
                                        int(bool(causal)), _LAYOUT[layout], _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                        _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attention rejected its inputs (rc={rc})")
    return o, lse


def attention_rows(qo_indptr, kv_len, page_indptr, page_indices, q, k_pool, v_pool,
                   num_qo_heads, num_kv_heads, scale, sel_row, sel_head, causal=True,
                   nthreads=0, mutant=0, layout=HND):
    """Selected (global q row, q head) pairs only. Returns (o [n][D], lse [n])."""
    qo_indptr, kv_len = _i32(qo_indptr), _i32(kv_len)
    page_indptr, page_indices = _i32(page_indptr), _i32(page_indices)
    q, k_pool, v_pool = (np.ascontiguousarray(x) for x in (q, k_pool, v_pool))
    sel_row, sel_head = _i32(sel_row), _i32(sel_head)
    dt = _dtype_code(q)
    total_qo, hq, d = q.shape
    _, hkv, p, _ = _pool_dims(k_pool, layout)
    assert hkv == num_kv_heads
    n = len(sel_row)
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = _load(mutant).oracle_attention_rows(len(kv_len), _ptr(qo_indptr), _ptr(kv_len),
                                             _ptr(page_indptr), _ptr(page_indices), hq, num_kv_heads,
                                             d, p, dt, float(scale), int(bool(causal)), _LAYOUT[layout], _ptr(q),
                                             _ptr(k_pool), _ptr(v_pool), n, _ptr(sel_row),
                                             _ptr(sel_head), _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attention_rows rejected its inputs (rc={rc})")
    return o, lse


def kv_append(new_indptr, kv_len, page_indptr, page_indices, k_new, v_new, k_pool, v_pool,
              mutant=0, layout=HND):
    """In-place append of k_new / v_new ([total_new][Hkv][D]) into the pools (HND or NHD)."""
    new_indptr, kv_len = _i32(new_indptr), _i32(kv_len)
    page_indptr, page_indices = _i32(page_indptr), _i32(page_indices)
    k_new, v_new = np.ascontiguousarray(k_new), np.ascontiguousarray(v_new)
    assert k_pool.flags["C_CONTIGUOUS"] and v_pool.flags["C_CONTIGUOUS"]
    num_pages, hkv, p, d = _pool_dims(k_pool, layout)
    rc = _load(mutant).oracle_kv_append(len(kv_len), _ptr(new_indptr), _ptr(kv_len), _ptr(page_indptr),
                                        _ptr(page_indices), num_pages, hkv, d, p, k_pool.itemsize,
                                        _LAYOUT[layout],
                                        _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool))
    if rc != 0:
        raise ValueError("oracle_kv_append rejected its inputs")


def kv_pack(kv_len, page_indptr, page_indices, k_pools, v_pools, dst_offsets, dst_bytes, mutant=0,
            head_begin=0, head_count=None, layout=HND):
    """k_pools / v_pools: [L][num_pages][Hkv][P][D] (HND) or [L][num_pages][P][Hkv][D] (NHD).
    Returns the packed uint8 buffer holding heads [head_begin, head_begin + head_count) (all heads
    by default)."""
    kv_len = _i32(kv_len)
    page_indptr, page_indices = _i32(page_indptr), _i32(page_indices)
    k_pools, v_pools = np.ascontiguousarray(k_pools), np.ascontiguousarray(v_pools)
    dst_offsets = np.ascontiguousarray(dst_offsets, dtype=np.int64)
    L = k_pools.shape[0]
    num_pages, hkv, p, d = _pool_dims(k_pools, layout)
    stride = k_pools[0].nbytes
    head_count = hkv - head_begin if head_count is None else head_count
    dst = np.zeros(int(dst_bytes), dtype=np.uint8)
    rc = _load(mutant).oracle_kv_pack(len(kv_len), _ptr(kv_len), _ptr(page_indptr), _ptr(page_indices),
                                      num_pages, L, stride, hkv, head_begin, head_count, d, p, k_pools.itemsize,
                                      _LAYOUT[layout], _ptr(k_pools), _ptr(v_pools), _ptr(dst), _ptr(dst_offsets))
    if rc != 0:
        raise ValueError("oracle_kv_pack rejected its inputs")
    return dst


def kv_unpack(kv_len, page_indptr, page_indices, src, src_offsets, k_pools, v_pools, mutant=0,
              head_begin=0, head_count=None, layout=HND):
    """In-place unpack of the packed uint8 buffer ``src`` (holding head_count heads) into heads
    [head_begin, head_begin + head_count) of [L][num_pages][Hkv][P][D] pools, or
    [L][num_pages][P][Hkv][D] for NHD (all heads by default)."""
    kv_len = _i32(kv_len)
    page_indptr, page_indices = _i32(page_indptr), _i32(page_indices)
    src = np.ascontiguousarray(src)
    src_offsets = np.ascontiguousarray(src_offsets, dtype=np.int64)
    assert k_pools.flags["C_CONTIGUOUS"] and v_pools.flags["C_CONTIGUOUS"]
    L = k_pools.shape[0]
    num_pages, hkv, p, d = _pool_dims(k_pools, layout)
    stride = k_pools[0].nbytes
    head_count = hkv - head_begin if head_count is None else head_count
    rc = _load(mutant).oracle_kv_unpack(len(kv_len), _ptr(kv_len), _ptr(page_indptr), _ptr(page_indices),
                                        num_pages, L, stride, hkv, head_begin, head_count, d, p, k_pools.itemsize,
                                        _LAYOUT[layout], _ptr(src), _ptr(src_offsets), _ptr(k_pools),
                                        _ptr(v_pools))
    if rc != 0:
        raise ValueError("oracle_kv_unpack rejected its inputs")


def mla_decode(kv_len, page_indptr, page_indices, q, kv_pool, d_c, scale, sel_req=None, sel_head=None,
               nthreads=0, mutant=0):
    """MLA decode over a paged latent cache. q [B][Hq][d_c + d_r]; kv_pool
    [num_pages][P][d_c + d_r]; scores over the whole row, values its first d_c
    entries. All pairs: returns (o fp64 [B][Hq][d_c], lse fp64 [B][Hq]); with
    sel_req / sel_head: (o [n][d_c], lse [n]) for those (request, head) pairs."""
    kv_len = _i32(kv_len)
    page_indptr, page_indices = _i32(page_indptr), _i32(page_indices)
    q, kv_pool = np.ascontiguousarray(q), np.ascontiguousarray(kv_pool)
    dt = _dtype_code(q)
    assert _dtype_code(kv_pool) == dt
    B, hq, w = q.shape
    _, p, w2 = kv_pool.shape
    assert w2 == w and 0 < d_c <= w
    if sel_req is None:
        n, sr, sh = 0, None, None
        o = np.zeros((B, hq, d_c), dtype=np.float64)
        lse = np.zeros((B, hq), dtype=np.float64)
    else:
        sr, sh = _i32(sel_req), _i32(sel_head)
        n = len(sr)
        o = np.zeros((n, d_c), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
    rc = _load(mutant).oracle_mla_decode(B, _ptr(kv_len), _ptr(page_indptr), _ptr(page_indices), hq, d_c,
                                         w - d_c, p, dt, float(scale), _ptr(q), _ptr(kv_pool), n,
                                         None if sr is None else _ptr(sr), None if sh is None else _ptr(sh),
                                         _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_mla_decode rejected its inputs (rc={rc})")
    return o, lse


def attention_case(case, nthreads=0, mutant=0):
    """Oracle over a ``workloads.AttnCase``."""
    return attention(case.qo_indptr, case.kv_len, case.table.page_indptr, case.table.page_indices,
                     case.q, case.k_pool, case.v_pool, case.num_qo_heads, case.num_kv_heads,
                     case.scale, causal=case.causal, nthreads=nthreads, mutant=mutant,
                     layout=getattr(case, "layout", HND))
