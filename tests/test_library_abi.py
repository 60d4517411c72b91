"""CPU checks of the C ABI: the library builds, loads and exports every
symbol that include/pd.h declares; host-side argument checks reject bad input
without touching a GPU."""
import ctypes
import os
import re

import pytest

import decode_ragged_paged_gb300 as pd
from decode_ragged_paged_gb300 import build as pdbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pd_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    pdbuild.build()
    return pd.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(pd.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert lib.pd_version() >= 100
    for code in (0, -1, -2, -3, -4):
        assert lib.pd_status_string(code)
    for code in range(7):
        assert lib.pd_device_status_string(code) != b"unknown device status"


def _desc(**kw):
    d = dict(num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16, kv_dtype=pd.PD_BF16,
             o_dtype=pd.PD_BF16, layout=0, causal=1, sm_scale=0.0)
    d.update(kw)
    return pd.AttnDesc(**d)


def _batch(**kw):
    fake = 0x1000  # never dereferenced: every call below fails host checks first
    b = dict(batch_size=2, qo_indptr=fake, kv_len=fake, page_indptr=fake, page_indices=fake, num_pages=4,
             total_qo=2, max_qo_len=1, max_kv_len=32)
    b.update(kw)
    return pd.Batch(**b)


@pytest.mark.parametrize("kw,code", [
    (dict(num_kv_heads=3), pd.PD_ERR_INVALID_ARG),
    (dict(head_dim=96), pd.PD_ERR_UNSUPPORTED),
    (dict(page_size=0), pd.PD_ERR_INVALID_ARG),
    (dict(kv_dtype=7), pd.PD_ERR_INVALID_ARG),
    (dict(layout=2), pd.PD_ERR_INVALID_ARG),     # neither HND (0) nor NHD (1)
])
def test_decode_rejects_bad_descriptor(lib, kw, code):
    rc = lib.pd_attn_decode(ctypes.byref(_desc(**kw)), ctypes.byref(_batch()), 16, 16, 16, 16, None, 16, 1 << 30,
                            None, None)
    assert rc == code


def test_decode_rejects_bad_batch_and_pointers(lib):
    d = _desc()
    assert lib.pd_attn_decode(ctypes.byref(d), ctypes.byref(_batch(num_pages=0)), 16, 16, 16, 16, None, 16,
                              1 << 30, None, None) == pd.PD_ERR_INVALID_ARG
    assert lib.pd_attn_decode(ctypes.byref(d), ctypes.byref(_batch(kv_len=None)), 16, 16, 16, 16, None, 16,
                              1 << 30, None, None) == pd.PD_ERR_INVALID_ARG
    # misaligned q
    assert lib.pd_attn_decode(ctypes.byref(d), ctypes.byref(_batch()), 18, 16, 16, 16, None, 16, 1 << 30,
                              None, None) == pd.PD_ERR_INVALID_ARG
    # workspace too small
    assert lib.pd_attn_decode(ctypes.byref(d), ctypes.byref(_batch()), 16, 16, 16, 16, None, 16, 8,
                              None, None) == pd.PD_ERR_WORKSPACE
    # empty batch is a no-op
    assert lib.pd_attn_decode(ctypes.byref(d), ctypes.byref(_batch(batch_size=0)), None, None, None, None,
                              None, None, 0, None, None) == pd.PD_OK


def test_workspace_size_query(lib):
    n = lib.pd_attn_workspace_size(ctypes.byref(_desc()), ctypes.byref(_batch()), pd.PD_KIND_DECODE)
    assert n > 0 and n % 256 == 0
    assert lib.pd_attn_workspace_size(ctypes.byref(_desc(num_kv_heads=3)), ctypes.byref(_batch()), 0) == 0


def test_kv_copies_reject_bad_descriptor(lib):
    b = _batch()
    bad = [pd.KvDesc(0, 128, 16, pd.PD_BF16, 0, 1, 0),            # no heads
           pd.KvDesc(2, 4, 16, pd.PD_BF16, 0, 1, 0),              # 8-byte rows
           pd.KvDesc(2, 128, 16, pd.PD_BF16, 0, 2, 8),            # unaligned layer stride
           pd.KvDesc(2, 128, 16, pd.PD_BF16, 2, 1, 0)]            # unknown layout
    for d in bad:
        assert lib.pd_kv_pack(ctypes.byref(d), ctypes.byref(b), 16, 16, 16, 1 << 20, 16, None, None) < 0
        assert lib.pd_kv_unpack(ctypes.byref(d), ctypes.byref(b), 16, 1 << 20, 16, 16, 16, None, None) < 0
    two_layers = pd.KvDesc(2, 128, 16, pd.PD_BF16, 0, 2, 1 << 20)
    assert lib.pd_kv_append(ctypes.byref(two_layers), ctypes.byref(b), 16, 16, 16, 16, None, None) == \
        pd.PD_ERR_INVALID_ARG


def test_head_ranges_outside_the_pool_are_rejected(lib):
    b = _batch()
    d = pd.KvDesc(4, 128, 16, pd.PD_BF16, 0, 1, 0)
    for h0, n in [(-1, 2), (0, 0), (3, 2), (4, 1)]:
        assert lib.pd_kv_pack_heads(ctypes.byref(d), ctypes.byref(b), h0, n, 16, 16, 16, 1 << 20, 16, None,
                                    None) == pd.PD_ERR_INVALID_ARG
        assert lib.pd_kv_unpack_heads(ctypes.byref(d), ctypes.byref(b), h0, n, 16, 1 << 20, 16, 16, 16, None,
                                      None) == pd.PD_ERR_INVALID_ARG


def _start(lib, word, batch, timeout_ms):
    d = pd.KvDesc(2, 128, 16, pd.PD_BF16, 0, 3, 1 << 20)
    h = ctypes.c_void_p()
    rc = lib.pd_messenger_start_pack(ctypes.byref(h), ctypes.addressof(word), ctypes.byref(d), ctypes.byref(batch),
                                     0x1000, 0x1000, 0x1000, 1 << 20, 0x1000, None, None, timeout_ms)
    return rc, h


def test_messenger_times_out_when_no_layer_is_signalled(lib):
    # host-side failure detection: the counter never advances, the thread gives
    # up after its timeout and reports it; nothing is launched
    import time
    word = ctypes.c_uint32(0)
    rc, h = _start(lib, word, _batch(), 50)
    assert rc == pd.PD_OK
    t0 = time.monotonic()
    sent = ctypes.c_int32(-1)
    assert lib.pd_messenger_join(h, ctypes.byref(sent)) == pd.PD_ERR_TIMEOUT
    assert sent.value == 0 and time.monotonic() - t0 < 5.0


def test_messenger_reports_a_failed_layer_pack(lib):
    # the counter says layer 0 is ready; its pack fails host validation
    # (no pages), so the thread stops with that error before any launch
    word = ctypes.c_uint32(1)
    rc, h = _start(lib, word, _batch(num_pages=0), 1000)
    assert rc == pd.PD_OK
    sent = ctypes.c_int32(-1)
    assert lib.pd_messenger_join(h, ctypes.byref(sent)) == pd.PD_ERR_INVALID_ARG
    assert sent.value == 0


def test_messenger_rejects_bad_arguments(lib):
    word = ctypes.c_uint32(0)
    assert _start(lib, word, _batch(), 0)[0] == pd.PD_ERR_INVALID_ARG
    d = pd.KvDesc(2, 128, 16, pd.PD_BF16, 0, 3, 1 << 20)
    h = ctypes.c_void_p()
    assert lib.pd_messenger_start_pack(ctypes.byref(h), None, ctypes.byref(d), ctypes.byref(_batch()), 0x1000, 0x1000,
                                       0x1000, 1 << 20, 0x1000, None, None, 100) == pd.PD_ERR_INVALID_ARG
    assert lib.pd_messenger_join(None, None) == pd.PD_ERR_INVALID_ARG
    assert lib.pd_layer_signal(None, 1, None) == pd.PD_ERR_INVALID_ARG


def test_layer_range_outside_the_pool_is_rejected(lib):
    b = _batch()
    d = pd.KvDesc(2, 128, 16, pd.PD_BF16, 0, 3, 1 << 20)
    for l0, n in [(-1, 1), (0, 0), (2, 2), (3, 1)]:
        assert lib.pd_kv_pack_layers(ctypes.byref(d), ctypes.byref(b), l0, n, 16, 16, 16, 1 << 20, 16, None,
                                     None) == pd.PD_ERR_INVALID_ARG


def _mla_desc(**kw):
    d = dict(num_qo_heads=128, kv_lora_rank=512, rope_dim=64, page_size=64, kv_dtype=pd.PD_BF16,
             o_dtype=pd.PD_BF16, sm_scale=0.0)
    d.update(kw)
    return pd.MlaDesc(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(num_qo_heads=0), pd.PD_ERR_INVALID_ARG),
    (dict(num_qo_heads=129), pd.PD_ERR_UNSUPPORTED),     # more heads than one 128-row tile
    (dict(kv_lora_rank=256), pd.PD_ERR_UNSUPPORTED),
    (dict(rope_dim=32), pd.PD_ERR_UNSUPPORTED),
    (dict(kv_dtype=pd.PD_F32), pd.PD_ERR_UNSUPPORTED),
    (dict(page_size=8), pd.PD_ERR_UNSUPPORTED),
    (dict(page_size=48), pd.PD_ERR_UNSUPPORTED),
    (dict(page_size=512), pd.PD_ERR_UNSUPPORTED),        # above the largest supported page
    (dict(o_dtype=9), pd.PD_ERR_INVALID_ARG),
])
def test_mla_rejects_bad_descriptor(lib, kw, code):
    rc = lib.pd_mla_decode(ctypes.byref(_mla_desc(**kw)), ctypes.byref(_batch()), 16, 16, 16, 16, 16, 1 << 30,
                           None, None)
    assert rc == code
    assert lib.pd_mla_workspace_size(ctypes.byref(_mla_desc(**kw)), ctypes.byref(_batch())) == 0


def test_mla_workspace_and_pointer_checks(lib):
    d, b = _mla_desc(), _batch()
    n = lib.pd_mla_workspace_size(ctypes.byref(d), ctypes.byref(b))
    assert n > 0 and n % 256 == 0
    # partial outputs for batch + one chunk per SM at most: grows with the batch
    assert lib.pd_mla_workspace_size(ctypes.byref(d), ctypes.byref(_batch(batch_size=20))) > n
    assert lib.pd_mla_decode(ctypes.byref(d), ctypes.byref(b), 16, 16, 16, 16, 16, n - 1, None,
                             None) == pd.PD_ERR_WORKSPACE
    assert lib.pd_mla_decode(ctypes.byref(d), ctypes.byref(b), 24, 16, 16, 16, 16, n, None,
                             None) == pd.PD_ERR_INVALID_ARG                                   # misaligned q
    assert lib.pd_mla_decode(ctypes.byref(d), ctypes.byref(_batch(kv_len=None)), 16, 16, 16, 16, 16, n, None,
                             None) == pd.PD_ERR_INVALID_ARG
    assert lib.pd_mla_decode(ctypes.byref(d), ctypes.byref(_batch(batch_size=0)), None, None, None, None, None, 0,
                             None, None) == pd.PD_OK


def _split(lib, d, b, num_prefill, prefill_sms=0, ws_bytes=1 << 30):
    return lib.pd_attn_mixed_split(ctypes.byref(d), ctypes.byref(b), num_prefill, prefill_sms, 16, 16, 16, 16,
                                   None, 16, ws_bytes, None, None)


def test_mixed_split_rejects_bad_arguments(lib):
    d = _desc()
    b = _batch(batch_size=3, total_qo=130, max_qo_len=128, max_kv_len=512)
    assert _split(lib, d, b, 4) == pd.PD_ERR_INVALID_ARG          # more prefill requests than requests
    assert _split(lib, d, b, -1) == pd.PD_ERR_INVALID_ARG
    assert _split(lib, d, b, 1, prefill_sms=-8) == pd.PD_ERR_INVALID_ARG
    assert _split(lib, d, _batch(batch_size=3, qo_indptr=None, total_qo=130, max_qo_len=128, max_kv_len=512),
                  1) == pd.PD_ERR_INVALID_ARG                    # the split needs qo_indptr
    assert _split(lib, d, _batch(batch_size=3, total_qo=1, max_qo_len=1, max_kv_len=512),
                  0) == pd.PD_ERR_INVALID_ARG                    # fewer rows than decode requests
    assert _split(lib, _desc(num_kv_heads=3), b, 1) == pd.PD_ERR_INVALID_ARG
    assert _split(lib, d, b, 1, ws_bytes=64) == pd.PD_ERR_WORKSPACE


def test_mixed_split_workspace_covers_both_parts(lib):
    d = _desc()
    b = _batch(batch_size=64, total_qo=1087, max_qo_len=1024, max_kv_len=1024)
    sizes = [lib.pd_attn_workspace_size(ctypes.byref(d), ctypes.byref(b), k) for k in range(4)]
    assert all(s > 0 for s in sizes)
    assert sizes[pd.PD_KIND_MIXED_SPLIT] >= sizes[pd.PD_KIND_PREFILL] + sizes[pd.PD_KIND_DECODE]
