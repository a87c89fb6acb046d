"""The C-ABI library loads and exports every entry point include/pkv.h
declares; host-side validation rejects bad arguments before any CUDA call.

No test here launches a kernel or passes a pointer that could be
dereferenced: every call below returns from the host-side checks.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_209_gb300 import build, pkv
    if not os.path.exists(pkv.LIB_PATH):
        build.build()
    return pkv.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"pkv_append", "pkv_copy_blocks", "pkv_decode_attention", "pkv_decode_workspace_size",
            "pkv_device_status", "pkv_status_string", "pkv_version"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    from paged_kv_cache_209_gb300 import pkv
    assert set(pkv.EXPORTS) == set(declared_functions())


def test_status_strings_and_version(lib):
    from paged_kv_cache_209_gb300 import pkv
    for code, name in enumerate(pkv.STATUS_NAMES):
        assert pkv.pkv_status_string(code) == name
    assert pkv.pkv_version() == 100


def _desc(**kw):
    from paged_kv_cache_209_gb300.pkv import CacheDesc
    d = dict(num_blocks=64, block_size=16, num_kv_heads=8, head_dim=128, dtype=1)
    d.update(kw)
    return CacheDesc(**d)


FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("desc_kw,status", [
    (dict(block_size=8), 2), (dict(head_dim=96), 2), (dict(num_kv_heads=0), 2), (dict(num_blocks=0), 2),
    (dict(dtype=7), 3), (dict(num_blocks=2 ** 40), 2),
])
def test_bad_geometry_is_rejected(lib, desc_kw, status):
    d = _desc(**desc_kw)
    assert lib.pkv_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), 0, None) == status
    assert lib.pkv_copy_blocks(FAKE, 1, FAKE, FAKE, ctypes.byref(d), 0, None) == status
    assert lib.pkv_decode_attention(FAKE, FAKE, FAKE, FAKE, 4, FAKE, 2, 32, ctypes.c_float(0.1), FAKE, FAKE,
                                    1 << 30, ctypes.byref(d), 0, None, None) == status


def test_null_and_alignment_are_rejected(lib):
    d = _desc()
    assert lib.pkv_append(FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, 0, None) == 1
    assert lib.pkv_append(None, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), 0, None) == 1
    assert lib.pkv_append(FAKE, FAKE, FAKE, 4, None, FAKE, ctypes.byref(d), 0, None) == 1
    assert lib.pkv_append(FAKE + 4, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), 0, None) == 4
    assert lib.pkv_append(FAKE, FAKE, FAKE + 4, 4, FAKE, FAKE, ctypes.byref(d), 0, None) == 4
    assert lib.pkv_append(FAKE, FAKE, FAKE, -1, FAKE, FAKE, ctypes.byref(d), 0, None) == 2
    assert lib.pkv_copy_blocks(None, 3, FAKE, FAKE, ctypes.byref(d), 0, None) == 1
    assert lib.pkv_copy_blocks(FAKE, -2, FAKE, FAKE, ctypes.byref(d), 0, None) == 2
    assert lib.pkv_copy_blocks(FAKE + 8, 1, FAKE + 8, FAKE, ctypes.byref(d), 0, None) == 4


def test_decode_argument_checks(lib):
    d = _desc()
    f = ctypes.c_float
    call = lambda **kw: lib.pkv_decode_attention(
        kw.get("q", FAKE), FAKE, FAKE, kw.get("tables", FAKE), kw.get("maxb", 4), FAKE, kw.get("batch", 2),
        kw.get("qh", 32), f(kw.get("scale", 0.1)), FAKE, kw.get("ws", FAKE), 1 << 30, ctypes.byref(d), 0, None,
        None)
    assert call(qh=30) == 2                      # not a multiple of the KV heads
    assert call(qh=1032) == 2                    # above PKV_MAX_Q_HEADS (1024)
    assert call(qh=0) == 2
    assert call(scale=float("inf")) == 2
    assert call(maxb=0) == 2
    assert call(maxb=1 << 27) == 2               # max_blocks * 16 reaches 2^31
    assert call(maxb=1 << 21, batch=1024) == 2   # the launch's blocks reach 2^31
    assert call(maxb=1 << 21, batch=0) == 0
    assert call(batch=-1) == 2
    assert call(q=None) == 1
    assert call(ws=None) == 1
    assert call(q=FAKE + 2) == 4
    assert call(ws=FAKE + 16) == 4               # workspace wants 256-byte alignment
    assert call(tables=FAKE + 2) == 4
    assert call(batch=0) == 0                    # empty batch: nothing to do


def test_zero_sized_moves_need_no_device(lib):
    d = _desc()
    assert lib.pkv_append(None, None, None, 0, FAKE, FAKE, ctypes.byref(d), 0, None) == 0
    assert lib.pkv_copy_blocks(None, 0, FAKE, FAKE, ctypes.byref(d), 0, None) == 0


def test_workspace_size_rejects_bad_geometry(lib):
    from paged_kv_cache_209_gb300.pkv import DecodeOpts
    assert lib.pkv_decode_workspace_size(2, 30, 4, ctypes.byref(_desc()), None) == 0
    assert lib.pkv_decode_workspace_size(2, 32, 4, None, None) == 0
    # the tensor-core kernel takes bf16 only
    assert lib.pkv_decode_workspace_size(2, 32, 4, ctypes.byref(_desc(dtype=0)),
                                         ctypes.byref(DecodeOpts(2, 0))) == 0


def test_multiquery_workspace_routing(lib):
    """Calls with more than 32 query rows per (sequence, KV head) take the
    tensor-core tile path, which combines on chip: a 256-byte workspace.
    Query counts above 65536 are rejected (size 0), as are float32 caches."""
    d = _desc()                                   # bf16, 8 KV heads
    assert lib.pkv_multiquery_workspace_size(4, 32, 16, 9, ctypes.byref(d), None) == 256    # 36 rows
    assert lib.pkv_multiquery_workspace_size(4, 32, 16, 65537, ctypes.byref(d), None) == 0
    assert lib.pkv_multiquery_workspace_size(4, 32, 16, 9, ctypes.byref(_desc(dtype=0)), None) == 0
    # more query heads than PKV_MAX_Q_HEADS: query-row counts would leave 32 bits
    assert lib.pkv_multiquery_workspace_size(4, 2048, 16, 65536, ctypes.byref(d), None) == 0
    assert lib.pkv_multiquery_workspace_size(4, 1024, 16, 65536, ctypes.byref(d), None) == 256   # both limits
    assert lib.pkv_decode_workspace_size(4, 2048, 16, ctypes.byref(d), None) == 0
    # rejected before anything is enqueued: more than 65536 queries, float32 caches
    args = [FAKE, FAKE, FAKE, FAKE, 16, FAKE, FAKE, 4, 32]
    tail = [ctypes.c_float(0.1), FAKE, FAKE, 256, ctypes.byref(d), 0, None, None]
    assert lib.pkv_multiquery_attention(*args, 65537, *tail) == 10          # PKV_ERR_UNSUPPORTED
    tail32 = [ctypes.c_float(0.1), FAKE, FAKE, 256, ctypes.byref(_desc(dtype=0)), 0, None, None]
    assert lib.pkv_multiquery_attention(*args, 9, *tail32) == 3             # PKV_ERR_DTYPE


def test_int8_entry_points_check_the_scale_pool(lib):
    """The int8 calls take one scale pool ([blocks][kv_heads][2][16] float):
    a null or misaligned pool is rejected before anything is enqueued."""
    d = _desc(dtype=2)                            # PKV_INT8, head_dim 128
    assert lib.pkv_append_q8(FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, ctypes.byref(d), 0, None) == 1
    assert lib.pkv_append_q8(FAKE, FAKE, FAKE, 4, FAKE, FAKE, FAKE + 4, ctypes.byref(d), 0, None) == 4
    assert lib.pkv_copy_blocks_q8(FAKE, 1, FAKE, FAKE, None, ctypes.byref(d), 0, None) == 1
    assert lib.pkv_copy_blocks_q8(FAKE, 1, FAKE, FAKE, FAKE + 8, ctypes.byref(d), 0, None) == 4
    assert lib.pkv_copy_blocks_q8(None, 0, FAKE, FAKE, FAKE, ctypes.byref(d), 0, None) == 0
    f = ctypes.c_float
    call = lambda sc: lib.pkv_decode_attention_q8(FAKE, FAKE, FAKE, sc, FAKE, 4, FAKE, None, 2, 32, 1, f(0.1),
                                                  FAKE, FAKE, 1 << 30, ctypes.byref(d), 0, None, None)
    assert call(None) == 1
    assert call(FAKE + 4) == 4
