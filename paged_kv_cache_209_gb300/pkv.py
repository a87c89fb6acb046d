"""Thin ctypes binding of libpkv.so (include/pkv.h), same function names.

Only argument marshalling happens here: tensors become device pointers, the
cache geometry becomes a ``pkv_cache_desc``, the current torch stream is
passed through, and a non-OK status raises ``PkvError``. Every step of the
decode path runs in the library's CUDA kernels. There is no fallback: if
``libpkv.so`` is missing or a tensor is not on a CUDA device, the call
raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_F32, PKV_BF16 = 0, 1
PKV_FLAG_CHECKED = 1
PKV_FLAG_TEST_STALL = 0x80000000
PKV_DEVERR_TIMEOUT, PKV_DEVERR_RANGE = 1, 2
STATUS_NAMES = ["PKV_OK", "PKV_ERR_NULL", "PKV_ERR_SHAPE", "PKV_ERR_DTYPE", "PKV_ERR_ALIGN", "PKV_ERR_RANGE",
                "PKV_ERR_OVERLAP", "PKV_ERR_WORKSPACE", "PKV_ERR_TIMEOUT", "PKV_ERR_CUDA", "PKV_ERR_UNSUPPORTED",
                "PKV_ERR_OUT_OF_BLOCKS", "PKV_ERR_UNKNOWN_SEQUENCE", "PKV_ERR_EXISTS", "PKV_ERR_INVARIANT"]


class PkvError(RuntimeError):
    """A libpkv call returned a status other than PKV_OK."""

    def __init__(self, fn: str, status: int):
        self.status = status
        self.name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else f"status {status}"
        super().__init__(f"{fn}: {self.name}")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class PoolStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "total_blocks", "free_blocks", "allocated_blocks", "physical_capacity_tokens", "physical_payload_tokens",
        "logical_tokens", "internal_waste_tokens", "sharing_savings_tokens", "sequences")]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("num_ctas", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("prefix_kernel", ctypes.c_int32)]


_lib = None

EXPORTS = ("pkv_append", "pkv_copy_blocks", "pkv_decode_workspace_size", "pkv_decode_attention",
           "pkv_decode_prefixed_workspace_size", "pkv_decode_attention_prefixed", "pkv_decode_attention_noalloc",
           "pkv_multiquery_workspace_size", "pkv_multiquery_attention",
           "pkv_append_q8", "pkv_copy_blocks_q8", "pkv_decode_q8_workspace_size", "pkv_decode_attention_q8", "pkv_device_status", "pkv_status_string", "pkv_version",
           "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_add_sequence", "pkv_pool_append", "pkv_pool_append_batch",
           "pkv_pool_share_prefix", "pkv_pool_release", "pkv_pool_sequence_length", "pkv_pool_page_table",
           "pkv_pool_block_tables", "pkv_pool_get_stats", "pkv_pool_validate")

# Size of the library's built-in workspace used by pkv_decode_attention_noalloc.
PKV_NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpkv.so once and declare the signatures of include/pkv.h."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with paged_kv_cache_209_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    desc_p, opts_p = ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeOpts)
    lib.pkv_append.argtypes = [vp, vp, vp, i64, vp, vp, desc_p, u32, vp]
    lib.pkv_append.restype = ctypes.c_int
    lib.pkv_copy_blocks.argtypes = [vp, i64, vp, vp, desc_p, u32, vp]
    lib.pkv_copy_blocks.restype = ctypes.c_int
    lib.pkv_decode_workspace_size.argtypes = [i32, i32, i32, desc_p, opts_p]
    lib.pkv_decode_workspace_size.restype = ctypes.c_size_t
    lib.pkv_decode_attention.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp,
                                         ctypes.c_size_t, desc_p, u32, opts_p, vp]
    lib.pkv_decode_attention.restype = ctypes.c_int
    lib.pkv_decode_prefixed_workspace_size.argtypes = [i32, i32, i32, i32, i32, desc_p, opts_p]
    lib.pkv_decode_prefixed_workspace_size.restype = ctypes.c_size_t
    lib.pkv_decode_attention_prefixed.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp, i32,
                                                  i32, vp, vp, ctypes.c_size_t, desc_p, u32, opts_p, vp]
    lib.pkv_decode_attention_prefixed.restype = ctypes.c_int
    lib.pkv_multiquery_workspace_size.argtypes = [i32, i32, i32, i32, desc_p, opts_p]
    lib.pkv_multiquery_workspace_size.restype = ctypes.c_size_t
    lib.pkv_multiquery_attention.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, ctypes.c_float, vp, vp,
                                             ctypes.c_size_t, desc_p, u32, opts_p, vp]
    lib.pkv_multiquery_attention.restype = ctypes.c_int
    lib.pkv_append_q8.argtypes = [vp, vp, vp, i64, vp, vp, vp, desc_p, u32, vp]
    lib.pkv_append_q8.restype = ctypes.c_int
    lib.pkv_copy_blocks_q8.argtypes = [vp, i64, vp, vp, vp, desc_p, u32, vp]
    lib.pkv_copy_blocks_q8.restype = ctypes.c_int
    lib.pkv_decode_q8_workspace_size.argtypes = [i32, i32, i32, i32, desc_p, opts_p]
    lib.pkv_decode_q8_workspace_size.restype = ctypes.c_size_t
    lib.pkv_decode_attention_q8.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, ctypes.c_float, vp,
                                            vp, ctypes.c_size_t, desc_p, u32, opts_p, vp]
    lib.pkv_decode_attention_q8.restype = ctypes.c_int
    lib.pkv_decode_attention_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp,
                                                 desc_p, u32, opts_p, vp]
    lib.pkv_decode_attention_noalloc.restype = ctypes.c_int
    lib.pkv_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, vp]
    lib.pkv_device_status.restype = ctypes.c_int
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = i32
    pp, i64p, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    lib.pkv_pool_create.argtypes = [i64, i32, vp, ctypes.POINTER(ctypes.c_void_p)]
    lib.pkv_pool_destroy.argtypes = [pp]
    lib.pkv_pool_destroy.restype = None
    lib.pkv_pool_add_sequence.argtypes = [pp, i64]
    lib.pkv_pool_append.argtypes = [pp, i64, i64, vp, vp, i32p]
    lib.pkv_pool_append_batch.argtypes = [pp, vp, vp, i64, vp, vp, i64p, i64p]
    lib.pkv_pool_share_prefix.argtypes = [pp, i64, i64, i64]
    lib.pkv_pool_release.argtypes = [pp, i64]
    lib.pkv_pool_sequence_length.argtypes = [pp, i64, i64p]
    lib.pkv_pool_page_table.argtypes = [pp, i64, vp, i64, i64p]
    lib.pkv_pool_block_tables.argtypes = [pp, vp, i64, vp, i64, vp]
    lib.pkv_pool_get_stats.argtypes = [pp, ctypes.POINTER(PoolStats)]
    lib.pkv_pool_validate.argtypes = [pp]
    for name in ("pkv_pool_create", "pkv_pool_add_sequence", "pkv_pool_append", "pkv_pool_append_batch",
                 "pkv_pool_share_prefix", "pkv_pool_release", "pkv_pool_sequence_length", "pkv_pool_page_table",
                 "pkv_pool_block_tables", "pkv_pool_get_stats", "pkv_pool_validate"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise PkvError(fn, status)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libpkv takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libpkv takes contiguous tensors only")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return PKV_F32
    if dt == torch.bfloat16:
        return PKV_BF16
    raise ValueError(f"unsupported dtype {dt}")


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    """Geometry of a pool tensor shaped [num_blocks][kv_heads][16][head_dim]."""
    if k_cache.dim() != 4:
        raise ValueError("a pool is [num_blocks][num_kv_heads][16][head_dim]")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d, _dtype_code(k_cache.dtype))


def _same_pools(k_cache, v_cache):
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("K and V pools must have one shape and dtype")


def pkv_append(k, v, slot_mapping, k_cache, v_cache, flags: int = 0, stream=None) -> None:
    """Write k[t], v[t] ([T][kv_heads][head_dim]) into slot slot_mapping[t] of the pools."""
    lib = load_library()
    _same_pools(k_cache, v_cache)
    desc = cache_desc(k_cache)
    T = int(slot_mapping.numel())
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping is int64")
    if T:
        want = (T, desc.num_kv_heads, desc.head_dim)
        if tuple(k.shape) != want or tuple(v.shape) != want or k.dtype != k_cache.dtype or v.dtype != k_cache.dtype:
            raise ValueError(f"k and v must be {want} of the pool dtype")
    _check("pkv_append", lib.pkv_append(_ptr(k) if T else None, _ptr(v) if T else None,
                                        _ptr(slot_mapping) if T else None, T, _ptr(k_cache), _ptr(v_cache),
                                        ctypes.byref(desc), flags, _stream(stream)))


def pkv_copy_blocks(src_dst_pairs, k_cache, v_cache, flags: int = 0, stream=None) -> None:
    """Copy block src onto block dst of both pools for every int64 (src, dst) row."""
    lib = load_library()
    _same_pools(k_cache, v_cache)
    desc = cache_desc(k_cache)
    n = int(src_dst_pairs.numel() // 2) if src_dst_pairs is not None else 0
    if n and (src_dst_pairs.dtype != torch.int64 or src_dst_pairs.shape[-1] != 2):
        raise ValueError("src_dst_pairs is int64 [n][2]")
    _check("pkv_copy_blocks", lib.pkv_copy_blocks(_ptr(src_dst_pairs) if n else None, n, _ptr(k_cache),
                                                  _ptr(v_cache), ctypes.byref(desc), flags, _stream(stream)))


def _opts(kernel: int, num_ctas: int, stages: int = 0, prefix_kernel: int = 0):
    if kernel == 0 and num_ctas == 0 and stages == 0 and prefix_kernel == 0:
        return None
    return ctypes.byref(DecodeOpts(kernel, num_ctas, stages, prefix_kernel))


def pkv_decode_workspace_size(batch: int, num_q_heads: int, max_blocks_per_seq: int, k_cache,
                              kernel: int = 0, num_ctas: int = 0, stages: int = 0) -> int:
    """Workspace bytes; allocate them zero-filled (``torch.zeros``) and reuse them."""
    lib = load_library()
    desc = cache_desc(k_cache)
    return int(lib.pkv_decode_workspace_size(batch, num_q_heads, max_blocks_per_seq, ctypes.byref(desc),
                                             _opts(kernel, num_ctas, stages)))


def pkv_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float, out=None,
                         workspace=None, flags: int = 0, kernel: int = 0, num_ctas: int = 0, stages: int = 0,
                         stream=None):
    """Decode attention; returns ``out`` ([batch][q_heads][head_dim], q's dtype)."""
    lib = load_library()
    _same_pools(k_cache, v_cache)
    desc = cache_desc(k_cache)
    batch, q_heads, d = q.shape
    if d != desc.head_dim or q.dtype != k_cache.dtype:
        raise ValueError("q must be [batch][q_heads][head_dim] of the pool dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens are int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != batch or context_lens.shape != (batch,):
        raise ValueError("block_tables is [batch][max_blocks], context_lens [batch]")
    max_blocks = int(block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    need = pkv_decode_workspace_size(batch, q_heads, max_blocks, k_cache, kernel, num_ctas, stages)
    if workspace is None:
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=q.device)
    _check("pkv_decode_attention", lib.pkv_decode_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(context_lens), batch,
        q_heads, ctypes.c_float(scale), _ptr(out), _ptr(workspace), workspace.numel(), ctypes.byref(desc), flags,
        _opts(kernel, num_ctas, stages), _stream(stream)))
    return out


def pkv_decode_prefixed_workspace_size(batch: int, num_q_heads: int, max_blocks_per_seq: int, num_groups: int,
                                       max_group_blocks: int, k_cache, kernel: int = 0, num_ctas: int = 0,
                                       stages: int = 0, prefix_kernel: int = 0) -> int:
    """Workspace bytes of the shared-prefix call; allocate them zero-filled and reuse them."""
    lib = load_library()
    desc = cache_desc(k_cache)
    return int(lib.pkv_decode_prefixed_workspace_size(batch, num_q_heads, max_blocks_per_seq, num_groups,
                                                      max_group_blocks, ctypes.byref(desc),
                                                      _opts(kernel, num_ctas, stages, prefix_kernel)))


def pkv_decode_attention_prefixed(q, k_cache, v_cache, block_tables, context_lens, scale: float, prefix_group,
                                  group_blocks, max_group_blocks: int, out=None, workspace=None, flags: int = 0,
                                  kernel: int = 0, num_ctas: int = 0, stages: int = 0, prefix_kernel: int = 0,
                                  stream=None):
    """Decode attention with shared-prefix groups (two phases); returns ``out``.

    ``prefix_group`` is int32 [batch] (group of each sequence or -1),
    ``group_blocks`` int32 [num_groups] (whole blocks each group shares),
    ``max_group_blocks`` a host-side bound on ``group_blocks``.
    """
    lib = load_library()
    _same_pools(k_cache, v_cache)
    desc = cache_desc(k_cache)
    batch, q_heads, d = q.shape
    if d != desc.head_dim or q.dtype != k_cache.dtype:
        raise ValueError("q must be [batch][q_heads][head_dim] of the pool dtype")
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens),
                    ("prefix_group", prefix_group), ("group_blocks", group_blocks)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} is int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != batch or context_lens.shape != (batch,):
        raise ValueError("block_tables is [batch][max_blocks], context_lens [batch]")
    if prefix_group.shape != (batch,) or group_blocks.dim() != 1:
        raise ValueError("prefix_group is [batch], group_blocks [num_groups]")
    max_blocks = int(block_tables.shape[1])
    num_groups = int(group_blocks.shape[0])
    if out is None:
        out = torch.empty_like(q)
    need = pkv_decode_prefixed_workspace_size(batch, q_heads, max_blocks, num_groups, max_group_blocks, k_cache,
                                              kernel, num_ctas, stages, prefix_kernel)
    if workspace is None:
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=q.device)
    _check("pkv_decode_attention_prefixed", lib.pkv_decode_attention_prefixed(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(context_lens), batch,
        q_heads, ctypes.c_float(scale), _ptr(prefix_group), _ptr(group_blocks), num_groups, max_group_blocks,
        _ptr(out), _ptr(workspace), workspace.numel(), ctypes.byref(desc), flags,
        _opts(kernel, num_ctas, stages, prefix_kernel), _stream(stream)))
    return out


def pkv_multiquery_workspace_size(batch: int, num_q_heads: int, max_blocks_per_seq: int, max_query_len: int,
                                  k_cache, num_ctas: int = 0) -> int:
    """Workspace bytes of the multi-query call; allocate them zero-filled and reuse them."""
    lib = load_library()
    desc = cache_desc(k_cache)
    return int(lib.pkv_multiquery_workspace_size(batch, num_q_heads, max_blocks_per_seq, max_query_len,
                                                 ctypes.byref(desc), _opts(0, num_ctas)))


def pkv_multiquery_attention(q, k_cache, v_cache, block_tables, context_lens, query_start, scale: float,
                             max_query_len: int, out=None, workspace=None, flags: int = 0, num_ctas: int = 0,
                             stream=None):
    """Causal multi-query attention; ``q``/``out`` are [query_start[-1]][q_heads][head_dim]
    and ``query_start`` int32 [batch + 1]. Returns ``out``.

    Up to 32 query rows per (sequence, KV head) (``max_query_len * q_heads / kv_heads``)
    run on the split decode kernel (``num_ctas`` applies there); more, a chunked
    prefill, on the tcgen05 tile kernel, which needs only 256 bytes of workspace."""
    lib = load_library()
    _same_pools(k_cache, v_cache)
    desc = cache_desc(k_cache)
    rows, q_heads, d = q.shape
    batch = int(context_lens.shape[0])
    if d != desc.head_dim or q.dtype != k_cache.dtype:
        raise ValueError("q must be [rows][q_heads][head_dim] of the pool dtype")
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens), ("query_start", query_start)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} is int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != batch or query_start.shape != (batch + 1,):
        raise ValueError("block_tables is [batch][max_blocks], query_start [batch + 1]")
    max_blocks = int(block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = pkv_multiquery_workspace_size(batch, q_heads, max_blocks, max_query_len, k_cache, num_ctas)
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=q.device)
    _check("pkv_multiquery_attention", lib.pkv_multiquery_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(context_lens),
        _ptr(query_start), batch, q_heads, max_query_len, ctypes.c_float(scale), _ptr(out), _ptr(workspace),
        workspace.numel(), ctypes.byref(desc), flags, _opts(0, num_ctas), _stream(stream)))
    return out


PKV_INT8 = 2


def q8_desc(k_codes: torch.Tensor) -> CacheDesc:
    """Geometry of int8 code pools: k_codes [num_blocks][kv_heads][16][head_dim]."""
    if k_codes.dim() != 4 or k_codes.dtype != torch.int8:
        raise ValueError("k_codes is int8 [num_blocks][num_kv_heads][16][head_dim]")
    nb, hkv, bs, d = k_codes.shape
    return CacheDesc(nb, bs, hkv, d, PKV_INT8)


def _check_q8_pools(k_codes, v_codes, scales):
    nb, hkv, bs, d = k_codes.shape
    if v_codes.shape != (nb, hkv, d, bs) or v_codes.dtype != torch.int8:
        raise ValueError("v_codes is int8 [num_blocks][num_kv_heads][head_dim][16]")
    if scales.shape != (nb, hkv, 2, bs) or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("scales are contiguous float32 [num_blocks][num_kv_heads][2][16] (K row, V row)")


def pkv_append_q8(k, v, slot_mapping, k_codes, v_codes, scales, flags: int = 0, stream=None) -> None:
    """Quantizing slot-mapped append of bf16 k/v [tokens][kv_heads][head_dim] into the int8 pools."""
    lib = load_library()
    _check_q8_pools(k_codes, v_codes, scales)
    desc = q8_desc(k_codes)
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16 or slot_mapping.dtype != torch.int64:
        raise ValueError("k/v are bf16, slot_mapping int64")
    _check("pkv_append_q8", lib.pkv_append_q8(
        _ptr(k), _ptr(v), _ptr(slot_mapping), int(slot_mapping.numel()), _ptr(k_codes), _ptr(v_codes),
        _ptr(scales), ctypes.byref(desc), flags, _stream(stream)))


def pkv_copy_blocks_q8(src_dst_pairs, k_codes, v_codes, scales, flags: int = 0, stream=None) -> None:
    lib = load_library()
    _check_q8_pools(k_codes, v_codes, scales)
    desc = q8_desc(k_codes)
    if src_dst_pairs.dtype != torch.int64:
        raise ValueError("pairs are int64 [n][2]")
    _check("pkv_copy_blocks_q8", lib.pkv_copy_blocks_q8(
        _ptr(src_dst_pairs) if src_dst_pairs.numel() else None, int(src_dst_pairs.shape[0]), _ptr(k_codes),
        _ptr(v_codes), _ptr(scales), ctypes.byref(desc), flags, _stream(stream)))


def pkv_decode_q8_workspace_size(batch: int, num_q_heads: int, max_blocks_per_seq: int, k_codes,
                                 max_query_len: int = 1, num_ctas: int = 0) -> int:
    lib = load_library()
    desc = q8_desc(k_codes)
    return int(lib.pkv_decode_q8_workspace_size(batch, num_q_heads, max_blocks_per_seq, max_query_len,
                                                ctypes.byref(desc), _opts(0, num_ctas)))


def pkv_decode_attention_q8(q, k_codes, v_codes, scales, block_tables, context_lens, scale: float,
                            query_start=None, max_query_len: int = 1, out=None, workspace=None, flags: int = 0,
                            num_ctas: int = 0, stream=None):
    """Attention over the int8 pools: decode (query_start None, q [batch][q_heads][head_dim]) or
    causal multi-query (q [query_start[-1]][q_heads][head_dim]). Returns ``out`` (bf16)."""
    lib = load_library()
    _check_q8_pools(k_codes, v_codes, scales)
    desc = q8_desc(k_codes)
    rows, q_heads, d = q.shape
    batch = int(context_lens.shape[0])
    if d != desc.head_dim or q.dtype != torch.bfloat16:
        raise ValueError("q is bf16 [rows][q_heads][head_dim]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens are int32")
    if query_start is not None and (query_start.dtype != torch.int32 or query_start.shape != (batch + 1,)):
        raise ValueError("query_start is int32 [batch + 1]")
    max_blocks = int(block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = pkv_decode_q8_workspace_size(batch, q_heads, max_blocks, k_codes, max_query_len, num_ctas)
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=q.device)
    _check("pkv_decode_attention_q8", lib.pkv_decode_attention_q8(
        _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(scales), _ptr(block_tables), max_blocks,
        _ptr(context_lens), _ptr(query_start), batch, q_heads, max_query_len, ctypes.c_float(scale), _ptr(out),
        _ptr(workspace), workspace.numel(), ctypes.byref(desc), flags, _opts(0, num_ctas), _stream(stream)))
    return out


def pkv_decode_attention_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale: float, out=None,
                                 flags: int = 0, kernel: int = 0, num_ctas: int = 0, stream=None):
    """Decode attention on the library's built-in workspace (no device allocation
    by the library; ``out`` is allocated here only when the caller passes none)."""
    lib = load_library()
    _same_pools(k_cache, v_cache)
    desc = cache_desc(k_cache)
    batch, q_heads, d = q.shape
    if d != desc.head_dim or q.dtype != k_cache.dtype:
        raise ValueError("q must be [batch][q_heads][head_dim] of the pool dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens are int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != batch or context_lens.shape != (batch,):
        raise ValueError("block_tables is [batch][max_blocks], context_lens [batch]")
    if out is None:
        out = torch.empty_like(q)
    _check("pkv_decode_attention_noalloc", lib.pkv_decode_attention_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
        batch, q_heads, ctypes.c_float(scale), _ptr(out), ctypes.byref(desc), flags, _opts(kernel, num_ctas),
        _stream(stream)))
    return out


def pkv_device_status(clear: bool = False, stream=None) -> int:
    """Sticky PKV_DEVERR_* bits of the current device (waits for the stream)."""
    lib = load_library()
    bits = ctypes.c_uint32(0)
    _check("pkv_device_status", lib.pkv_device_status(ctypes.byref(bits), int(clear), _stream(stream)))
    return int(bits.value)


def pkv_status_string(status: int) -> str:
    return load_library().pkv_status_string(status).decode()


def pkv_version() -> int:
    return int(load_library().pkv_version())


class BlockPool:
    """Host-side page table of the paged cache (the library's pkv_pool_*).

    Sequence ids are ints. Methods raise PkvError on a non-OK status; the
    pool is unchanged after a failed call (an append batch keeps the appends
    before the failing one, see ``append_batch``).
    """

    def __init__(self, total_blocks: int, block_size: int = 16, pop_order=None):
        import numpy as np
        self._lib = load_library()
        self._np = np
        handle = ctypes.c_void_p()
        order = None if pop_order is None else np.ascontiguousarray(pop_order, dtype=np.int64)
        _check("pkv_pool_create", self._lib.pkv_pool_create(
            int(total_blocks), int(block_size), None if order is None else order.ctypes.data, ctypes.byref(handle)))
        self._h = handle
        self.total_blocks = int(total_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pkv_pool_destroy(h)
            self._h = None

    def add_sequence(self, seq: int) -> None:
        _check("pkv_pool_add_sequence", self._lib.pkv_pool_add_sequence(self._h, int(seq)))

    def append(self, seq: int, tokens: int):
        """Returns (slot ids of the new tokens, copy pair (old, new) or None)."""
        np = self._np
        slots = np.empty(max(int(tokens), 0), dtype=np.int64)
        pair = np.empty(2, dtype=np.int64)
        n = ctypes.c_int32(0)
        _check("pkv_pool_append", self._lib.pkv_pool_append(
            self._h, int(seq), int(tokens), slots.ctypes.data if len(slots) else None, pair.ctypes.data,
            ctypes.byref(n)))
        return slots, (int(pair[0]), int(pair[1])) if n.value else None

    def append_batch(self, seqs, tokens):
        """One append per sequence, in order. Returns (slots, copy pairs [k][2])."""
        np = self._np
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        slots = np.empty(int(tokens.sum()), dtype=np.int64)
        pairs = np.empty((len(seqs), 2), dtype=np.int64)
        npairs, ndone = ctypes.c_int64(0), ctypes.c_int64(0)
        _check("pkv_pool_append_batch", self._lib.pkv_pool_append_batch(
            self._h, seqs.ctypes.data, tokens.ctypes.data, len(seqs), slots.ctypes.data if len(slots) else None,
            pairs.ctypes.data, ctypes.byref(npairs), ctypes.byref(ndone)))
        return slots, pairs[:npairs.value].copy()

    def share_prefix(self, source: int, target: int, prefix_tokens: int) -> None:
        _check("pkv_pool_share_prefix", self._lib.pkv_pool_share_prefix(self._h, int(source), int(target),
                                                                         int(prefix_tokens)))

    def release(self, seq: int) -> None:
        _check("pkv_pool_release", self._lib.pkv_pool_release(self._h, int(seq)))

    def sequence_length(self, seq: int) -> int:
        n = ctypes.c_int64(0)
        _check("pkv_pool_sequence_length", self._lib.pkv_pool_sequence_length(self._h, int(seq), ctypes.byref(n)))
        return n.value

    def page_table(self, seq: int):
        np = self._np
        n = ctypes.c_int64(0)
        st = self._lib.pkv_pool_page_table(self._h, int(seq), None, 0, ctypes.byref(n))
        if st not in (0, 2):
            _check("pkv_pool_page_table", st)
        out = np.empty(n.value, dtype=np.int32)
        _check("pkv_pool_page_table", self._lib.pkv_pool_page_table(
            self._h, int(seq), out.ctypes.data if n.value else None, n.value, ctypes.byref(n)))
        return tuple(int(b) for b in out)

    def block_tables(self, seqs, width: int):
        """(int32 tables [n][width] padded with -1, int32 lengths [n])."""
        np = self._np
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        tables = np.empty((len(seqs), int(width)), dtype=np.int32)
        lens = np.empty(len(seqs), dtype=np.int32)
        _check("pkv_pool_block_tables", self._lib.pkv_pool_block_tables(
            self._h, seqs.ctypes.data, len(seqs), tables.ctypes.data, int(width), lens.ctypes.data))
        return tables, lens

    def stats(self) -> dict:
        st = PoolStats()
        _check("pkv_pool_get_stats", self._lib.pkv_pool_get_stats(self._h, ctypes.byref(st)))
        return {name: getattr(st, name) for name, _ in PoolStats._fields_}

    def validate(self) -> None:
        _check("pkv_pool_validate", self._lib.pkv_pool_validate(self._h))
