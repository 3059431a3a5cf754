"""Python binding of ``libpaged_kv.so`` (the C ABI in ``include/paged_kv.h``).

Argument marshalling only: each function takes torch CUDA tensors, passes
their device pointers, element strides and the current CUDA stream to the C
entry point of the same name, and raises ``RuntimeError`` on a non-OK status.
Every step of the decode path runs in the library's CUDA kernels; there is no
fallback.  The library is loaded on first use and a missing build raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "PKV_ERRF_BLOCK_ID",
    "PKV_ERRF_SEQ_LEN",
    "PKV_ERRF_SPLITS",
    "PKV_ERRF_INDPTR",
    "PKV_ERRF_TIMEOUT",
    "PKV_ERRF_ORDER",
    "lib",
    "lib_path",
    "version",
    "set_attention_warps",
    "set_wait_limit_ns",
    "set_fp8_kernel",
    "paged_attention_decode",
    "paged_attention_v2_partition",
    "paged_attention_v2_reduce",
    "copy_page_indices",
    "compute_num_kv_splits",
    "prepare_decode_metadata",
    "normal_decode_set_metadata",
    "prepare_swa_spec_page_table",
    "paged_attention_v2_noalloc",
    "noalloc_scratch_bytes",
    "order_by_length",
]

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libpaged_kv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA = 0, 1, 2, 3
PKV_ERR_SCRATCH_TOO_SMALL = 4
PKV_ERRF_BLOCK_ID, PKV_ERRF_SEQ_LEN, PKV_ERRF_SPLITS, PKV_ERRF_INDPTR, PKV_ERRF_TIMEOUT = (
    1, 2, 4, 8, 16)
PKV_ERRF_ORDER = 32

_DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

# kv_cache_dtype names (vLLM's) -> pkv_kv_cache_dtype_t
_KV_CACHE_CODE = {"auto": 0, "fp8": 1, "fp8_e4m3": 1, "fp8_e5m2": 2}
_FP8_TORCH = {getattr(torch, n): c for n, c in (("float8_e4m3fn", 1), ("float8_e5m2", 2))
              if hasattr(torch, n)}

_c_i32, _c_i64, _c_f32, _c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
_I64x3 = _c_i64 * 3


class DecodeArgs(ctypes.Structure):
    """Mirror of ``pkv_decode_args_t``."""

    _fields_ = [
        ("num_seqs", _c_i32), ("num_heads", _c_i32), ("num_kv_heads", _c_i32),
        ("head_size", _c_i32), ("block_size", _c_i32), ("x", _c_i32),
        ("max_blocks_per_seq", _c_i32), ("num_blocks", _c_i32),
        ("dtype", ctypes.c_int), ("scale", _c_f32),
        ("query", _c_p), ("q_stride", _c_i64 * 3),
        ("key_cache", _c_p), ("k_stride", _c_i64 * 5),
        ("value_cache", _c_p), ("v_stride", _c_i64 * 4),
        ("block_tables", _c_p), ("bt_stride", _c_i64 * 2),
        ("kv_indptr", _c_p), ("seq_lens", _c_p), ("err_flag", _c_p),
        ("kv_cache_dtype", _c_i32), ("k_scale", _c_f32), ("v_scale", _c_f32),
        ("alibi_slopes", _c_p), ("seq_order", _c_p),
    ]


class DecodeMetadataArgs(ctypes.Structure):
    """Mirror of ``pkv_decode_metadata_args_t``."""

    _fields_ = [
        ("batch_size", _c_i32), ("max_seq_pages", _c_i32), ("seq_len_delta", _c_i32),
        ("page_size", _c_i32),
        ("seq_lens", _c_p), ("seq_lens_stride", _c_i64),
        ("req_to_token", _c_p), ("req_to_token_stride", _c_i64 * 2),
        ("req_to_token_rows", _c_i64), ("req_to_token_cols", _c_i64),
        ("req_pool_indices", _c_p), ("req_pool_indices_stride", _c_i64),
        ("cache_seqlens", _c_p), ("cache_seqlens_stride", _c_i64),
        ("cu_seqlens_k", _c_p), ("cu_seqlens_k_stride", _c_i64),
        ("page_table", _c_p), ("page_table_stride", _c_i64 * 2),
        ("swa_page_table", _c_p), ("swa_page_table_stride", _c_i64 * 2),
        ("full_to_swa_mapping", _c_p), ("full_to_swa_stride", _c_i64),
        ("full_to_swa_len", _c_i64),
        ("err_flag", _c_p),
        ("cu_num_pages", _c_p), ("cu_num_pages_stride", _c_i64),
    ]


class SwaSpecArgs(ctypes.Structure):
    """Mirror of ``pkv_swa_spec_args_t``."""

    _fields_ = [
        ("bs", _c_i32), ("num_draft_tokens", _c_i32), ("len_a", _c_i32), ("len_b", _c_i32),
        ("page_table_a", _c_p), ("a_stride", _c_i64 * 2),
        ("page_table_b", _c_p), ("b_stride", _c_i64 * 2),
        ("seq_len_a", _c_p), ("seq_len_a_stride", _c_i64),
        ("seq_len_b", _c_p), ("seq_len_b_stride", _c_i64),
        ("dst", _c_p), ("dst_stride", _c_i64 * 2),
        ("err_flag", _c_p),
    ]


_LIB = None


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with `python -m paged_kv_decode_tables_gb300._build` "
            "(or __graft_entry__.build()); there is no fallback implementation")
    L = ctypes.CDLL(_LIB_PATH)
    L.pkv_version.restype = ctypes.c_char_p
    L.pkv_version.argtypes = []
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_decode_args_size.restype = ctypes.c_size_t
    L.pkv_decode_args_size.argtypes = []
    L.pkv_set_attention_warps.restype = ctypes.c_int
    L.pkv_set_attention_warps.argtypes = [_c_i32]
    L.pkv_set_fp8_kernel.restype = ctypes.c_int
    L.pkv_set_fp8_kernel.argtypes = [_c_i32]
    L.pkv_set_split_fold.restype = ctypes.c_int
    L.pkv_set_split_fold.argtypes = [_c_i32]
    L.pkv_set_wait_limit_ns.restype = ctypes.c_int
    L.pkv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.pkv_test_set_unarrived_bytes.restype = ctypes.c_int
    L.pkv_test_set_unarrived_bytes.argtypes = [ctypes.c_uint32]
    L.paged_attention_decode.restype = ctypes.c_int
    L.paged_attention_decode.argtypes = [_c_p, ctypes.POINTER(_c_i64), ctypes.POINTER(DecodeArgs),
                                         _c_p]
    L.paged_attention_v2_partition.restype = ctypes.c_int
    L.paged_attention_v2_partition.argtypes = [_c_p, _c_p, _c_p, _c_i32, _c_i32, _c_p,
                                               ctypes.POINTER(DecodeArgs), _c_p]
    L.paged_attention_v2_reduce.restype = ctypes.c_int
    L.paged_attention_v2_reduce.argtypes = [_c_p, ctypes.POINTER(_c_i64), _c_p, _c_p, _c_p, _c_p,
                                            _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                            ctypes.c_int, _c_p, _c_p]
    L.copy_page_indices.restype = ctypes.c_int
    L.copy_page_indices.argtypes = [_c_p, _c_i64, _c_p, _c_i32, _c_i64, _c_i64, _c_p, _c_i32,
                                    _c_p, _c_p]
    L.pkv_order_by_length.restype = ctypes.c_int
    L.pkv_order_by_length.argtypes = [_c_p, _c_p, _c_i32, _c_p]
    L.compute_num_kv_splits.restype = ctypes.c_int
    L.compute_num_kv_splits.argtypes = [_c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                        _c_i32, _c_p]
    L.prepare_decode_metadata.restype = ctypes.c_int
    L.prepare_decode_metadata.argtypes = [_c_p, _c_i64, _c_p, _c_i32, _c_i64, _c_i64, _c_p, _c_i32,
                                          _c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_p,
                                          _c_p]
    L.pkv_decode_metadata_args_size.restype = ctypes.c_size_t
    L.pkv_decode_metadata_args_size.argtypes = []
    if L.pkv_decode_metadata_args_size() != ctypes.sizeof(DecodeMetadataArgs):
        raise RuntimeError("pkv_decode_metadata_args_t layout mismatch")
    L.pkv_swa_spec_args_size.restype = ctypes.c_size_t
    L.pkv_swa_spec_args_size.argtypes = []
    if L.pkv_swa_spec_args_size() != ctypes.sizeof(SwaSpecArgs):
        raise RuntimeError("pkv_swa_spec_args_t layout mismatch")
    L.prepare_swa_spec_page_table.restype = ctypes.c_int
    L.prepare_swa_spec_page_table.argtypes = [ctypes.POINTER(SwaSpecArgs), _c_p]
    L.normal_decode_set_metadata.restype = ctypes.c_int
    L.normal_decode_set_metadata.argtypes = [ctypes.POINTER(DecodeMetadataArgs), _c_p]
    L.paged_attention_v2_noalloc.restype = ctypes.c_int
    L.paged_attention_v2_noalloc.argtypes = [_c_p, ctypes.POINTER(_c_i64), _c_i32, _c_i32, _c_p,
                                             ctypes.POINTER(DecodeArgs), _c_p]
    L.pkv_noalloc_scratch_bytes.restype = ctypes.c_size_t
    L.pkv_noalloc_scratch_bytes.argtypes = []
    if L.pkv_decode_args_size() != ctypes.sizeof(DecodeArgs):
        raise RuntimeError("pkv_decode_args_t layout mismatch between the library and the binding")
    _LIB = L
    return L


def version() -> str:
    return lib().pkv_version().decode()


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        msg = lib().pkv_status_string(status).decode()
        raise RuntimeError(f"{what} failed: {msg} (status {status})")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _cuda(t: Optional[torch.Tensor], name: str) -> None:
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library works on device memory)")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def set_attention_warps(warps: int) -> None:
    """Force warps per CTA (1, 2 or 4) for the attention kernels where that
    instance exists; 0 restores the measured per-call choice."""
    _check(lib().pkv_set_attention_warps(int(warps)), "pkv_set_attention_warps")


def set_fp8_kernel(which: int) -> None:
    """Kernel for fp8 caches (head size 128, block size 16): 0 the mma.sync
    kernel (default), 1 the tensor-memory kernel (see ``pkv_set_fp8_kernel``)."""
    _check(lib().pkv_set_fp8_kernel(int(which)), "pkv_set_fp8_kernel")


def set_split_fold(mode: int) -> None:
    """Split-KV over an fp8 cache on two-warp CTAs: 1 (default) half the
    partition slots with two partitions per CTA on batches that fill the GPU
    twice, 2 always, 0 never (see ``pkv_set_split_fold``)."""
    _check(lib().pkv_set_split_fold(int(mode)), "pkv_set_split_fold")


def set_wait_limit_ns(ns: int) -> None:
    """Limit of every copy wait in the attention kernels (0: the 2 s default)."""
    _check(lib().pkv_set_wait_limit_ns(int(ns)), "pkv_set_wait_limit_ns")


def _test_set_unarrived_bytes(nbytes: int) -> None:
    """Test hook: stages expect ``nbytes`` that never arrive, so waits time out."""
    _check(lib().pkv_test_set_unarrived_bytes(int(nbytes)), "pkv_test_set_unarrived_bytes")


def _kv_cache_code(key_cache, value_cache, query, kv_cache_dtype) -> int:
    """pkv_kv_cache_dtype_t of the caches.  fp8 caches are uint8 tensors of
    codes with an explicit ``kv_cache_dtype`` ("fp8", "fp8_e4m3", "fp8_e5m2"),
    or float8_e4m3fn / float8_e5m2 tensors ("auto" reads the format from them)."""
    if kv_cache_dtype not in _KV_CACHE_CODE:
        raise ValueError(f"unknown kv_cache_dtype {kv_cache_dtype!r}")
    if key_cache.dtype != value_cache.dtype:
        raise ValueError("key_cache and value_cache must share a dtype")
    code = _KV_CACHE_CODE[kv_cache_dtype]
    if key_cache.dtype in _FP8_TORCH:
        if code not in (0, _FP8_TORCH[key_cache.dtype]):
            raise ValueError(f"kv_cache_dtype {kv_cache_dtype!r} contradicts {key_cache.dtype}")
        return _FP8_TORCH[key_cache.dtype]
    if code == 0:
        if key_cache.dtype != query.dtype:
            raise ValueError("query, key_cache and value_cache must share a dtype")
        return 0
    if key_cache.dtype != torch.uint8:
        raise ValueError("fp8 caches are uint8 (codes) or float8 tensors")
    return code


def _decode_args(query, key_cache, value_cache, block_tables, seq_lens, scale, kv_indptr,
                 err_flag, max_blocks_per_seq, kv_cache_dtype="auto", k_scale=1.0, v_scale=1.0,
                 alibi_slopes=None) -> DecodeArgs:
    for t, n in ((query, "query"), (key_cache, "key_cache"), (value_cache, "value_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens"),
                 (kv_indptr, "kv_indptr"), (err_flag, "err_flag"),
                 (alibi_slopes, "alibi_slopes")):
        _cuda(t, n)
    if query.dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {query.dtype}")
    kv_code = _kv_cache_code(key_cache, value_cache, query, kv_cache_dtype)
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or
                                     not alibi_slopes.is_contiguous() or
                                     tuple(alibi_slopes.shape) != (query.shape[1],)):
        raise ValueError("alibi_slopes must be a contiguous float32 [num_heads] tensor")
    for t, n in ((block_tables, "block_tables"), (seq_lens, "seq_lens"), (kv_indptr, "kv_indptr"),
                 (err_flag, "err_flag")):
        if t is not None and t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    if query.dim() != 3 or key_cache.dim() != 5 or value_cache.dim() != 4:
        raise ValueError("expected query [B,H,D], key_cache [NB,Hk,D/x,bs,x], value_cache [NB,Hk,D,bs]")
    a = DecodeArgs()
    a.num_seqs, a.num_heads, a.head_size = query.shape
    a.num_kv_heads = key_cache.shape[1]
    a.block_size = key_cache.shape[3]
    a.x = key_cache.shape[4]
    a.num_blocks = key_cache.shape[0]
    if kv_indptr is None:
        if block_tables.dim() != 2:
            raise ValueError("block_tables must be 2-D [num_seqs, max_blocks_per_seq]")
        a.max_blocks_per_seq = block_tables.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq
        a.bt_stride[0], a.bt_stride[1] = block_tables.stride()
    else:
        if block_tables.dim() != 1:
            raise ValueError("with kv_indptr, block_tables is the flat page list (1-D)")
        a.max_blocks_per_seq = 0 if max_blocks_per_seq is None else max_blocks_per_seq
        a.bt_stride[0], a.bt_stride[1] = 0, block_tables.stride(0)
    a.dtype = _DTYPE_CODE[query.dtype]
    a.scale = float(scale)
    a.query = _ptr(query)
    for i, s in enumerate(query.stride()):
        a.q_stride[i] = s
    a.key_cache = _ptr(key_cache)
    for i, s in enumerate(key_cache.stride()):
        a.k_stride[i] = s
    a.value_cache = _ptr(value_cache)
    for i, s in enumerate(value_cache.stride()):
        a.v_stride[i] = s
    a.block_tables = _ptr(block_tables)
    a.kv_indptr = _ptr(kv_indptr)
    a.seq_lens = _ptr(seq_lens)
    a.err_flag = _ptr(err_flag)
    a.kv_cache_dtype = kv_code
    a.k_scale = float(k_scale)
    a.v_scale = float(v_scale)
    a.alibi_slopes = _ptr(alibi_slopes)
    return a


def paged_attention_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, block_tables: torch.Tensor,
                           seq_lens: torch.Tensor, scale: float, *,
                           kv_indptr: Optional[torch.Tensor] = None,
                           err_flag: Optional[torch.Tensor] = None,
                           max_blocks_per_seq: Optional[int] = None,
                           kv_cache_dtype: str = "auto", k_scale: float = 1.0,
                           v_scale: float = 1.0, alibi_slopes: Optional[torch.Tensor] = None,
                           seq_order: Optional[torch.Tensor] = None, stream=None) -> None:
    """Single-pass decode into ``out [num_seqs, num_heads, head_size]`` (query's dtype).

    ``kv_cache_dtype`` ("auto", "fp8", "fp8_e4m3", "fp8_e5m2") with uint8 code
    caches, or float8 caches under "auto", selects an fp8 cache dequantised as
    ``code * k_scale`` / ``code * v_scale``; ``alibi_slopes`` (float32
    ``[num_heads]``) adds ``slope_h * (t - seq_len + 1)`` to the logits;
    ``seq_order`` (int32 ``[num_seqs]``, a permutation, e.g. from
    :func:`order_by_length`) sets the order in which sequences are launched."""
    _cuda(out, "out")
    if out.dtype != query.dtype or tuple(out.shape) != tuple(query.shape):
        raise ValueError("out must match query's shape and dtype")
    a = _decode_args(query, key_cache, value_cache, block_tables, seq_lens, scale, kv_indptr,
                     err_flag, max_blocks_per_seq, kv_cache_dtype, k_scale,
                     v_scale, alibi_slopes)
    if seq_order is not None:
        _cuda(seq_order, "seq_order")
        if (seq_order.dtype != torch.int32 or not seq_order.is_contiguous() or
                tuple(seq_order.shape) != (query.shape[0],)):
            raise ValueError("seq_order must be a contiguous int32 [num_seqs] tensor")
        a.seq_order = _ptr(seq_order)
    os_ = _I64x3(*out.stride())
    _check(lib().paged_attention_decode(_ptr(out), os_, ctypes.byref(a), _stream(stream)),
           "paged_attention_decode")


def order_by_length(order: torch.Tensor, seq_lens: torch.Tensor, stream=None) -> None:
    """Longest-first launch order of ``seq_lens`` into ``order`` (int32, same length)."""
    for t, n in ((order, "order"), (seq_lens, "seq_lens")):
        _cuda(t, n)
        if t.dtype != torch.int32 or not t.is_contiguous() or t.dim() != 1:
            raise ValueError(f"{n} must be a contiguous 1-D int32 tensor")
    if order.numel() != seq_lens.numel():
        raise ValueError("order and seq_lens must have the same length")
    _check(lib().pkv_order_by_length(_ptr(order), _ptr(seq_lens), order.numel(), _stream(stream)),
           "pkv_order_by_length")


def paged_attention_v2_partition(tmp_out: torch.Tensor, exp_sums: torch.Tensor,
                                 max_logits: torch.Tensor, query: torch.Tensor,
                                 key_cache: torch.Tensor, value_cache: torch.Tensor,
                                 block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                                 *, partition_size: int = 512,
                                 num_kv_splits: Optional[torch.Tensor] = None,
                                 kv_indptr: Optional[torch.Tensor] = None,
                                 err_flag: Optional[torch.Tensor] = None,
                                 max_blocks_per_seq: Optional[int] = None,
                                 kv_cache_dtype: str = "auto", k_scale: float = 1.0,
                                 v_scale: float = 1.0, alibi_slopes: Optional[torch.Tensor] = None,
                                 stream=None) -> None:
    """Split-KV partition pass; ``tmp_out [B,H,maxP,D]``, ``exp_sums``/``max_logits [B,H,maxP]`` fp32."""
    for t, n in ((tmp_out, "tmp_out"), (exp_sums, "exp_sums"), (max_logits, "max_logits"),
                 (num_kv_splits, "num_kv_splits")):
        _cuda(t, n)
    for t in (tmp_out, exp_sums, max_logits):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("tmp_out, exp_sums and max_logits must be contiguous float32")
    B, H, maxP, D = tmp_out.shape
    if (B, H, D) != tuple(query.shape) or tuple(exp_sums.shape) != (B, H, maxP) or \
            tuple(max_logits.shape) != (B, H, maxP):
        raise ValueError("scratch shapes do not match the query")
    if num_kv_splits is not None and num_kv_splits.dtype != torch.int32:
        raise ValueError("num_kv_splits must be int32")
    a = _decode_args(query, key_cache, value_cache, block_tables, seq_lens, scale, kv_indptr,
                     err_flag, max_blocks_per_seq, kv_cache_dtype, k_scale,
                     v_scale, alibi_slopes)
    _check(lib().paged_attention_v2_partition(_ptr(tmp_out), _ptr(exp_sums), _ptr(max_logits),
                                              maxP, int(partition_size), _ptr(num_kv_splits),
                                              ctypes.byref(a), _stream(stream)),
           "paged_attention_v2_partition")


def paged_attention_v2_reduce(out: torch.Tensor, tmp_out: torch.Tensor, exp_sums: torch.Tensor,
                              max_logits: torch.Tensor, seq_lens: torch.Tensor, *,
                              partition_size: int = 512,
                              num_kv_splits: Optional[torch.Tensor] = None, block_size: int = 16,
                              err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """Log-sum-exp combination of the partitions into ``out [B, H, D]``."""
    for t, n in ((out, "out"), (tmp_out, "tmp_out"), (exp_sums, "exp_sums"),
                 (max_logits, "max_logits"), (seq_lens, "seq_lens"),
                 (num_kv_splits, "num_kv_splits"), (err_flag, "err_flag")):
        _cuda(t, n)
    if out.dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {out.dtype}")
    for t in (tmp_out, exp_sums, max_logits):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("tmp_out, exp_sums and max_logits must be contiguous float32")
    B, H, maxP, D = tmp_out.shape
    if tuple(out.shape) != (B, H, D):
        raise ValueError("out must be [num_seqs, num_heads, head_size]")
    os_ = _I64x3(*out.stride())
    _check(lib().paged_attention_v2_reduce(_ptr(out), os_, _ptr(tmp_out), _ptr(exp_sums),
                                           _ptr(max_logits), _ptr(seq_lens), _ptr(num_kv_splits),
                                           B, H, D, int(block_size), maxP, int(partition_size),
                                           _DTYPE_CODE[out.dtype], _ptr(err_flag),
                                           _stream(stream)),
           "paged_attention_v2_reduce")


def copy_page_indices(page_indices: torch.Tensor, block_table: torch.Tensor,
                      cu_num_blocks: torch.Tensor, *, err_flag: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    """``page_indices[cu[i] + j] = block_table[i, j]`` for ``j < cu[i+1] - cu[i]`` (any strides)."""
    for t, n in ((page_indices, "page_indices"), (block_table, "block_table"),
                 (cu_num_blocks, "cu_num_blocks"), (err_flag, "err_flag")):
        _cuda(t, n)
        if t is not None and t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    if block_table.dim() != 2 or cu_num_blocks.dim() != 1 or page_indices.dim() != 1:
        raise ValueError("expected block_table [R, C], cu_num_blocks [R+1], page_indices [N]")
    if not page_indices.is_contiguous() or not cu_num_blocks.is_contiguous():
        raise ValueError("page_indices and cu_num_blocks must be contiguous")
    R = cu_num_blocks.shape[0] - 1
    if R > block_table.shape[0]:
        raise ValueError("cu_num_blocks has more rows than block_table")
    s0, s1 = block_table.stride()
    _check(lib().copy_page_indices(_ptr(page_indices), page_indices.numel(), _ptr(block_table),
                                   block_table.shape[1], s0, s1, _ptr(cu_num_blocks), R,
                                   _ptr(err_flag), _stream(stream)),
           "copy_page_indices")


def compute_num_kv_splits(num_kv_splits: torch.Tensor, seq_lens: torch.Tensor, *, num_group: int,
                          num_head: int, num_kv_head: int, max_kv_splits: int,
                          device_core_count: int, stream=None) -> None:
    """Per-sequence split count into ``num_kv_splits [num_seq * num_group]`` (int32)."""
    for t, n in ((num_kv_splits, "num_kv_splits"), (seq_lens, "seq_lens")):
        _cuda(t, n)
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous int32")
    n = seq_lens.numel()
    if num_kv_splits.numel() < n * num_group:
        raise ValueError("num_kv_splits is too small")
    _check(lib().compute_num_kv_splits(_ptr(num_kv_splits), _ptr(seq_lens), n, int(num_group),
                                       int(num_head), int(num_kv_head), int(max_kv_splits),
                                       int(device_core_count), _stream(stream)),
           "compute_num_kv_splits")


def prepare_decode_metadata(page_indices: torch.Tensor, block_table: torch.Tensor,
                            cu_num_blocks: torch.Tensor, num_kv_splits: torch.Tensor,
                            seq_lens: torch.Tensor, *, num_group: int, num_head: int,
                            num_kv_head: int, max_kv_splits: int, device_core_count: int,
                            err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """``copy_page_indices`` and ``compute_num_kv_splits`` in one launch."""
    for t, n in ((page_indices, "page_indices"), (block_table, "block_table"),
                 (cu_num_blocks, "cu_num_blocks"), (num_kv_splits, "num_kv_splits"),
                 (seq_lens, "seq_lens"), (err_flag, "err_flag")):
        _cuda(t, n)
        if t is not None and t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    if block_table.dim() != 2 or cu_num_blocks.dim() != 1 or page_indices.dim() != 1:
        raise ValueError("expected block_table [R, C], cu_num_blocks [R+1], page_indices [N]")
    for t, n in ((page_indices, "page_indices"), (cu_num_blocks, "cu_num_blocks"),
                 (num_kv_splits, "num_kv_splits"), (seq_lens, "seq_lens")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    R = cu_num_blocks.shape[0] - 1
    if R > block_table.shape[0] or seq_lens.numel() != R or num_kv_splits.numel() < R * num_group:
        raise ValueError("inconsistent row counts")
    s0, s1 = block_table.stride()
    _check(lib().prepare_decode_metadata(_ptr(page_indices), page_indices.numel(),
                                         _ptr(block_table), block_table.shape[1], s0, s1,
                                         _ptr(cu_num_blocks), R, _ptr(num_kv_splits),
                                         _ptr(seq_lens), int(num_group), int(num_head),
                                         int(num_kv_head), int(max_kv_splits),
                                         int(device_core_count), _ptr(err_flag), _stream(stream)),
           "prepare_decode_metadata")


def decode_metadata_args(cache_seqlens, cu_seqlens_k, page_table, req_to_token, req_pool_indices,
                         seq_lens, *, seq_len_delta: int, page_size: int,
                         max_seq_pages: Optional[int] = None, swa_page_table=None,
                         full_to_swa_mapping=None, err_flag=None,
                         cu_num_pages=None) -> DecodeMetadataArgs:
    """Fill the argument struct of ``normal_decode_set_metadata`` from tensors."""
    checks = ((cache_seqlens, "cache_seqlens", torch.int32), (cu_seqlens_k, "cu_seqlens_k", torch.int32),
              (page_table, "page_table", torch.int32), (req_to_token, "req_to_token", torch.int32),
              (req_pool_indices, "req_pool_indices", torch.int64), (seq_lens, "seq_lens", torch.int64),
              (swa_page_table, "swa_page_table", torch.int32),
              (full_to_swa_mapping, "full_to_swa_mapping", torch.int64),
              (err_flag, "err_flag", torch.int32), (cu_num_pages, "cu_num_pages", torch.int32))
    for t, n, dt in checks:
        _cuda(t, n)
        if t is not None and t.dtype != dt:
            raise ValueError(f"{n} must be {dt}")
    B = seq_lens.shape[0]
    if max_seq_pages is None:
        max_seq_pages = page_table.shape[1]
    if page_table.dim() != 2 or page_table.shape[0] < B or page_table.shape[1] < max_seq_pages:
        raise ValueError("page_table must be at least [batch_size, max_seq_pages]")
    if cu_seqlens_k.shape[0] < B + 1 or cache_seqlens.shape[0] < B or req_pool_indices.shape[0] < B:
        raise ValueError("output / index tensors are too short for the batch")
    a = DecodeMetadataArgs()
    a.batch_size, a.max_seq_pages = B, int(max_seq_pages)
    a.seq_len_delta, a.page_size = int(seq_len_delta), int(page_size)
    a.seq_lens, a.seq_lens_stride = _ptr(seq_lens), seq_lens.stride(0)
    a.req_to_token = _ptr(req_to_token)
    a.req_to_token_stride[0], a.req_to_token_stride[1] = req_to_token.stride()
    a.req_to_token_rows, a.req_to_token_cols = req_to_token.shape
    a.req_pool_indices, a.req_pool_indices_stride = _ptr(req_pool_indices), req_pool_indices.stride(0)
    a.cache_seqlens, a.cache_seqlens_stride = _ptr(cache_seqlens), cache_seqlens.stride(0)
    a.cu_seqlens_k, a.cu_seqlens_k_stride = _ptr(cu_seqlens_k), cu_seqlens_k.stride(0)
    a.page_table = _ptr(page_table)
    a.page_table_stride[0], a.page_table_stride[1] = page_table.stride()
    if swa_page_table is not None:
        if full_to_swa_mapping is None:
            raise ValueError("swa_page_table needs full_to_swa_mapping")
        a.swa_page_table = _ptr(swa_page_table)
        a.swa_page_table_stride[0], a.swa_page_table_stride[1] = swa_page_table.stride()
        a.full_to_swa_mapping = _ptr(full_to_swa_mapping)
        a.full_to_swa_stride = full_to_swa_mapping.stride(0)
        a.full_to_swa_len = full_to_swa_mapping.shape[0]
    a.err_flag = _ptr(err_flag)
    if cu_num_pages is not None:
        if cu_num_pages.dim() != 1 or cu_num_pages.shape[0] < B + 1:
            raise ValueError("cu_num_pages must hold batch_size + 1 entries")
        a.cu_num_pages, a.cu_num_pages_stride = _ptr(cu_num_pages), cu_num_pages.stride(0)
    return a


def normal_decode_set_metadata(cache_seqlens, cu_seqlens_k, page_table, req_to_token,
                               req_pool_indices, seq_lens, *, seq_len_delta: int, page_size: int,
                               max_seq_pages: Optional[int] = None, swa_page_table=None,
                               full_to_swa_mapping=None, err_flag=None, cu_num_pages=None,
                               stream=None) -> None:
    """Fused decode metadata: lengths + delta, their int32 indptr, the page
    table gathered from ``req_to_token`` (and the sliding-window table); with
    ``cu_num_pages`` (int32 ``[batch_size + 1]``) also the page-count indptr
    that the page-index copy takes as ``cu_num_blocks``."""
    a = decode_metadata_args(cache_seqlens, cu_seqlens_k, page_table, req_to_token,
                             req_pool_indices, seq_lens, seq_len_delta=seq_len_delta,
                             page_size=page_size, max_seq_pages=max_seq_pages,
                             swa_page_table=swa_page_table, full_to_swa_mapping=full_to_swa_mapping,
                             err_flag=err_flag, cu_num_pages=cu_num_pages)
    _check(lib().normal_decode_set_metadata(ctypes.byref(a), _stream(stream)),
           "normal_decode_set_metadata")


def prepare_swa_spec_page_table(dst: torch.Tensor, page_table_a: torch.Tensor,
                                page_table_b: torch.Tensor, seq_len_a: torch.Tensor,
                                seq_len_b: torch.Tensor, num_draft_tokens: int, *,
                                err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """Row m of ``dst`` = row m // R of table A cut to its length, then row m of B."""
    for t, n in ((dst, "dst"), (page_table_a, "page_table_a"), (page_table_b, "page_table_b"),
                 (seq_len_a, "seq_len_a"), (seq_len_b, "seq_len_b"), (err_flag, "err_flag")):
        _cuda(t, n)
        if t is not None and t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    bs = seq_len_a.shape[0]
    R = int(num_draft_tokens)
    if seq_len_b.shape[0] != bs * R:
        raise ValueError("seq_len_b must have bs * num_draft_tokens entries")
    LA, LB = page_table_a.shape[1], page_table_b.shape[1]
    if page_table_a.shape[0] < bs or page_table_b.shape[0] < bs * R:
        raise ValueError("page tables have too few rows")
    if dst.shape[0] < bs * R or dst.shape[1] < LA + LB:
        raise ValueError("dst must be at least [bs * num_draft_tokens, len_a + len_b]")
    a = SwaSpecArgs()
    a.bs, a.num_draft_tokens, a.len_a, a.len_b = bs, R, LA, LB
    a.page_table_a = _ptr(page_table_a)
    a.a_stride[0], a.a_stride[1] = page_table_a.stride()
    a.page_table_b = _ptr(page_table_b)
    a.b_stride[0], a.b_stride[1] = page_table_b.stride()
    a.seq_len_a, a.seq_len_a_stride = _ptr(seq_len_a), seq_len_a.stride(0)
    a.seq_len_b, a.seq_len_b_stride = _ptr(seq_len_b), seq_len_b.stride(0)
    a.dst = _ptr(dst)
    a.dst_stride[0], a.dst_stride[1] = dst.stride()
    a.err_flag = _ptr(err_flag)
    _check(lib().prepare_swa_spec_page_table(ctypes.byref(a), _stream(stream)),
           "prepare_swa_spec_page_table")


def noalloc_scratch_bytes() -> int:
    """Size of the fixed device scratch array behind ``paged_attention_v2_noalloc``."""
    return int(lib().pkv_noalloc_scratch_bytes())


def paged_attention_v2_noalloc(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                               value_cache: torch.Tensor, block_tables: torch.Tensor,
                               seq_lens: torch.Tensor, scale: float, *, max_num_partitions: int,
                               partition_size: int = 512,
                               num_kv_splits: Optional[torch.Tensor] = None,
                               kv_indptr: Optional[torch.Tensor] = None,
                               err_flag: Optional[torch.Tensor] = None,
                               max_blocks_per_seq: Optional[int] = None,
                               kv_cache_dtype: str = "auto", k_scale: float = 1.0,
                               v_scale: float = 1.0, alibi_slopes: Optional[torch.Tensor] = None,
                               stream=None) -> None:
    """Split-KV decode into ``out`` for callers that cannot allocate device
    memory: the partition scratch lives in the library's fixed device array
    (see ``noalloc_scratch_bytes``) instead of caller-provided buffers.  Calls
    share that array, so calls that overlap on the GPU race."""
    _cuda(out, "out")
    _cuda(num_kv_splits, "num_kv_splits")
    if out.dtype != query.dtype or tuple(out.shape) != tuple(query.shape):
        raise ValueError("out must match query's shape and dtype")
    if num_kv_splits is not None and num_kv_splits.dtype != torch.int32:
        raise ValueError("num_kv_splits must be int32")
    a = _decode_args(query, key_cache, value_cache, block_tables, seq_lens, scale, kv_indptr,
                     err_flag, max_blocks_per_seq, kv_cache_dtype, k_scale,
                     v_scale, alibi_slopes)
    os_ = _I64x3(*out.stride())
    _check(lib().paged_attention_v2_noalloc(_ptr(out), os_, int(max_num_partitions),
                                            int(partition_size), _ptr(num_kv_splits),
                                            ctypes.byref(a), _stream(stream)),
           "paged_attention_v2_noalloc")
