"""CPU oracle for the sync-free decode metadata steps.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.

* ``copy_page_indices``: vLLM PR 35765 ("AITER MLA backend: Avoid CPU sync in
  _build_decode"), ``_copy_page_indices_kernel`` with the review's
  ``block_table_stride_1`` change: row ``i`` of the block table, columns
  ``0 .. cu_num_blocks[i+1] - cu_num_blocks[i] - 1``, lands at
  ``page_indices[cu_num_blocks[i] + j]``.
* ``num_kv_splits``: sglang ``python/sglang/kernels/ops/attention/metadata.py``,
  ``get_num_kv_splits_triton``, restated step by step in integer arithmetic
  except for the one float32 step the page has (``log2`` of ``max_seq_len /
  64`` in float32, times the core count, truncated to int32).
"""
from __future__ import annotations

import math
from typing import List, Sequence

import numpy as np

__all__ = ["copy_page_indices", "num_kv_splits", "ext_device_core_count", "log2_f32", "cdiv",
           "decode_set_metadata", "wrap_int32", "swa_spec_page_table"]


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def copy_page_indices(block_table, cu_num_blocks: Sequence[int], page_indices_len: int,
                      fill: int = -12345) -> List[int]:
    """Flatten block-table rows through an indptr.

    ``block_table`` is anything indexable as ``block_table[i][j]`` (a strided
    torch view works).  Positions of ``page_indices`` that no row writes keep
    ``fill`` so a test can see that a kernel left them untouched.
    """
    out = [fill] * page_indices_len
    num_reqs = len(cu_num_blocks) - 1
    for i in range(num_reqs):
        start = int(cu_num_blocks[i])
        n = int(cu_num_blocks[i + 1]) - start
        for j in range(n):
            out[start + j] = int(block_table[i][j])
    return out


def log2_f32(x: np.float32) -> np.float32:
    """log2 of a float32, correctly rounded to float32.

    Reading of ``tl.log2`` on a float32 tensor: the page does not fix the
    accuracy, so the float32 nearest to the exact value is taken.  It is
    computed as the float64 ``log2`` rounded once to float32.
    """
    return np.float32(math.log2(float(x)))


def ext_device_core_count(max_seq_len: int, device_core_count: int) -> int:
    """Step 3 of ``get_num_kv_splits_triton``: the core count stretched by
    ``max(log2(max_seq_len / 64), 1)``, evaluated in float32 and truncated
    toward zero like the page's cast to int32."""
    ext_seq_len = np.float32(max_seq_len) / np.float32(64.0)
    lg = log2_f32(ext_seq_len)
    prod = np.float32(device_core_count) * np.maximum(lg, np.float32(1.0))
    return int(prod)


def num_kv_splits(seq_lens: Sequence[int], num_group: int, num_head: int, num_kv_head: int,
                  max_kv_splits: int, device_core_count: int) -> List[int]:
    """Per-sequence split count, output indexed ``seq * num_group + i``.

    Follows ``get_num_kv_splits_triton`` in the page's order:

    1. ``max_seq_len`` and ``min_seq_len`` over the batch; if
       ``max * 8 < min * 10`` the batch counts as uniform (``min = max``).
    2. ``max_kv_splits_1 = min(cdiv(max, min), max_kv_splits)``,
       ``kv_chunk_size_1 = cdiv(max, max_kv_splits_1)``.
    3. ``ext_device_core_count = int32(core_count * max(log2(max / 64), 1))``
       with the division and log2 in float32.
    4. ``token_grid``: ``num_seq * num_group * num_head`` without GQA,
       else ``num_seq * num_group * cdiv(num_head, min(16, num_head // num_kv_head))``.
    5. ``max_kv_splits_2 = min(cdiv(ext, token_grid), max_kv_splits)``,
       ``kv_chunk_size_2 = cdiv(max, max_kv_splits_2)``.
    6. ``num_kv_splits = max(cdiv(len, chunk_1), cdiv(len, chunk_2))``.

    Reading for empty sequences (the page divides by ``min_seq_len``): the
    batch statistics use ``max(len, 1)``; the per-sequence count uses the
    true length, so a zero-length sequence gets 0 splits.
    """
    lens = [int(v) for v in seq_lens]
    num_seq = len(lens)
    if num_seq == 0:
        return []
    mx = max(max(v, 1) for v in lens)
    mn = min(max(v, 1) for v in lens)
    if mx * 8 < mn * 10:
        mn = mx
    s1 = min(cdiv(mx, mn), max_kv_splits)
    c1 = cdiv(mx, s1)

    ext = ext_device_core_count(mx, device_core_count)

    block_h = 16
    kv_group = num_head // num_kv_head
    if kv_group == 1:
        token_grid = num_seq * num_group * num_head
    else:
        block_h = min(block_h, kv_group)
        token_grid = num_seq * num_group * cdiv(num_head, block_h)
    s2 = min(cdiv(ext, token_grid), max_kv_splits)
    c2 = cdiv(mx, s2)

    out = [0] * (num_seq * num_group)
    for s, L in enumerate(lens):
        v = max(cdiv(max(L, 0), c1), cdiv(max(L, 0), c2))
        for i in range(num_group):
            out[s * num_group + i] = v
    return out


def wrap_int32(v: int) -> int:
    """Two's-complement int32 value of ``v`` (what a cast to int32 keeps)."""
    v &= 0xFFFFFFFF
    return v - (1 << 32) if v >= (1 << 31) else v


def decode_set_metadata(seq_lens, req_to_token, req_pool_indices, max_seq_pages: int,
                        seq_len_delta: int, page_size: int, full_to_swa_mapping=None):
    """sglang ``normal_decode_set_metadata`` (python/sglang/kernels/ops/attention/
    metadata.py) with its kernels ``_fused_metadata_kernel_general`` and
    ``_fused_metadata_kernel_ps1_no_swa``, step by step:

    1. ``cache_seqlens[i] = int32(seq_lens[i] + seq_len_delta)``;
    2. ``cu_seqlens_k``: running int32 sum, ``cu[i]`` before adding entry i,
       ``cu[B]`` the total;
    3. ``page_index = req_to_token[req_pool_indices[i], c << SHIFT]`` for every
       column ``c < max_seq_pages`` (``SHIFT = log2(page_size)``);
    4. ``page_table[i, c] = page_index >> SHIFT``;
    5. with a ``full_to_swa_mapping``: ``swa_page_table[i, c] =
       full_to_swa_mapping[page_index] >> SHIFT``, stored as int32.

    Returns ``(cache_seqlens, cu_seqlens_k, page_table, swa_page_table)`` as
    Python lists (``swa_page_table`` is None without a mapping).
    """
    if page_size <= 0 or page_size & (page_size - 1):
        raise ValueError("page_size must be a power of two")
    shift = page_size.bit_length() - 1
    B = len(seq_lens)
    cache = []
    cu = []
    acc = 0
    for i in range(B):
        val = wrap_int32(int(seq_lens[i]) + seq_len_delta)
        cache.append(val)
        cu.append(acc)
        acc = wrap_int32(acc + val)
    cu.append(acc)
    page_table, swa = [], ([] if full_to_swa_mapping is not None else None)
    for i in range(B):
        row = int(req_pool_indices[i])
        pt_row, swa_row = [], []
        for c in range(max_seq_pages):
            page_index = int(req_to_token[row][c << shift])
            pt_row.append(page_index >> shift)
            if swa is not None:
                swa_row.append(wrap_int32(int(full_to_swa_mapping[page_index]) >> shift))
        page_table.append(pt_row)
        if swa is not None:
            swa.append(swa_row)
    return cache, cu, page_table, swa


def cu_num_pages(cache_seqlens: Sequence[int], page_size: int):
    """Page-count indptr of a decode batch: ``cu[0] = 0`` and ``cu[i + 1] =
    cu[i] + ceil(cache_seqlens[i] / page_size)`` as a running int32 sum (a
    negative length holds no page).  It is the ``cu_num_blocks`` indptr that
    ``copy_page_indices`` (vLLM PR 35765, ``_copy_page_indices_kernel``)
    reads, built from the lengths the fused decode metadata produces (sglang
    ``normal_decode_set_metadata``, ``cache_seqlens``); the pages leave its
    construction to the caller, so this is the plain definition."""
    if page_size <= 0:
        raise ValueError("page_size must be positive")
    cu = [0]
    acc = 0
    for n in cache_seqlens:
        pages = cdiv(int(n), page_size) if int(n) > 0 else 0
        acc = wrap_int32(acc + pages)
        cu.append(acc)
    return cu


def swa_spec_page_table(dst, page_table_a, page_table_b, seq_len_a, seq_len_b,
                        num_draft_tokens: int):
    """sglang ``prepare_swa_spec_page_table_triton`` / ``_prepare_swa_spec_page_table_kernel``
    (python/sglang/kernels/ops/attention/metadata.py): row ``m`` of the output
    (one per draft token; ``bs_expand = bs * num_draft_tokens`` rows) is row
    ``m // num_draft_tokens`` of table A, cut to that request's ``seq_len_a``,
    followed by row ``m`` of table B, cut to ``seq_len_b[m]``.  With
    ``la = seq_len_a[m // R]``, ``lb = seq_len_b[m]`` and widths ``LEN_A``,
    ``LEN_B``, for every column ``n < min(la + lb, LEN_A + LEN_B)``:

    * ``n < la``: ``A[m // R, n]`` if ``n < LEN_A`` else 0;
    * otherwise, ``k = n - la``: ``B[m, k]`` if ``k < LEN_B`` else 0.

    Columns at or beyond ``la + lb`` keep their old value.  ``dst`` is a list
    of lists updated in place and returned.
    """
    R = num_draft_tokens
    len_a = len(page_table_a[0]) if len(page_table_a) else 0
    len_b = len(page_table_b[0]) if len(page_table_b) else 0
    for m in range(len(seq_len_b)):
        la = int(seq_len_a[m // R])
        lb = int(seq_len_b[m])
        for n in range(min(la + lb, len_a + len_b)):
            if n < la:
                dst[m][n] = int(page_table_a[m // R][n]) if n < len_a else 0
            else:
                k = n - la
                dst[m][n] = int(page_table_b[m][k]) if k < len_b else 0
    return dst
