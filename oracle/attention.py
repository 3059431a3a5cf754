"""CPU float64 oracle for paged-KV decode attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  The CUDA library never
calls it and shares no code with it.

It computes the plain definition that the single-pass (v1) and split-KV (v2)
decode kernels reach faster, step by step as the pages state it:

* Token -> (physical block, slot): ``block = block_tables[seq, t // block_size]``,
  ``slot = t % block_size``.  Page "Needs help on performance optimization"
  (triton-lang/triton issue 2522), the worked example table, and page
  "paged_attention_v2_triton.py", module docstring ("The Phase 1 paged gather
  is the hard part", steps 1 and 2).
* K/V gather from ``key_cache [num_blocks, num_kv_heads, head_size/x,
  block_size, x]`` and ``value_cache [num_blocks, num_kv_heads, head_size,
  block_size]`` (same page, partition-kernel argument comments).
* score = q . k * scale, softmax, weighted sum over V (same page, "Algorithm
  per instance" steps 1-4).
* v2: per partition the max logit, the sum of exponentials and the
  normalised partial output; empty partitions carry -inf / 0 (same page,
  ``_paged_attn_v2_partition_kernel``), then the log-sum-exp reduce
  (``_paged_attn_v2_reduce_kernel``: global max, rescale, weighted sum).

Everything is upcast to float64 from the exact stored values before any
arithmetic.

Two variants the same page's wrapper names but does not define
(``alibi_slopes``, ``kv_cache_dtype`` / ``k_scale`` / ``v_scale``), in the
reading stated in ``oracle.fp8`` and ``alibi_bias``: fp8 caches are decoded
from their 8-bit codes and scaled, and ALiBi adds ``slope_h * (t - L + 1)``
to the logit of token ``t``.  The query-head -> kv-head map is ``h // (num_heads //
num_kv_heads)`` (contiguous groups, the vLLM convention the page says it
follows; its own mapping line is a placeholder marked TODO).
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import torch

from . import fp8

__all__ = [
    "token_offsets",
    "sequence_block_ids",
    "gather_kv",
    "attention_one_head",
    "kv_head_of",
    "decode_v1",
    "split_chunk_size",
    "partition_ranges",
    "v2_partition",
    "v2_reduce",
    "alibi_bias",
]

NEG_INF = float("-inf")


def token_offsets(block_table_row: Sequence[int], block_size: int, seq_len: int,
                  block_stride: int = 1, slot_stride: int = 1):
    """Offset of every token of one sequence in a cache addressed by
    ``block * block_stride + slot * slot_stride``.

    With unit strides this is the table printed in "Needs help on performance
    optimization" (triton-lang/triton issue 2522): block table [40, 30] and
    block_size 8 give offsets 40..47 then 30..37.
    """
    out = []
    for t in range(seq_len):
        block = int(block_table_row[t // block_size])
        slot = t % block_size
        out.append(block * block_stride + slot * slot_stride)
    return out


def sequence_block_ids(block_tables: torch.Tensor, seq: int, num_pages: int,
                       kv_indptr: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Physical block ids of the first ``num_pages`` logical pages of ``seq``.

    ``block_tables`` is a 2-D (possibly strided) table, or, when ``kv_indptr``
    is given, the flat ``page_indices`` list whose row ``seq`` starts at
    ``kv_indptr[seq]`` (the CSR form built by the page-index copy of vLLM PR
    35765).
    """
    if kv_indptr is None:
        return block_tables[seq, :num_pages].to(torch.int64)
    start = int(kv_indptr[seq])
    return block_tables[start:start + num_pages].to(torch.int64)


def gather_kv(key_cache: torch.Tensor, value_cache: torch.Tensor, block_ids: torch.Tensor,
              seq_len: int, kv_head: int, kv_format: Optional[str] = None, k_scale: float = 1.0,
              v_scale: float = 1.0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Materialise one sequence's keys and values, ``[seq_len, head_size]`` float64.

    ``k_t[d] = key_cache[b, kv_head, d // x, t % bs, d % x]`` and
    ``v_t[d] = value_cache[b, kv_head, d, t % bs]`` with ``b = block_ids[t // bs]``.
    With an fp8 ``kv_format`` the caches hold uint8 codes: keys are
    ``decode(code) * k_scale`` and values ``decode(code) * v_scale``.
    """
    bs = key_cache.shape[3]
    D = value_cache.shape[2]
    t = torch.arange(seq_len)
    blk = block_ids[t // bs]
    slot = t % bs
    # Advanced indices (blk, kv_head, slot) are separated by a slice, so the
    # token axis comes first: [seq_len, head_size // x, x] and [seq_len, head_size].
    K = key_cache[blk, kv_head, :, slot, :].reshape(seq_len, D)
    V = value_cache[blk, kv_head, :, slot]
    if kv_format is None:
        return K.to(torch.float64), V.to(torch.float64)
    return fp8.decode(K, kv_format) * k_scale, fp8.decode(V, kv_format) * v_scale


def alibi_bias(slope: float, seq_len: int) -> torch.Tensor:
    """ALiBi term of every logit of one decode query, ``[seq_len]`` float64.

    The split-KV wrapper on page "paged_attention_v2_triton.py" takes
    ``alibi_slopes`` without defining them.  Reading: ALiBi as defined in
    "Train Short, Test Long: Attention with Linear Biases" (Press, Smith,
    Lewis, 2022), a bias of ``-slope * distance`` between the query and key
    positions, with the decode query at position ``seq_len - 1``:
    ``slope * (t - seq_len + 1)`` for key ``t``, added to the scaled score.
    """
    t = torch.arange(seq_len, dtype=torch.float64)
    return float(slope) * (t - (seq_len - 1))


def _kv_options(key_cache, value_cache, kv_cache_dtype, k_scale, v_scale):
    """(caches as stored codes, keyword arguments for gather_kv)."""
    fmt = fp8.format_of(kv_cache_dtype)
    if fmt is None:
        return key_cache, value_cache, {}
    if key_cache.dtype != torch.uint8:
        key_cache = key_cache.view(torch.uint8)
    if value_cache.dtype != torch.uint8:
        value_cache = value_cache.view(torch.uint8)
    return key_cache, value_cache, dict(kv_format=fmt, k_scale=float(k_scale),
                                        v_scale=float(v_scale))


def attention_one_head(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float,
                       bias: Optional[torch.Tensor] = None):
    """Textbook softmax attention of one query vector over ``K``/``V`` (float64).

    ``bias`` (optional, ``[seq_len]``) is added to the scaled scores.
    Returns ``(out, logits)``; an empty sequence gives a zero output.
    """
    q = q.to(torch.float64)
    if K.shape[0] == 0:
        return torch.zeros(V.shape[1], dtype=torch.float64), torch.zeros(0, dtype=torch.float64)
    z = (K @ q) * scale
    if bias is not None:
        z = z + bias
    p = torch.exp(z - z.max())
    p = p / p.sum()
    return p @ V, z


def kv_head_of(head: int, num_heads: int, num_kv_heads: int) -> int:
    """KV head serving query ``head``: contiguous groups of ``num_heads //
    num_kv_heads`` query heads share one KV head."""
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    return head // (num_heads // num_kv_heads)


def decode_v1(query, key_cache, value_cache, block_tables, seq_lens, scale: float,
              seqs: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None,
              kv_indptr: Optional[torch.Tensor] = None, kv_cache_dtype: str = "auto",
              k_scale: float = 1.0, v_scale: float = 1.0,
              alibi_slopes: Optional[Sequence[float]] = None) -> torch.Tensor:
    """Single-pass decode output ``[num_seqs, num_heads, head_size]`` float64.

    ``seqs`` / ``heads`` restrict the work to a subset (other rows stay NaN),
    so that full-size batches can be checked on sampled outputs.
    ``kv_cache_dtype`` / ``k_scale`` / ``v_scale``: see ``oracle.fp8``;
    ``alibi_slopes`` (``[num_heads]``): see ``alibi_bias``.
    """
    B, H, D = query.shape
    Hk = key_cache.shape[1]
    bs = key_cache.shape[3]
    key_cache, value_cache, kvq = _kv_options(key_cache, value_cache, kv_cache_dtype, k_scale,
                                              v_scale)
    out = torch.full((B, H, D), float("nan"), dtype=torch.float64)
    seqs = range(B) if seqs is None else seqs
    heads = range(H) if heads is None else heads
    for s in seqs:
        L = int(seq_lens[s])
        ids = sequence_block_ids(block_tables, s, (L + bs - 1) // bs, kv_indptr)
        cache = {}
        for h in heads:
            kvh = kv_head_of(h, H, Hk)
            if kvh not in cache:
                cache[kvh] = gather_kv(key_cache, value_cache, ids, L, kvh, **kvq)
            K, V = cache[kvh]
            bias = None if alibi_slopes is None else alibi_bias(float(alibi_slopes[h]), L)
            out[s, h], _ = attention_one_head(query[s, h], K, V, scale, bias)
    return out


def split_chunk_size(seq_len: int, num_splits: int, block_size: int) -> int:
    """Tokens per partition when a sequence is cut into ``num_splits`` pieces.

    sglang's ``get_num_kv_splits_triton`` gives only the count.  Reading: the
    chunk is ``cdiv(seq_len, num_splits)`` rounded up to a whole block, so
    every partition starts on a block boundary; at most ``num_splits``
    partitions are non-empty.
    """
    if seq_len <= 0 or num_splits <= 0:
        return block_size
    c = -(-seq_len // num_splits)
    return -(-c // block_size) * block_size


def partition_ranges(seq_len: int, max_num_partitions: int, block_size: int,
                     partition_size: Optional[int] = None,
                     num_splits: Optional[int] = None):
    """``[(start, end)]`` of every partition slot; empty slots have start >= end.

    Fixed mode: partition p covers ``[p*P, min((p+1)*P, seq_len))`` (page
    "paged_attention_v2_triton.py", ``_paged_attn_v2_partition_kernel``:
    part_start / part_end).  Split mode: the same with ``P`` replaced by
    ``split_chunk_size``.
    """
    if (partition_size is None) == (num_splits is None):
        raise ValueError("give exactly one of partition_size / num_splits")
    P = partition_size if partition_size is not None else split_chunk_size(seq_len, num_splits,
                                                                           block_size)
    out = []
    for p in range(max_num_partitions):
        a = p * P
        b = min(a + P, seq_len)
        if num_splits is not None and p >= num_splits:
            b = a  # beyond the requested split count: empty
        out.append((a, b))
    return out


def v2_partition(query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                 max_num_partitions: int, partition_size: Optional[int] = None,
                 num_kv_splits: Optional[Sequence[int]] = None,
                 seqs: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None,
                 kv_indptr: Optional[torch.Tensor] = None, kv_cache_dtype: str = "auto",
                 k_scale: float = 1.0, v_scale: float = 1.0,
                 alibi_slopes: Optional[Sequence[float]] = None):
    """Per-partition statistics of split-KV decode, all float64.

    Returns ``tmp_output [B, H, maxP, D]``, ``exp_sums [B, H, maxP]`` and
    ``max_logits [B, H, maxP]`` where, over the logits ``z`` of the partition's
    tokens: ``max_logits = max z``, ``exp_sums = sum exp(z - max)`` and
    ``tmp_output = sum exp(z - max) v / exp_sums`` (normalised: that is what
    the page's reduce weights assume).  Empty partitions hold ``-inf`` / ``0``
    and a NaN ``tmp_output`` row (the kernels leave it untouched).  The
    logits include the ALiBi term when ``alibi_slopes`` is given, and fp8
    caches are decoded as in ``decode_v1``.
    """
    B, H, D = query.shape
    Hk = key_cache.shape[1]
    bs = key_cache.shape[3]
    key_cache, value_cache, kvq = _kv_options(key_cache, value_cache, kv_cache_dtype, k_scale,
                                              v_scale)
    tmp = torch.full((B, H, max_num_partitions, D), float("nan"), dtype=torch.float64)
    es = torch.full((B, H, max_num_partitions), float("nan"), dtype=torch.float64)
    ml = torch.full((B, H, max_num_partitions), float("nan"), dtype=torch.float64)
    seqs = range(B) if seqs is None else seqs
    heads = range(H) if heads is None else heads
    for s in seqs:
        L = int(seq_lens[s])
        ranges = partition_ranges(
            L, max_num_partitions, bs, partition_size=partition_size,
            num_splits=None if num_kv_splits is None else int(num_kv_splits[s]))
        ids = sequence_block_ids(block_tables, s, (L + bs - 1) // bs, kv_indptr)
        cache = {}
        for h in heads:
            kvh = kv_head_of(h, H, Hk)
            if kvh not in cache:
                cache[kvh] = gather_kv(key_cache, value_cache, ids, L, kvh, **kvq)
            K, V = cache[kvh]
            z = (K @ query[s, h].to(torch.float64)) * scale if L else torch.zeros(0, dtype=torch.float64)
            if alibi_slopes is not None:
                z = z + alibi_bias(float(alibi_slopes[h]), L)
            for p, (a, b) in enumerate(ranges):
                if a >= b:
                    ml[s, h, p] = NEG_INF
                    es[s, h, p] = 0.0
                    continue
                zp = z[a:b]
                m = zp.max()
                e = torch.exp(zp - m)
                ml[s, h, p] = m
                es[s, h, p] = e.sum()
                tmp[s, h, p] = (e @ V[a:b]) / e.sum()
    return tmp, es, ml


def v2_reduce(tmp_output, exp_sums, max_logits, seq_lens, block_size: int,
              partition_size: Optional[int] = None, num_kv_splits: Optional[Sequence[int]] = None,
              seqs: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None):
    """Log-sum-exp combination of the partitions (page "paged_attention_v2_triton.py",
    ``_paged_attn_v2_reduce_kernel``).

    ``num_parts`` is the number of non-empty partitions (``cdiv(seq_len, P)``
    in fixed mode); ``M = max_p max_logits[p]``, ``w_p = exp(max_logits[p] - M)
    * exp_sums[p]``, ``out = sum_p w_p * tmp_output[p] / sum_p w_p``.  A
    sequence with no tokens gives a zero output.
    """
    B, H, maxP, D = tmp_output.shape
    out = torch.full((B, H, D), float("nan"), dtype=torch.float64)
    seqs = range(B) if seqs is None else seqs
    heads = range(H) if heads is None else heads
    for s in seqs:
        L = int(seq_lens[s])
        if partition_size is not None:
            num_parts = -(-L // partition_size)
        else:
            n = int(num_kv_splits[s])
            num_parts = -(-L // split_chunk_size(L, n, block_size)) if L > 0 else 0
        for h in heads:
            if num_parts == 0:
                out[s, h] = 0.0
                continue
            m = max_logits[s, h, :num_parts].to(torch.float64)
            l = exp_sums[s, h, :num_parts].to(torch.float64)
            M = m.max()
            w = torch.exp(m - M) * l
            w = w / w.sum()
            out[s, h] = w @ tmp_output[s, h, :num_parts].to(torch.float64)
    return out
