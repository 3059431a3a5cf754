"""Seeded synthetic inputs for paged-KV decode.

This module only draws random numbers and lays them out in the paged cache
format; it holds none of the attention or metadata arithmetic.  Both the CUDA
path (through the ctypes binding) and the CPU oracle consume exactly the bytes
produced here.

Cache layouts are the vLLM ones restated on the page "paged_attention_v2_triton.py"
(kernel argument comments of ``_paged_attn_v2_partition_kernel``):

* ``query``        ``[num_seqs, num_heads, head_size]``
* ``key_cache``    ``[num_blocks, num_kv_heads, head_size // x, block_size, x]``
  with ``x = 16 // element_size``
* ``value_cache``  ``[num_blocks, num_kv_heads, head_size, block_size]``
* ``block_tables`` ``[num_seqs, max_blocks_per_seq]`` int32 (may be a strided view)
* ``seq_lens``     ``[num_seqs]`` int32

Named workloads (``WORKLOADS``) are the decode batches this library is
measured on; each is described by what it is and its sizes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import torch

__all__ = [
    "DTYPES",
    "WorkloadSpec",
    "WORKLOADS",
    "make_inputs",
    "make_workload",
    "x_pack",
]

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# Sentinels written into block-table entries that no sequence owns.  Any kernel
# that reads one would see an out-of-range block id.
UNUSED_ENTRY = -1
GAP_ENTRY = -7  # columns skipped by a strided (column-step) view


def x_pack(dtype: torch.dtype) -> int:
    """Elements per 16-byte group of the key cache's innermost dimension."""
    return 16 // torch.empty((), dtype=dtype).element_size()


# kv_cache_dtype names -> torch float8 type used to round the drawn values
FP8_TORCH = {"fp8": torch.float8_e4m3fn, "fp8_e4m3": torch.float8_e4m3fn,
             "fp8_e5m2": torch.float8_e5m2}


def alibi_slopes(num_heads: int) -> torch.Tensor:
    """Per-head ALiBi slopes 2^(-8 (h+1) / num_heads): the geometric sequence of
    "Train Short, Test Long" (Press et al.), used here only as an input."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / num_heads) for h in range(num_heads)],
                        dtype=torch.float32)


@dataclass
class WorkloadSpec:
    """Shape and value recipe of one synthetic decode batch."""

    name: str
    description: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: str
    seq_len_recipe: str  # "fixed", "uniform", "lognormal"
    seq_lens: Optional[List[int]] = None  # for "fixed"
    seq_len_lo: int = 1
    seq_len_hi: int = 1
    lognormal_median: float = 1024.0
    lognormal_sigma: float = 1.0
    num_blocks: Optional[int] = None  # None -> ceil(1.1 * blocks needed)
    first_row: Optional[List[int]] = None  # fixed block-table row for seq 0
    bt_col_step: int = 1  # >1: table allocated wider and read as [:, ::step]
    max_blocks_per_seq: Optional[int] = None  # None -> cdiv(max seq_len, block_size)
    peaky_fraction: float = 0.0  # fraction of (token, kv_head) key vectors scaled
    peaky_scale: float = 8.0
    mode: str = "v1"  # "v1", "v2_fixed", "v2_splits"
    partition_size: int = 512
    max_kv_splits: int = 16
    device_core_count: int = 148
    kv_cache_dtype: str = "auto"  # or "fp8_e4m3" / "fp8_e5m2": one-byte cache codes
    k_scale: float = 1.0
    v_scale: float = 1.0
    alibi: bool = False
    extra: Dict = field(default_factory=dict)


WORKLOADS: Dict[str, WorkloadSpec] = {
    "tiny_mha_fp32": WorkloadSpec(
        name="tiny_mha_fp32",
        description=("tiny MHA decode, fp32: 2 seqs, seq_lens {16, 13}, 4 heads = 4 kv heads, "
                     "head_size 64, block_size 8, 64 blocks; seq 0 block table [40, 30]"),
        num_seqs=2, num_heads=4, num_kv_heads=4, head_size=64, block_size=8, dtype="f32",
        seq_len_recipe="fixed", seq_lens=[16, 13], num_blocks=64, first_row=[40, 30],
        mode="v1",
    ),
    "mha_v1_fp16": WorkloadSpec(
        name="mha_v1_fp16",
        description=("MHA single-pass decode, fp16: 64 seqs, 32 heads = 32 kv heads, head_size 128, "
                     "block_size 16, seq_lens uniform in [512, 4096]"),
        num_seqs=64, num_heads=32, num_kv_heads=32, head_size=128, block_size=16, dtype="f16",
        seq_len_recipe="uniform", seq_len_lo=512, seq_len_hi=4096, mode="v1",
    ),
    "gqa_v1_bf16": WorkloadSpec(
        name="gqa_v1_bf16",
        description=("GQA single-pass decode, bf16: 256 seqs, 32 query heads / 8 kv heads, "
                     "head_size 128, block_size 16, seq_lens uniform in [128, 2048]"),
        num_seqs=256, num_heads=32, num_kv_heads=8, head_size=128, block_size=16, dtype="bf16",
        seq_len_recipe="uniform", seq_len_lo=128, seq_len_hi=2048, mode="v1",
    ),
    "gqa_v1_fp32": WorkloadSpec(
        name="gqa_v1_fp32",
        description=("GQA single-pass decode, fp32: the GQA batch (256 seqs, 32 query heads / 8 kv "
                     "heads, head_size 128, block_size 16, seq_lens uniform in [128, 2048]) with "
                     "fp32 queries, caches and output"),
        num_seqs=256, num_heads=32, num_kv_heads=8, head_size=128, block_size=16, dtype="f32",
        seq_len_recipe="uniform", seq_len_lo=128, seq_len_hi=2048, mode="v1",
    ),
    "long_v2_bf16": WorkloadSpec(
        name="long_v2_bf16",
        description=("long-context split-KV decode, bf16: 8 seqs of 16k..128k tokens, 64 query heads / "
                     "8 kv heads, head_size 128, block_size 16, partition 512, 1% of keys x8"),
        num_seqs=8, num_heads=64, num_kv_heads=8, head_size=128, block_size=16, dtype="bf16",
        seq_len_recipe="fixed",
        seq_lens=[k * 1024 for k in (16, 24, 32, 48, 64, 96, 112, 128)],
        peaky_fraction=0.01, peaky_scale=8.0, mode="v2_fixed", partition_size=512,
    ),
    "ragged_v2_bf16": WorkloadSpec(
        name="ragged_v2_bf16",
        description=("ragged serving batch + metadata, bf16: 512 seqs, log-normal seq_lens "
                     "(median 1024, sigma 1, clipped to [1, 32768]), 32 query heads / 8 kv heads, "
                     "head_size 128, block_size 16; int32 table [512, 2048] read as a stride-2 "
                     "column view; page_indices copy, num_kv_splits (max 16, 148 SMs), split-KV"),
        num_seqs=512, num_heads=32, num_kv_heads=8, head_size=128, block_size=16, dtype="bf16",
        seq_len_recipe="lognormal", lognormal_median=1024.0, lognormal_sigma=1.0,
        seq_len_lo=1, seq_len_hi=32768, bt_col_step=2, max_blocks_per_seq=2048,
        mode="v2_splits", max_kv_splits=16, device_core_count=148,
    ),
    "ragged_v2_fp8": WorkloadSpec(
        name="ragged_v2_fp8",
        description=("ragged serving batch + metadata over an fp8 E4M3 cache: the ragged bf16 "
                     "batch (512 seqs, log-normal seq_lens, 32 query heads / 8 kv heads, head_size "
                     "128, block_size 16, stride-2 table view, split-KV) with one-byte key/value "
                     "codes, bf16 queries and output, k_scale 0.5, v_scale 2"),
        num_seqs=512, num_heads=32, num_kv_heads=8, head_size=128, block_size=16, dtype="bf16",
        seq_len_recipe="lognormal", lognormal_median=1024.0, lognormal_sigma=1.0,
        seq_len_lo=1, seq_len_hi=32768, bt_col_step=2, max_blocks_per_seq=2048,
        mode="v2_splits", max_kv_splits=16, device_core_count=148,
        kv_cache_dtype="fp8_e4m3", k_scale=0.5, v_scale=2.0,
    ),
    "long_v2_fp8": WorkloadSpec(
        name="long_v2_fp8",
        description=("long-context split-KV decode over an fp8 E4M3 cache: 8 seqs of 16k..128k "
                     "tokens, 64 query heads / 8 kv heads, head_size 128, block_size 16, "
                     "partition 512, 1% of keys x8, bf16 queries and output, k_scale 0.5, "
                     "v_scale 2"),
        num_seqs=8, num_heads=64, num_kv_heads=8, head_size=128, block_size=16, dtype="bf16",
        seq_len_recipe="fixed",
        seq_lens=[k * 1024 for k in (16, 24, 32, 48, 64, 96, 112, 128)],
        peaky_fraction=0.01, peaky_scale=8.0, mode="v2_fixed", partition_size=512,
        kv_cache_dtype="fp8_e4m3", k_scale=0.5, v_scale=2.0,
    ),
    "mha_v1_alibi_fp16": WorkloadSpec(
        name="mha_v1_alibi_fp16",
        description=("MHA single-pass decode with ALiBi, fp16: the MHA batch (64 seqs, 32 heads = "
                     "32 kv heads, head_size 128, block_size 16, seq_lens uniform in [512, 4096]) "
                     "with slopes 2^(-8(h+1)/32)"),
        num_seqs=64, num_heads=32, num_kv_heads=32, head_size=128, block_size=16, dtype="f16",
        seq_len_recipe="uniform", seq_len_lo=512, seq_len_hi=4096, mode="v1", alibi=True,
    ),
}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1009 + stream)
    return g


def _draw_seq_lens(spec: WorkloadSpec, seed: int) -> List[int]:
    g = _gen(seed, 1, "cpu")
    if spec.seq_len_recipe == "fixed":
        return list(spec.seq_lens)
    if spec.seq_len_recipe == "uniform":
        t = torch.randint(spec.seq_len_lo, spec.seq_len_hi + 1, (spec.num_seqs,), generator=g)
        return [int(v) for v in t]
    if spec.seq_len_recipe == "lognormal":
        z = torch.randn(spec.num_seqs, generator=g, dtype=torch.float64)
        raw = torch.exp(math.log(spec.lognormal_median) + spec.lognormal_sigma * z)
        lens = torch.clamp(torch.round(raw), spec.seq_len_lo, spec.seq_len_hi)
        return [int(v) for v in lens]
    raise ValueError(spec.seq_len_recipe)


def make_inputs(
    *,
    num_heads: int,
    num_kv_heads: int,
    head_size: int,
    block_size: int,
    dtype: str,
    seq_lens: Sequence[int],
    num_blocks: Optional[int] = None,
    first_row: Optional[Sequence[int]] = None,
    bt_col_step: int = 1,
    max_blocks_per_seq: Optional[int] = None,
    peaky_fraction: float = 0.0,
    peaky_scale: float = 8.0,
    unused_slot_fill: Optional[float] = None,
    seed: int = 0,
    device="cpu",
    kv_cache_dtype: str = "auto",
    k_scale: float = 1.0,
    v_scale: float = 1.0,
    alibi: bool = False,
) -> Dict:
    """Draw one paged decode batch.

    * query, key_cache and value_cache entries are N(0, 1) drawn in float32 and
      rounded once to ``dtype``.
    * Every sequence gets ``cdiv(seq_len, block_size)`` distinct physical
      blocks; no block is shared between sequences.  Block ids are a seeded
      random permutation of ``range(num_blocks)``, except that ``first_row``
      (when given) pins sequence 0's blocks and the others avoid them.
    * ``peaky_fraction``: each (block, slot, kv_head) key vector is multiplied
      by ``peaky_scale`` when a seeded uniform draw is below the fraction
      (applied in float32, before rounding to ``dtype``).
    * ``unused_slot_fill``: when set, cache slots that no sequence owns (and
      the tail slots of each sequence's last block) are overwritten with this
      value, e.g. NaN, to check that kernels never let them reach a result.
    * The block table is allocated ``[num_seqs, max_blocks_per_seq * bt_col_step]``
      and returned as the column view ``[:, ::bt_col_step]``; entries that no
      sequence owns hold -1, skipped columns hold -7.

    * ``kv_cache_dtype`` "fp8" / "fp8_e4m3" / "fp8_e5m2": the caches hold one-byte
      codes (uint8 tensors, ``x = 16``): the same float32 draws rounded once to
      that float8 format; ``k_scale`` / ``v_scale`` are returned for the
      consumer (the codes do not depend on them).
    * ``alibi``: also return ``alibi_slopes`` (float32 ``[num_heads]``).

    Random draws happen on ``device`` (a CUDA generator when it is a GPU) so
    multi-GB batches need no host-side generation; small batches default to
    the CPU.  Returned tensors live on ``device``.
    """
    dt = DTYPES[dtype]
    fp8 = FP8_TORCH.get(kv_cache_dtype)
    if kv_cache_dtype != "auto" and fp8 is None:
        raise ValueError(f"unknown kv_cache_dtype {kv_cache_dtype!r}")
    cache_dt = torch.uint8 if fp8 is not None else dt
    x = 16 if fp8 is not None else x_pack(dt)
    seq_lens = [int(v) for v in seq_lens]
    B = len(seq_lens)
    if head_size % x:
        raise ValueError("head_size must be a multiple of x")
    nblk = [(L + block_size - 1) // block_size for L in seq_lens]
    needed = sum(nblk)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(1.1 * needed))
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max([1] + nblk)
    if max(nblk + [0]) > max_blocks_per_seq:
        raise ValueError("a sequence needs more blocks than max_blocks_per_seq")

    # --- block tables (host side: small) ---
    g_tab = _gen(seed, 2, "cpu")
    perm = torch.randperm(num_blocks, generator=g_tab).tolist()
    rows: List[List[int]] = []
    if first_row is not None:
        if len(first_row) != nblk[0]:
            raise ValueError("first_row length must equal cdiv(seq_lens[0], block_size)")
        pinned = set(int(b) for b in first_row)
        pool = [b for b in perm if b not in pinned]
        rows.append([int(b) for b in first_row])
        start = 1
    else:
        pool = perm
        start = 0
    if needed - (nblk[0] if first_row is not None else 0) > len(pool):
        raise ValueError("num_blocks too small")
    off = 0
    for s in range(start, B):
        rows.append(pool[off:off + nblk[s]])
        off += nblk[s]
    full = torch.full((B, max_blocks_per_seq * bt_col_step), GAP_ENTRY, dtype=torch.int32)
    view = full[:, ::bt_col_step]
    view.fill_(UNUSED_ENTRY)
    for s in range(B):
        if nblk[s]:
            view[s, : nblk[s]] = torch.tensor(rows[s], dtype=torch.int32)
    full = full.to(device)
    block_tables = full[:, ::bt_col_step]

    # --- dense tensors, drawn on the target device ---
    Hk, D = num_kv_heads, head_size
    g_q = _gen(seed, 3, device)
    g_k = _gen(seed, 4, device)
    g_v = _gen(seed, 5, device)
    query = torch.randn((B, num_heads, D), generator=g_q, device=device, dtype=torch.float32).to(dt)
    key_cache = torch.empty((num_blocks, Hk, D // x, block_size, x), dtype=cache_dt, device=device)
    value_cache = torch.empty((num_blocks, Hk, D, block_size), dtype=cache_dt, device=device)

    def rounded(v):
        return v.to(dt) if fp8 is None else v.to(fp8).view(torch.uint8)

    # Draw block by block in slabs to bound float32 temporaries.
    slab = max(1, (1 << 26) // (Hk * D * block_size))
    g_p = _gen(seed, 6, device)
    for b0 in range(0, num_blocks, slab):
        b1 = min(num_blocks, b0 + slab)
        kk = torch.randn((b1 - b0, Hk, D // x, block_size, x), generator=g_k, device=device,
                         dtype=torch.float32)
        if peaky_fraction > 0.0:
            u = torch.rand((b1 - b0, Hk, 1, block_size, 1), generator=g_p, device=device,
                           dtype=torch.float32)
            kk = torch.where(u < peaky_fraction, kk * peaky_scale, kk)
        key_cache[b0:b1] = rounded(kk)
        vv = torch.randn((b1 - b0, Hk, D, block_size), generator=g_v, device=device,
                         dtype=torch.float32)
        value_cache[b0:b1] = rounded(vv)
        del kk, vv

    if unused_slot_fill is not None:
        owned = torch.zeros((num_blocks, block_size), dtype=torch.bool)
        for s in range(B):
            for j, b in enumerate(rows[s]):
                n = min(block_size, seq_lens[s] - j * block_size)
                owned[b, :n] = True
        owned = owned.to(device)
        kmask = (~owned).view(num_blocks, 1, 1, block_size, 1).expand_as(key_cache)
        vmask = (~owned).view(num_blocks, 1, 1, block_size).expand_as(value_cache)
        fill = unused_slot_fill
        if fp8 is not None:
            fill = int(torch.tensor([unused_slot_fill], dtype=torch.float32).to(fp8)
                       .view(torch.uint8)[0])
        key_cache[kmask] = fill
        value_cache[vmask] = fill

    seq_lens_t = torch.tensor(seq_lens, dtype=torch.int32, device=device)
    return {
        "query": query,
        "key_cache": key_cache,
        "value_cache": value_cache,
        "block_tables": block_tables,
        "block_tables_storage": full,
        "seq_lens": seq_lens_t,
        "seq_lens_list": seq_lens,
        "block_rows": rows,
        "num_blocks": num_blocks,
        "num_heads": num_heads,
        "num_kv_heads": num_kv_heads,
        "head_size": D,
        "block_size": block_size,
        "x": x,
        "dtype": dtype,
        "scale": 1.0 / math.sqrt(D),
        "max_blocks_per_seq": max_blocks_per_seq,
        "kv_cache_dtype": kv_cache_dtype,
        "k_scale": float(k_scale),
        "v_scale": float(v_scale),
        "alibi_slopes": alibi_slopes(num_heads).to(device) if alibi else None,
    }


def make_workload(name: str, seed: int = 0, device="cpu", **overrides) -> Dict:
    """Inputs of a named workload; ``overrides`` replace spec fields (e.g. ``num_seqs``)."""
    spec = WORKLOADS[name]
    if overrides:
        spec = WorkloadSpec(**{**spec.__dict__, **overrides})
    lens = _draw_seq_lens(spec, seed)[: spec.num_seqs]
    inp = make_inputs(
        num_heads=spec.num_heads,
        num_kv_heads=spec.num_kv_heads,
        head_size=spec.head_size,
        block_size=spec.block_size,
        dtype=spec.dtype,
        seq_lens=lens,
        num_blocks=spec.num_blocks,
        first_row=spec.first_row,
        bt_col_step=spec.bt_col_step,
        max_blocks_per_seq=spec.max_blocks_per_seq,
        peaky_fraction=spec.peaky_fraction,
        peaky_scale=spec.peaky_scale,
        seed=seed,
        device=device,
        kv_cache_dtype=spec.kv_cache_dtype,
        k_scale=spec.k_scale,
        v_scale=spec.v_scale,
        alibi=spec.alibi,
    )
    # cu_num_blocks: the indptr a serving engine hands to the page-index copy
    # (exclusive scan of each sequence's block count).
    nblk = [len(r) for r in inp["block_rows"]]
    cu = [0]
    for n in nblk:
        cu.append(cu[-1] + n)
    inp["cu_num_blocks"] = torch.tensor(cu, dtype=torch.int32, device=device)
    inp["spec"] = spec
    return inp


# ------------------------------------------------ fused decode metadata inputs --

METADATA_WORKLOADS = {
    "decode_metadata_ps1": dict(
        description=("fused decode metadata, page size 1, no sliding window: 512 requests "
                     "(log-normal lengths as the ragged batch), token pool [1024, 32768] int32, "
                     "max_seq_pages 32768, delta 1"),
        batch=512, pool_rows=1024, pool_cols=32768, page_size=1, max_seq_pages=32768, swa=False),
    "decode_metadata_ps16_swa": dict(
        description=("fused decode metadata, page size 16 with the sliding-window table: 512 "
                     "requests, token pool [1024, 32768] int32, max_seq_pages 2048, delta 1, "
                     "full-to-SWA mapping of 2^25 int64 entries"),
        batch=512, pool_rows=1024, pool_cols=32768, page_size=16, max_seq_pages=2048, swa=True),
}


def make_decode_metadata_inputs(name: str, seed: int = 0, device="cpu") -> Dict:
    """Token pool, request rows, lengths (and SWA mapping) for one metadata launch.

    ``req_to_token`` holds distinct token slot ids drawn as a seeded
    permutation; requests use distinct pool rows; lengths follow the ragged
    batch's log-normal recipe (clipped to the pool width).
    """
    cfg = METADATA_WORKLOADS[name]
    g = _gen(seed, 7, "cpu")
    B, rows, cols = cfg["batch"], cfg["pool_rows"], cfg["pool_cols"]
    spec = WORKLOADS["ragged_v2_bf16"]
    lens = _draw_seq_lens(WorkloadSpec(**{**spec.__dict__, "num_seqs": B,
                                          "seq_len_hi": cols - 1}), seed)
    gd = _gen(seed, 8, device)
    req_to_token = torch.randint(0, rows * cols, (rows, cols), generator=gd, device=device,
                                 dtype=torch.int32)
    pool = torch.randperm(rows, generator=g)[:B].to(torch.int64).to(device)
    out = {
        "req_to_token": req_to_token,
        "req_pool_indices": pool,
        "seq_lens": torch.tensor(lens, dtype=torch.int64, device=device),
        "page_size": cfg["page_size"],
        "max_seq_pages": cfg["max_seq_pages"],
        "seq_len_delta": 1,
        "description": cfg["description"],
        "full_to_swa_mapping": None,
    }
    if cfg["swa"]:
        out["full_to_swa_mapping"] = torch.randint(0, 1 << 30, (rows * cols,), generator=gd,
                                                   device=device, dtype=torch.int64)
    return out


SWA_SPEC_WORKLOADS = {
    "swa_spec_page_table": dict(
        description=("sliding-window speculative page table: 128 requests x 4 draft tokens, "
                     "table A [128, 4096] int32 (window pages), table B [512, 64] int32 "
                     "(draft pages), lengths uniform in [0, width]"),
        bs=128, draft_tokens=4, len_a=4096, len_b=64),
}


def make_swa_spec_inputs(name: str, seed: int = 0, device="cpu") -> Dict:
    """Tables A and B and their per-row lengths for one SWA speculative table launch."""
    cfg = SWA_SPEC_WORKLOADS[name]
    g = _gen(seed, 9, "cpu")
    bs, R, LA, LB = cfg["bs"], cfg["draft_tokens"], cfg["len_a"], cfg["len_b"]
    A = torch.randint(0, 1 << 30, (bs, LA), generator=g, dtype=torch.int32)
    B = torch.randint(0, 1 << 30, (bs * R, LB), generator=g, dtype=torch.int32)
    la = torch.randint(0, LA + 1, (bs,), generator=g, dtype=torch.int32)
    lb = torch.randint(0, LB + 1, (bs * R,), generator=g, dtype=torch.int32)
    return {"page_table_a": A.to(device), "page_table_b": B.to(device),
            "seq_len_a": la.to(device), "seq_len_b": lb.to(device), "num_draft_tokens": R,
            "description": cfg["description"]}
