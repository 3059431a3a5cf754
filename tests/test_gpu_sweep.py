"""Randomised and extreme-size GPU parity against the float64 oracle.

* A seeded sweep over dtype, head size, block size, GQA group, single pass /
  fixed partitions / split counts, strided query and output views, column-step
  block tables and warps per CTA.
* A cache of about 10 GB per tensor whose last blocks hold a sequence, so that
  element offsets pass 2^32 (64-bit address arithmetic in the bulk copies).
* One 128k-token sequence decoded in a single pass.
"""
import random

import pytest
import torch

import bench
import oracle
import paged_kv_decode_tables_gb300 as pkv
import workloads
from gpu_support import assert_attention_close, on_device

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_decode_tables_gb300 import _build
    _build.build()
    yield
    pkv.set_attention_warps(0)


def _strided_like(t, rng):
    """A view with the same shape as ``t`` but a padded innermost stride."""
    pad = rng.choice([0, 8, 24])
    B, H, D = t.shape
    store = torch.zeros(B, H, D + pad, dtype=t.dtype, device=t.device)
    v = store[:, :, :D]
    v.copy_(t)
    return v


CASES = 48


@pytest.mark.parametrize("case", range(CASES))
def test_random_configuration(case):
    rng = random.Random(1000 + case)
    dtype = rng.choice(["f16", "bf16", "f32"])
    D = rng.choice([64, 128] if dtype == "f32" else [64, 128, 256])
    bs = rng.choice([8, 16, 32])
    Hk = rng.choice([1, 2, 4])
    g = rng.choice([1, 2, 3, 4, 5, 8])
    B = rng.randint(1, 6)
    lens = [rng.choice([0, 1, bs, 16, 2 * bs + 1, rng.randint(1, 700)]) for _ in range(B)]
    if max(lens) == 0:
        lens[0] = 5
    mode = rng.choice(["v1", "fixed", "splits"])
    warps = rng.choice([0, 1, 2, 4])
    inp = workloads.make_inputs(num_heads=Hk * g, num_kv_heads=Hk, head_size=D, block_size=bs,
                                dtype=dtype, seq_lens=lens, seed=case,
                                bt_col_step=rng.choice([1, 2]), peaky_fraction=0.01)
    gd = on_device(inp)
    q = _strided_like(gd["query"], rng)
    out_ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                               inp["block_tables"], lens, inp["scale"])
    out = _strided_like(torch.zeros_like(gd["query"]), rng)
    pkv.set_attention_warps(warps)
    try:
        if mode == "v1":
            pkv.paged_attention_decode(out, q, gd["key_cache"], gd["value_cache"],
                                       gd["block_tables"], gd["seq_lens"], inp["scale"])
        else:
            Bq, H, _ = q.shape
            cap = inp["max_blocks_per_seq"] * bs
            if mode == "fixed":
                P = bs * rng.choice([1, 2, 4, 32])
                maxP = -(-cap // P)
                splits = None
            else:
                P = 512
                maxP = rng.randint(1, 12)
                splits = torch.tensor([rng.randint(1, maxP) for _ in range(B)], dtype=torch.int32,
                                      device="cuda")
            tmp = torch.empty(Bq, H, maxP, D, dtype=torch.float32, device="cuda")
            es = torch.empty(Bq, H, maxP, dtype=torch.float32, device="cuda")
            ml = torch.empty(Bq, H, maxP, dtype=torch.float32, device="cuda")
            pkv.paged_attention_v2_partition(tmp, es, ml, q, gd["key_cache"], gd["value_cache"],
                                             gd["block_tables"], gd["seq_lens"], inp["scale"],
                                             partition_size=P, num_kv_splits=splits)
            pkv.paged_attention_v2_reduce(out, tmp, es, ml, gd["seq_lens"], partition_size=P,
                                          num_kv_splits=splits, block_size=bs)
    finally:
        pkv.set_attention_warps(0)
    torch.cuda.synchronize()
    assert_attention_close(out, out_ref, DT[dtype],
                           f"case {case}: {dtype} D{D} bs{bs} {Hk}x{g} {mode} w{warps} {lens}")


# 40 seeds, plus two that once exposed fp32 rounding growing with the length
# of a warp's sequential accumulation (one warp, 800-token sequences).
VARIANT_CASES = list(range(40)) + [179, 228]


@pytest.mark.parametrize("case", VARIANT_CASES)
def test_random_variant_configuration(case):
    """Seeded sweep over the cache format (16-bit, E4M3, E5M2), ALiBi, GQA
    groups up to 16 (sub-groups), single pass / fixed partitions / split
    counts, block tables given as a strided 2-D table or as a flat page list
    with an indptr, strided query/output views and warps per CTA."""
    rng = random.Random(5000 + case)
    dtype = rng.choice(["f16", "bf16", "bf16", "f32"])
    kv = "auto" if dtype == "f32" else rng.choice(["auto", "fp8_e4m3", "fp8_e5m2"])
    D = rng.choice([64, 128] if dtype == "f32" else [64, 128, 256])
    bs = rng.choice([8, 16, 32])
    Hk = rng.choice([1, 2])
    g = rng.choice([1, 2, 4, 6, 8, 12, 16])
    B = rng.randint(1, 5)
    lens = [rng.choice([0, 1, bs, 2 * bs + 1, rng.randint(1, 900)]) for _ in range(B)]
    if max(lens) == 0:
        lens[0] = 7
    alibi = rng.random() < 0.5
    mode = rng.choice(["v1", "fixed", "splits"])
    warps = rng.choice([0, 1, 2, 4])
    csr = rng.random() < 0.5
    inp = workloads.make_inputs(num_heads=Hk * g, num_kv_heads=Hk, head_size=D, block_size=bs,
                                dtype=dtype, seq_lens=lens, seed=700 + case,
                                bt_col_step=rng.choice([1, 2]), peaky_fraction=0.01,
                                kv_cache_dtype=kv, k_scale=rng.choice([0.5, 1.0, 1.75]),
                                v_scale=rng.choice([0.25, 1.0, 3.0]), alibi=alibi)
    gd = on_device(inp)
    kw = dict(kv_cache_dtype=kv, k_scale=inp["k_scale"], v_scale=inp["v_scale"],
              alibi_slopes=gd["alibi_slopes"])
    okw = dict(kw, alibi_slopes=None if not alibi else [float(v) for v in inp["alibi_slopes"]])
    out_ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                               inp["block_tables"], lens, inp["scale"], **okw)
    if csr:
        flat = [b for r in inp["block_rows"] for b in r] or [0]
        cu = [0]
        for r in inp["block_rows"]:
            cu.append(cu[-1] + len(r))
        table = torch.tensor(flat, dtype=torch.int32, device="cuda")
        indptr = torch.tensor(cu, dtype=torch.int32, device="cuda")
    else:
        table, indptr = gd["block_tables"], None
    q = _strided_like(gd["query"], rng)
    out = _strided_like(torch.zeros_like(gd["query"]), rng)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_attention_warps(warps)
    try:
        if mode == "v1":
            pkv.paged_attention_decode(out, q, gd["key_cache"], gd["value_cache"], table,
                                       gd["seq_lens"], inp["scale"], kv_indptr=indptr,
                                       err_flag=err, **kw)
        else:
            Bq, H, _ = q.shape
            cap = inp["max_blocks_per_seq"] * bs
            if mode == "fixed":
                P = bs * rng.choice([1, 2, 4, 32])
                maxP = -(-cap // P)
                splits = None
            else:
                P = 512
                maxP = rng.randint(1, 12)
                splits = torch.tensor([rng.randint(1, maxP) for _ in range(B)], dtype=torch.int32,
                                      device="cuda")
            tmp = torch.empty(Bq, H, maxP, D, dtype=torch.float32, device="cuda")
            es = torch.empty(Bq, H, maxP, dtype=torch.float32, device="cuda")
            ml = torch.empty(Bq, H, maxP, dtype=torch.float32, device="cuda")
            pkv.paged_attention_v2_partition(tmp, es, ml, q, gd["key_cache"], gd["value_cache"],
                                             table, gd["seq_lens"], inp["scale"],
                                             partition_size=P, num_kv_splits=splits,
                                             kv_indptr=indptr, err_flag=err,
                                             max_blocks_per_seq=inp["max_blocks_per_seq"],
                                             **kw)
            pkv.paged_attention_v2_reduce(out, tmp, es, ml, gd["seq_lens"], partition_size=P,
                                          num_kv_splits=splits, block_size=bs, err_flag=err)
    finally:
        pkv.set_attention_warps(0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, out_ref, DT[dtype],
                           f"variant case {case}: {dtype}/{kv} D{D} bs{bs} {Hk}x{g} alibi={alibi} "
                           f"{mode} csr={csr} w{warps} {lens}")


@pytest.mark.parametrize("kv,NB", [("auto", 300_000), ("fp8_e4m3", 600_000)])
def test_offsets_beyond_four_gigabytes(kv, NB):
    """Sequence 0 lives in the last blocks of a cache whose byte offsets exceed
    2^32 (bf16: 300,000 blocks, 9.8 GB per tensor; fp8: 600,000 blocks,
    9.8 GB of one-byte codes per tensor)."""
    Hk, D, bs = 8, 128, 16
    lens = [64, 100, 37]
    last = list(range(NB - 4, NB))
    inp = workloads.make_inputs(num_heads=32, num_kv_heads=Hk, head_size=D, block_size=bs,
                                dtype="bf16", seq_lens=lens, num_blocks=NB, first_row=last[::-1],
                                seed=7, device="cuda", kv_cache_dtype=kv, k_scale=0.5,
                                v_scale=2.0)
    elem = inp["key_cache"].element_size()
    assert int(inp["block_tables"][0].max()) * Hk * D * bs * elem > 2 ** 33
    out = torch.empty_like(inp["query"])
    pkv.paged_attention_decode(out, inp["query"], inp["key_cache"], inp["value_cache"],
                               inp["block_tables"], inp["seq_lens"], inp["scale"],
                               kv_cache_dtype=kv, k_scale=0.5, v_scale=2.0)
    torch.cuda.synchronize()
    q, kc, vc, bt, ls = bench.oracle_sample_inputs(inp, [0, 1, 2])
    ref = oracle.decode_v1(q, kc, vc, bt, ls, inp["scale"], kv_cache_dtype=kv, k_scale=0.5,
                           v_scale=2.0)
    assert_attention_close(out, ref, torch.bfloat16, f"offsets beyond 2^32 ({kv})")
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kv,alibi", [("auto", False), ("fp8_e5m2", True)])
def test_single_pass_128k_tokens(kv, alibi):
    lens = [131072]
    inp = workloads.make_inputs(num_heads=8, num_kv_heads=1, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=lens, seed=8, device="cuda",
                                peaky_fraction=0.01, kv_cache_dtype=kv, alibi=alibi)
    if alibi:
        inp["alibi_slopes"] = inp["alibi_slopes"] * 1e-4  # keep far tokens in play
    out = torch.empty_like(inp["query"])
    pkv.paged_attention_decode(out, inp["query"], inp["key_cache"], inp["value_cache"],
                               inp["block_tables"], inp["seq_lens"], inp["scale"],
                               kv_cache_dtype=kv, alibi_slopes=inp["alibi_slopes"])
    torch.cuda.synchronize()
    q, kc, vc, bt, ls = bench.oracle_sample_inputs(inp, [0])
    sl = None if not alibi else [float(v) for v in inp["alibi_slopes"].cpu()]
    ref = oracle.decode_v1(q, kc, vc, bt, ls, inp["scale"], kv_cache_dtype=kv, alibi_slopes=sl)
    assert_attention_close(out, ref, torch.bfloat16, f"128k single pass ({kv}, alibi={alibi})")
