"""GPU parity of the attention kernels against the float64 oracle, through
the C ABI, on small batches that span several pipeline chunks and partitions
and end in ragged tails; plus the edge cases of the method."""
import math

import pytest
import torch

import oracle
import paged_kv_decode_tables_gb300 as pkv
import workloads
from gpu_support import (assert_attention_close, assert_partials_close, on_device, run_v1,
                         run_v2, variant_kwargs, oracle_kwargs)

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


def _inputs(dtype, D, bs, H, Hk, lens, seed=0, **kw):
    return workloads.make_inputs(num_heads=H, num_kv_heads=Hk, head_size=D, block_size=bs,
                                 dtype=dtype, seq_lens=lens, seed=seed, **kw)


def _oracle_v1(inp, **kw):
    return oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                            inp["block_tables"], inp["seq_lens_list"], inp["scale"], **kw)


# ------------------------------------------------------- worked example ---

def test_worked_example_fp32_single_pass():
    inp = workloads.make_workload("tiny_mha_fp32")
    g = on_device(inp)
    out = run_v1(g)
    err = assert_attention_close(out, _oracle_v1(inp), torch.float32, "tiny fp32")
    assert err <= 1e-5


# ------------------------------------------------------- v1 parity grid ---

V1_CASES = [
    # dtype, D, bs, H, Hk
    ("bf16", 128, 16, 32, 8),
    ("bf16", 128, 16, 8, 1),
    ("bf16", 128, 16, 8, 8),
    ("bf16", 128, 8, 16, 4),
    ("bf16", 128, 32, 16, 2),
    ("bf16", 64, 16, 12, 4),
    ("bf16", 256, 16, 8, 2),
    ("f16", 128, 16, 32, 32),
    ("f16", 128, 8, 8, 4),
    ("f16", 64, 32, 6, 3),
    ("f16", 256, 8, 4, 1),
    ("f32", 64, 8, 4, 4),
    ("f32", 128, 16, 8, 1),
    ("f32", 64, 32, 6, 2),
    ("f32", 128, 8, 16, 8),
]


@pytest.mark.parametrize("warps", [1, 4])
@pytest.mark.parametrize("dtype,D,bs,H,Hk", V1_CASES)
def test_single_pass_parity(dtype, D, bs, H, Hk, warps):
    lens = [1, bs - 1, 16 * 5 + 3, 333, bs * 7, 1000]
    inp = _inputs(dtype, D, bs, H, Hk, lens, seed=D + bs + H)
    g = on_device(inp)
    pkv.set_attention_warps(warps)
    try:
        out = run_v1(g)
    finally:
        pkv.set_attention_warps(0)
    assert_attention_close(out, _oracle_v1(inp), DT[dtype], f"v1 {dtype} D{D} bs{bs} {H}/{Hk}")


def test_single_pass_peaky_keys_bf16():
    """1% of keys scaled x8: near one-hot softmax rows, outputs of order 1-3."""
    inp = _inputs("bf16", 128, 16, 64, 8, [4000, 1500, 777], seed=5, peaky_fraction=0.01)
    g = on_device(inp)
    assert_attention_close(run_v1(g), _oracle_v1(inp), torch.bfloat16, "peaky v1")


# ------------------------------------------------------------ split-KV ---

@pytest.mark.parametrize("dtype,D,bs,H,Hk", [("bf16", 128, 16, 64, 8), ("f16", 128, 16, 8, 8),
                                             ("bf16", 64, 8, 8, 2), ("f32", 128, 16, 8, 2),
                                             ("bf16", 256, 32, 4, 1)])
@pytest.mark.parametrize("P", [32, 64, 512])
def test_v2_fixed_partitions_parity(dtype, D, bs, H, Hk, P):
    if P % bs:
        pytest.skip("partition size must be a multiple of block_size")
    lens = [1, P - 1, P, P + 1, 3 * P + 17, 1100]
    inp = _inputs(dtype, D, bs, H, Hk, lens, seed=P + D, peaky_fraction=0.01)
    g = on_device(inp)
    maxP = -(-inp["max_blocks_per_seq"] * bs // P)
    tmp, es, ml, out = run_v2(g, maxP, partition_size=P)
    rtmp, res, rml = oracle.v2_partition(inp["query"], inp["key_cache"], inp["value_cache"],
                                         inp["block_tables"], lens, inp["scale"], maxP,
                                         partition_size=P)
    assert_partials_close(tmp, es, ml, rtmp, res, rml, f"v2 partials {dtype} P{P}")
    assert_attention_close(out, _oracle_v1(inp), DT[dtype], f"v2 {dtype} P{P}")


def test_v2_matches_single_pass_on_gpu():
    inp = _inputs("bf16", 128, 16, 32, 8, [2000, 513, 1], seed=9)
    g = on_device(inp)
    ref = _oracle_v1(inp)
    assert_attention_close(run_v1(g), ref, torch.bfloat16, "v1")
    for P in (16, 128, 512, 2048):
        maxP = -(-inp["max_blocks_per_seq"] * 16 // P)
        _, _, _, v2 = run_v2(g, maxP, partition_size=P)
        assert_attention_close(v2, ref, torch.bfloat16, f"v2 P{P}")


def test_v2_with_split_counts_parity():
    lens = [5, 2047, 2048, 2049, 9000, 130, 64]
    inp = _inputs("bf16", 128, 16, 32, 8, lens, seed=11)
    g = on_device(inp)
    splits = torch.empty(len(lens), dtype=torch.int32, device="cuda")
    pkv.compute_num_kv_splits(splits, g["seq_lens"], num_group=1, num_head=32, num_kv_head=8,
                              max_kv_splits=16, device_core_count=148)
    want = oracle.num_kv_splits(lens, 1, 32, 8, 16, 148)
    assert splits.cpu().tolist() == want
    tmp, es, ml, out = run_v2(g, 16, splits=splits)
    rtmp, res, rml = oracle.v2_partition(inp["query"], inp["key_cache"], inp["value_cache"],
                                         inp["block_tables"], lens, inp["scale"], 16,
                                         num_kv_splits=want)
    assert_partials_close(tmp, es, ml, rtmp, res, rml, "split partials")
    assert_attention_close(out, _oracle_v1(inp), torch.bfloat16, "split-KV")


def test_reduce_alone_on_oracle_partials():
    """The reduce kernel fed with the oracle's partials (rounded to fp32)."""
    lens = [1, 700, 2500, 0]
    inp = _inputs("bf16", 128, 16, 8, 2, lens, seed=12)
    maxP = 6
    rtmp, res, rml = oracle.v2_partition(inp["query"], inp["key_cache"], inp["value_cache"],
                                         inp["block_tables"], lens, inp["scale"], maxP,
                                         partition_size=512)
    ref = oracle.v2_reduce(rtmp, res, rml, lens, 16, partition_size=512)
    tmp = torch.nan_to_num(rtmp, nan=12345.0).float().cuda()
    out = torch.empty(4, 8, 128, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_v2_reduce(out, tmp, res.float().cuda(), rml.float().cuda(),
                                  torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                  partition_size=512)
    assert_attention_close(out, ref, torch.bfloat16, "reduce")
    assert bool((out[3].float() == 0).all())


# ------------------------------------------------------------ invariants ---

def test_flat_page_list_equals_block_table_bitwise():
    lens = [100, 1, 555, 2048, 17]
    inp = _inputs("bf16", 128, 16, 32, 8, lens, seed=13, bt_col_step=2)
    g = on_device(inp)
    nblk = [len(r) for r in inp["block_rows"]]
    cu = torch.tensor([0] + torch.tensor(nblk).cumsum(0).tolist(), dtype=torch.int32,
                      device="cuda")
    flat = torch.empty(int(cu[-1]), dtype=torch.int32, device="cuda")
    pkv.copy_page_indices(flat, g["block_tables"], cu)
    a = run_v1(g)
    b = run_v1(g, block_tables=flat, kv_indptr=cu)
    assert torch.equal(a, b)
    _, _, _, c = run_v2(g, 8, partition_size=512)
    _, _, _, d = run_v2(g, 8, partition_size=512, block_tables=flat, kv_indptr=cu)
    assert torch.equal(c, d)


def test_block_relabelling_is_bitwise_invariant():
    lens = [1234, 77, 512]
    inp = _inputs("bf16", 128, 16, 16, 4, lens, seed=14)
    g = on_device(inp)
    base = run_v1(g)
    NB = inp["num_blocks"]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(3)).cuda()
    kc = torch.empty_like(g["key_cache"])
    vc = torch.empty_like(g["value_cache"])
    kc[perm] = g["key_cache"]
    vc[perm] = g["value_cache"]
    bt = g["block_tables"].clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    g2 = dict(g, key_cache=kc, value_cache=vc, block_tables=bt)
    assert torch.equal(base, run_v1(g2))


def test_gqa_heads_with_equal_queries_agree():
    inp = _inputs("bf16", 128, 16, 32, 4, [900, 33], seed=15)
    q = inp["query"].view(2, 4, 8, 128)
    q.copy_(q[:, :, :1, :].clone().expand_as(q))  # every head of a group: the group's first query
    g = on_device(inp)
    out = run_v1(g).view(2, 4, 8, 128)
    assert torch.equal(out, out[:, :, :1, :].expand_as(out))


def test_unused_cache_slots_never_reach_the_output():
    """NaN in every slot no sequence owns, including the tails of last pages."""
    lens = [3, 17, 250, 1025]
    inp = _inputs("bf16", 128, 16, 16, 4, lens, seed=16, unused_slot_fill=float("nan"))
    g = on_device(inp)
    ref = _oracle_v1(inp)
    for warps in (1, 4):
        pkv.set_attention_warps(warps)
        try:
            assert_attention_close(run_v1(g), ref, torch.bfloat16, f"NaN slots w{warps}")
            maxP = -(-inp["max_blocks_per_seq"] * 16 // 128)
            _, _, _, out = run_v2(g, maxP, partition_size=128)
            assert_attention_close(out, ref, torch.bfloat16, f"NaN slots v2 w{warps}")
        finally:
            pkv.set_attention_warps(0)
    inp32 = _inputs("f32", 64, 8, 4, 2, lens, seed=17, unused_slot_fill=float("nan"))
    assert_attention_close(run_v1(on_device(inp32)), _oracle_v1(inp32), torch.float32, "NaN f32")


@pytest.mark.parametrize("D,bs", [(64, 16), (128, 8), (128, 32)])
def test_fp32_long_sequences_keep_the_fp32_bound(D, bs):
    """fp32 on the tf32 tensor path: one warp walks a whole long sequence (up
    to 9000 tokens, 1 % of keys x8), so the running sums take hundreds of
    chunks; the output stays within the 1e-5 fp32 bound, single pass and
    split-KV."""
    lens = [597, 4099, 9000, 33]
    inp = _inputs("f32", D, bs, 8, 2, lens, seed=23, peaky_fraction=0.01, peaky_scale=8.0)
    g = on_device(inp)
    ref = _oracle_v1(inp)
    pkv.set_attention_warps(1)
    try:
        assert_attention_close(run_v1(g), ref, torch.float32, f"fp32 long D{D} bs{bs} v1")
        maxP = -(-inp["max_blocks_per_seq"] * bs // 4096)
        _, _, _, out = run_v2(g, maxP, partition_size=4096)
        assert_attention_close(out, ref, torch.float32, f"fp32 long D{D} bs{bs} v2")
    finally:
        pkv.set_attention_warps(0)


def test_zero_length_sequences():
    lens = [0, 5, 0, 300]
    inp = _inputs("bf16", 128, 16, 8, 2, lens, seed=18)
    g = on_device(inp)
    out = run_v1(g)
    assert bool((out[0] == 0).all()) and bool((out[2] == 0).all())
    _, es, ml, out2 = run_v2(g, 4, partition_size=128)
    assert bool((out2[0] == 0).all()) and bool((es[0] == 0).all())
    assert bool((ml[0] == -math.inf).all())
    ref = _oracle_v1(inp)
    assert_attention_close(out, ref, torch.bfloat16, "zero-len v1")
    assert_attention_close(out2, ref, torch.bfloat16, "zero-len v2")


def test_single_token_returns_value_row():
    inp = _inputs("bf16", 128, 16, 8, 8, [1, 1], seed=19)
    g = on_device(inp)
    out = run_v1(g)
    for s in range(2):
        blk = inp["block_rows"][s][0]
        v0 = inp["value_cache"][blk, :, :, 0]  # [Hk, D]
        assert torch.equal(out[s].cpu(), v0)


def test_non_default_stream_and_strided_query():
    inp = _inputs("f16", 128, 16, 16, 4, [600, 31], seed=20)
    g = on_device(inp)
    wide = torch.zeros(2, 16, 256, dtype=torch.float16, device="cuda")
    wide[:, :, :128] = g["query"]
    g["query"] = wide[:, :, :128]
    out_wide = torch.zeros(2, 16, 256, dtype=torch.float16, device="cuda")
    out = out_wide[:, :, 64:192]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.paged_attention_decode(out, g["query"], g["key_cache"], g["value_cache"],
                                   g["block_tables"], g["seq_lens"], g["scale"])
    s.synchronize()
    assert_attention_close(out, _oracle_v1(inp), torch.float16, "strided")
    assert bool((out_wide[:, :, :64] == 0).all()) and bool((out_wide[:, :, 192:] == 0).all())


# ------------------------------------------------------------ error flags ---

def test_bad_device_data_sets_flags_without_faulting():
    lens = [40, 300]
    inp = _inputs("bf16", 128, 16, 8, 2, lens, seed=21)
    g = on_device(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = g["block_tables"].clone()
    bt[1, 3] = inp["num_blocks"] + 100  # out-of-range block id
    run_v1(g, err=err, block_tables=bt)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_BLOCK_ID
    err.zero_()
    g2 = dict(g, seq_lens=torch.tensor([40, 10 ** 6], dtype=torch.int32, device="cuda"))
    run_v1(g2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_SEQ_LEN
    err.zero_()
    splits = torch.tensor([0, 99], dtype=torch.int32, device="cuda")
    run_v2(g, 4, splits=splits, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_SPLITS
    # the context is still usable
    assert_attention_close(run_v1(g), _oracle_v1(inp), torch.bfloat16, "after errors")


def _check_longest_first(order, lens):
    o = order.cpu().tolist()
    assert sorted(o) == list(range(len(lens))), "not a permutation"
    ml = max(max(lens), 0)
    buckets = [(ml - max(lens[i], 0)) * 256 // (ml + 1) for i in o]
    assert buckets == sorted(buckets), "buckets out of order"


def test_longest_first_order_and_decode_in_that_order():
    """pkv_order_by_length gives a permutation whose length buckets never
    decrease (the order within a bucket is not fixed); decoding in that order
    gives bit-identical outputs; an entry out of range sets PKV_ERRF_ORDER."""
    lens = [5, 1200, 0, 333, 1200, 17, 64, 900, 1, 2048]
    inp = _inputs("bf16", 128, 16, 16, 4, lens, seed=41)
    g = on_device(inp)
    order = torch.empty(len(lens), dtype=torch.int32, device="cuda")
    pkv.order_by_length(order, g["seq_lens"])
    torch.cuda.synchronize()
    _check_longest_first(order, lens)
    ref = run_v1(g)
    out = torch.empty_like(g["query"])
    pkv.paged_attention_decode(out, g["query"], g["key_cache"], g["value_cache"],
                               g["block_tables"], g["seq_lens"], g["scale"], seq_order=order,
                               **variant_kwargs(g))
    assert torch.equal(out, ref)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = order.clone()
    bad[3] = len(lens) + 5
    pkv.paged_attention_decode(out, g["query"], g["key_cache"], g["value_cache"],
                               g["block_tables"], g["seq_lens"], g["scale"], seq_order=bad,
                               err_flag=err, **variant_kwargs(g))
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_ORDER
    # many sequences per thread of the ordering CTA, ties and negative lengths
    gen = torch.Generator().manual_seed(43)
    big = torch.randint(-3, 5000, (3000,), generator=gen, dtype=torch.int32)
    big[:500] = 777
    order = torch.empty(3000, dtype=torch.int32, device="cuda")
    pkv.order_by_length(order, big.cuda())
    torch.cuda.synchronize()
    _check_longest_first(order, big.tolist())


def test_copy_wait_timeout_is_reported_and_the_context_survives():
    """Failure detection without a fault: with the test hook every stage
    expects 16 bytes that never arrive, so each bounded wait runs out (20 ms
    here); the kernel reports PKV_ERRF_TIMEOUT and finishes, and the next
    launches in the same context are correct."""
    cases = [("bf16", 128, 16, 4, 1, [64]), ("f32", 64, 8, 4, 4, [16, 13])]
    for dtype, D, bs, H, Hk, lens in cases:
        inp = _inputs(dtype, D, bs, H, Hk, lens, seed=50)
        g = on_device(inp)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.set_wait_limit_ns(20_000_000)
        pkv._test_set_unarrived_bytes(16)
        try:
            run_v1(g, err=err)
            torch.cuda.synchronize()
        finally:
            pkv._test_set_unarrived_bytes(0)
            pkv.set_wait_limit_ns(0)
        assert int(err.item()) & pkv.PKV_ERRF_TIMEOUT, dtype
        err.zero_()
        out = run_v1(g, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attention_close(out, _oracle_v1(inp), DT[dtype], f"after timeout {dtype}")


def test_fp8_split_fold_stops_after_a_copy_timeout():
    """Two partitions per CTA (fp8 cache, split-KV, halved grid forced): when
    the first partition's copy waits run out (test hook, 20 ms limit) the
    CTA reports PKV_ERRF_TIMEOUT and does not start its second partition on
    the ring whose barriers still expect bytes; the next launches in the same
    context are correct."""
    lens = [700, 900]
    inp = _inputs("bf16", 128, 16, 4, 1, lens, seed=51, kv_cache_dtype="fp8_e4m3", k_scale=0.5,
                  v_scale=2.0)
    g = on_device(inp)
    splits = torch.full((len(lens),), 4, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_attention_warps(2)  # the fold exists on two-warp CTAs; small batches pick four
    pkv.set_split_fold(2)
    try:
        pkv.set_wait_limit_ns(20_000_000)
        pkv._test_set_unarrived_bytes(16)
        try:
            run_v2(g, 4, splits=splits, err=err)
            torch.cuda.synchronize()
        finally:
            pkv._test_set_unarrived_bytes(0)
            pkv.set_wait_limit_ns(0)
        assert int(err.item()) & pkv.PKV_ERRF_TIMEOUT
        err.zero_()
        _, _, _, out = run_v2(g, 4, splits=splits, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    finally:
        pkv.set_split_fold(1)
        pkv.set_attention_warps(0)
    assert_attention_close(out, _oracle_v1(inp, **oracle_kwargs(inp)), torch.bfloat16,
                           "after a timeout, two partitions per CTA")


@pytest.mark.parametrize("dtype,kv,alibi", [("f32", "auto", False), ("bf16", "auto", True),
                                             ("f16", "fp8_e4m3", False), ("bf16", "fp8_e5m2", True)])
def test_column_pair_and_full_forms_agree(dtype, kv, alibi):
    """A group of 4 query heads runs the column-pair kernel, a group of 8 the
    full one: the same 4 queries duplicated into a group of 8 must give the
    same outputs and partials for heads 0-3 up to rounding (one ulp of the
    output type; fp32 4e-6)."""
    lens = [1000, 37, 2500, 1]
    inp = _inputs(dtype, 128, 16, 8, 2, lens, seed=31, kv_cache_dtype=kv, k_scale=0.5,
                  v_scale=2.0, alibi=alibi)
    g4 = on_device(inp)
    sel = torch.tensor([k * 8 + j for k in range(2) for j in range(4)], device="cuda")
    src = torch.tensor([k * 4 + j % 4 for k in range(2) for j in range(8)], device="cuda")
    g8 = dict(g4)
    g8["query"] = g4["query"].index_select(1, src).contiguous()
    g8["num_heads"] = 16
    if alibi:
        g8["alibi_slopes"] = g4["alibi_slopes"].index_select(0, src).contiguous()
    o4 = run_v1(g4).double()
    o8 = run_v1(g8).index_select(1, sel).double()
    if dtype == "f32":
        tol = torch.full_like(o4, 4e-6)
    else:
        m = {"f16": 10, "bf16": 7}[dtype]
        tol = torch.pow(2.0, torch.floor(torch.log2(o4.abs().clamp_min(1e-30))) - m) + 1e-6
    diff = (o4 - o8).abs()
    assert bool((diff <= tol).all()), f"{dtype}/{kv}: max diff {float(diff.max()):.3e}"
    maxP = -(-inp["max_blocks_per_seq"] * 16 // 512)
    t4, e4, m4, _ = run_v2(g4, maxP, partition_size=512)
    t8, e8, m8, _ = run_v2(g8, maxP, partition_size=512)
    t8, e8, m8 = (x.index_select(1, sel) for x in (t8, e8, m8))
    live = e4 > 0
    assert torch.equal(live, e8 > 0)
    assert bool(((t4 - t8).abs()[live] <= 1e-5 * (1 + t4.abs()[live])).all())
    assert bool(((e4 - e8).abs()[live] <= 1e-5 * e4.abs()[live]).all())
    assert bool(((m4 - m8).abs()[live] <= 1e-5 * (1 + m4.abs()[live])).all())


@pytest.mark.parametrize("dtype,D,bs,H,Hk", [("bf16", 128, 16, 16, 1), ("bf16", 128, 16, 128, 8),
                                             ("f16", 64, 8, 18, 2), ("bf16", 256, 32, 64, 2),
                                             ("f32", 64, 16, 32, 1), ("bf16", 128, 16, 64, 1)])
def test_groups_larger_than_eight(dtype, D, bs, H, Hk):
    """A kv head serving 9..64 query heads (sub-groups of 8 per CTA): single
    pass, fixed partitions and split counts all match the oracle."""
    lens = [1, 300, 1025, 17]
    inp = _inputs(dtype, D, bs, H, Hk, lens, seed=H + Hk + D, peaky_fraction=0.01)
    g = on_device(inp)
    ref = _oracle_v1(inp)
    assert_attention_close(run_v1(g), ref, DT[dtype], f"v1 {H}/{Hk}")
    maxP = -(-inp["max_blocks_per_seq"] * bs // 128)
    _, _, _, out = run_v2(g, maxP, partition_size=128)
    assert_attention_close(out, ref, DT[dtype], f"v2 fixed {H}/{Hk}")
    splits = torch.tensor([1, 2, 3, 1], dtype=torch.int32, device="cuda")
    _, _, _, out = run_v2(g, 4, splits=splits)
    assert_attention_close(out, ref, DT[dtype], f"v2 splits {H}/{Hk}")


def _same(a, b):
    return bool(((a == b) | (torch.isnan(a) & torch.isnan(b))).all())


@pytest.mark.parametrize("dtype,kv,D,bs,H,Hk,maxP", [
    ("f16", "fp8_e4m3", 128, 16, 32, 8, 16), ("bf16", "fp8_e4m3", 128, 16, 64, 8, 16),
    ("bf16", "fp8_e5m2", 64, 8, 16, 4, 9), ("f16", "fp8_e4m3", 256, 16, 72, 4, 5),
    ("bf16", "fp8_e4m3", 128, 16, 8, 8, 2), ("bf16", "fp8_e4m3", 128, 16, 32, 8, 40)])
def test_split_fold_is_bitwise_identical(dtype, kv, D, bs, H, Hk, maxP):
    """Split-KV over an fp8 cache with half the partition slots (a CTA runs
    partitions x and x + slots of its sequence) gives bit-identical partials,
    statistics and outputs to one CTA per slot, for even and odd
    max_num_partitions, head groups of 1 to 18 and zero-length sequences;
    every (sequence, partition) row of the statistics is written."""
    rng = torch.Generator().manual_seed(43)
    lens = [int(x) for x in torch.randint(1, 3000, (40,), generator=rng)]
    lens[:6] = [0, 1, 16, 17, 4096, 0]
    inp = _inputs(dtype, D, bs, H, Hk, lens, seed=43, kv_cache_dtype=kv, k_scale=0.5,
                  v_scale=2.0)
    g = on_device(inp)
    splits = torch.empty(len(lens), dtype=torch.int32, device="cuda")
    pkv.compute_num_kv_splits(splits, g["seq_lens"], num_group=1, num_head=H, num_kv_head=Hk,
                              max_kv_splits=maxP, device_core_count=148)
    s = splits.cpu()
    s[2] = maxP  # as many splits as slots on 17 tokens: some of them empty
    s[4] = maxP - 1 if maxP > 1 else 1
    splits = s.to("cuda")
    pkv.set_attention_warps(2)  # the fold exists on two-warp CTAs; small batches pick four
    try:
        pkv.set_split_fold(0)
        full = run_v2(g, maxP, splits=splits)
        pkv.set_split_fold(2)  # halved grid whatever the batch size
        folded = run_v2(g, maxP, splits=splits)
    finally:
        pkv.set_split_fold(1)
        pkv.set_attention_warps(0)
    for a, b, what in zip(full, folded, ("tmp_out", "exp_sums", "max_logits", "output")):
        assert _same(a, b), f"{what} differs between one and two partitions per CTA"
    tmp, es, ml, _ = folded
    assert not bool(torch.isnan(es).any()) and not bool(torch.isnan(ml).any())
    n = 8  # the oracle on the first sequences (zero lengths and full split counts among them)
    rtmp, res, rml = oracle.v2_partition(inp["query"][:n], inp["key_cache"], inp["value_cache"],
                                         inp["block_tables"][:n], lens[:n], inp["scale"], maxP,
                                         num_kv_splits=s.tolist()[:n], **oracle_kwargs(inp))
    assert_partials_close(tmp[:n], es[:n], ml[:n], rtmp, res, rml, "two partitions per CTA")
