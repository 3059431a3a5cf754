"""GPU parity of the tensor-memory kernel for fp8 caches (pkv_set_fp8_kernel(1):
persistent CTAs fed from the launch queue, both products as tcgen05
kind::f8f6f4 MMAs on the cache codes, accumulators in tensor memory) against
the float64 oracle, through the C ABI: single pass, fixed partitions (partials
compared too) and split counts; E4M3 and E5M2 codes; f16 and bf16 queries;
1 to 16 query heads per kv head; ALiBi; NaN codes in unowned slots; empty and
one-token sequences; peaky keys that move the running max (the accumulator
rescale in tensor memory); batches with many units and empty partitions (the
launch-queue takeover); bf16 queries far from 1 in magnitude; and the bounded
waits of the kernel's pipeline (a wait that runs out reports
PKV_ERRF_TIMEOUT and the context stays usable)."""
import pytest
import torch

import oracle
import paged_kv_decode_tables_gb300 as pkv
import workloads
from gpu_support import (assert_attention_close, assert_partials_close, on_device, oracle_kwargs,
                         run_v1, run_v2)

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _tensor_memory_kernel():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_decode_tables_gb300 import _build
    _build.build()
    pkv.set_attention_warps(0)
    pkv.set_fp8_kernel(1)
    yield
    pkv.set_fp8_kernel(0)


def _check_all_modes(inp, dtype, what, partition_size=128, max_splits=8):
    g = on_device(inp)
    kw = oracle_kwargs(inp)
    lens = inp["seq_lens_list"]
    ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                           inp["block_tables"], lens, inp["scale"], **kw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert_attention_close(run_v1(g, err=err), ref, DT[dtype], f"{what} v1")

    maxP = -(-inp["max_blocks_per_seq"] * 16 // partition_size)
    tmp, es, ml, out = run_v2(g, maxP, partition_size=partition_size, err=err)
    rtmp, res, rml = oracle.v2_partition(inp["query"], inp["key_cache"], inp["value_cache"],
                                         inp["block_tables"], lens, inp["scale"], maxP,
                                         partition_size=partition_size, **kw)
    assert_partials_close(tmp, es, ml, rtmp, res, rml, f"{what} partials")
    assert_attention_close(out, ref, DT[dtype], f"{what} v2 fixed")

    H, Hk = inp["num_heads"], inp["num_kv_heads"]
    splits = torch.empty(len(lens), dtype=torch.int32, device="cuda")
    pkv.compute_num_kv_splits(splits, g["seq_lens"], num_group=1, num_head=H, num_kv_head=Hk,
                              max_kv_splits=max_splits, device_core_count=148)
    _, _, _, out = run_v2(g, max_splits, splits=splits, err=err)
    assert_attention_close(out, ref, DT[dtype], f"{what} v2 splits")
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: error flag {int(err.item())}"


CASES = [
    # dtype, kv, H, Hk
    ("bf16", "fp8_e4m3", 32, 8),
    ("bf16", "fp8_e5m2", 8, 1),
    ("f16", "fp8_e4m3", 16, 4),
    ("f16", "fp8_e5m2", 12, 4),
    ("bf16", "fp8_e4m3", 64, 8),
    ("f16", "fp8_e4m3", 24, 3),
    ("bf16", "fp8_e5m2", 32, 2),   # 16 query heads per kv head: two sub-groups
    ("f16", "fp8_e4m3", 4, 4),
]


@pytest.mark.parametrize("alibi", [False, True])
@pytest.mark.parametrize("dtype,kv,H,Hk", CASES)
def test_tensor_memory_fp8_parity(dtype, kv, H, Hk, alibi):
    lens = [1, 15, 16 * 5 + 3, 333, 128, 129, 1000, 0]
    inp = workloads.make_inputs(num_heads=H, num_kv_heads=Hk, head_size=128, block_size=16,
                                dtype=dtype, seq_lens=lens, seed=H + Hk + int(alibi),
                                kv_cache_dtype=kv, k_scale=0.75, v_scale=1.5,
                                peaky_fraction=0.01, unused_slot_fill=float("nan"), alibi=alibi)
    _check_all_modes(inp, dtype, f"{dtype}/{kv} {H}/{Hk} alibi {alibi}")


def test_tensor_memory_many_units_and_empty_partitions():
    """A batch whose split-KV grid is mostly empty partitions, with more
    non-empty units than resident CTAs: every CTA takes over launches from the
    queue and retires the empty ones."""
    g_ = torch.Generator().manual_seed(11)
    lens = [int(x) for x in torch.randint(1, 3000, (96,), generator=g_)] + [0, 0, 40000]
    inp = workloads.make_inputs(num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=lens, seed=12, kv_cache_dtype="fp8_e4m3",
                                k_scale=0.5, v_scale=2.0)
    _check_all_modes(inp, "bf16", "many units", partition_size=256, max_splits=16)


@pytest.mark.parametrize("v_scale", [1.0, 64.0])
def test_tensor_memory_peaky_long_sequences(v_scale):
    """Long sequences with 5 % of keys x8: the running max keeps moving, so the
    output accumulator is rescaled in tensor memory; a large v_scale makes the
    probabilities' four-term encoding carry the precision."""
    inp = workloads.make_inputs(num_heads=64, num_kv_heads=8, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=[9000, 4097, 300], seed=13,
                                kv_cache_dtype="fp8_e4m3", k_scale=1.0, v_scale=v_scale,
                                peaky_fraction=0.05, peaky_scale=8.0)
    _check_all_modes(inp, "bf16", f"peaky v_scale {v_scale}", partition_size=512)


@pytest.mark.parametrize("shift", [-40, 40])
def test_tensor_memory_query_range(shift):
    """bf16 queries scaled by 2^shift with k_scale 2^-shift: the per-head power
    of two that puts the query's E4M3 terms in range is taken back out."""
    inp = workloads.make_inputs(num_heads=16, num_kv_heads=2, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=[700, 33, 129], seed=5,
                                kv_cache_dtype="fp8_e4m3", k_scale=2.0 ** -shift, v_scale=1.0)
    inp["query"] = (inp["query"].float() * 2.0 ** shift).to(torch.bfloat16)
    g = on_device(inp)
    ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                           inp["block_tables"], inp["seq_lens_list"], inp["scale"],
                           **oracle_kwargs(inp))
    assert_attention_close(run_v1(g), ref, torch.bfloat16, f"query x 2^{shift}")


def test_tensor_memory_wait_timeout_is_reported_and_the_context_survives():
    """With the test hook every key stage expects 16 bytes that never arrive;
    the pipeline's waits run out (20 ms), the kernel winds down, reports
    PKV_ERRF_TIMEOUT, frees its tensor memory, and the next launch is right."""
    inp = workloads.make_inputs(num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=[64, 300], seed=51,
                                kv_cache_dtype="fp8_e4m3", k_scale=0.5, v_scale=2.0)
    g = on_device(inp)
    ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                           inp["block_tables"], inp["seq_lens_list"], inp["scale"],
                           **oracle_kwargs(inp))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_wait_limit_ns(20_000_000)
    pkv._test_set_unarrived_bytes(16)
    try:
        run_v1(g, err=err)
        torch.cuda.synchronize()
    finally:
        pkv._test_set_unarrived_bytes(0)
        pkv.set_wait_limit_ns(0)
    assert int(err.item()) & pkv.PKV_ERRF_TIMEOUT
    err.zero_()
    out = run_v1(g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, torch.bfloat16, "after timeout")
