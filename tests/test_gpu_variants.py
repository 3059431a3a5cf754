"""GPU parity of the decode variants against the float64 oracle, through the
C ABI: fp8 KV caches (E4M3 / E5M2 codes with k_scale and v_scale) and ALiBi
logit biases, in the single pass, fixed partitions (partials compared too)
and split counts, for every warps-per-CTA instance; plus the f16 range
scaling that bf16 queries over an fp8 cache go through."""
import math

import pytest
import torch

import oracle
import paged_kv_decode_tables_gb300 as pkv
import workloads
from gpu_support import (assert_attention_close, assert_partials_close, on_device, oracle_kwargs,
                         run_v1, run_v2)

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


def _check_all_modes(inp, dtype, what, partition_size=128):
    """v1, fixed partitions (with partials) and split counts against the oracle."""
    g = on_device(inp)
    kw = oracle_kwargs(inp)
    lens = inp["seq_lens_list"]
    ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                           inp["block_tables"], lens, inp["scale"], **kw)
    assert_attention_close(run_v1(g), ref, DT[dtype], f"{what} v1")

    bs = inp["block_size"]
    maxP = -(-inp["max_blocks_per_seq"] * bs // partition_size)
    tmp, es, ml, out = run_v2(g, maxP, partition_size=partition_size)
    rtmp, res, rml = oracle.v2_partition(inp["query"], inp["key_cache"], inp["value_cache"],
                                         inp["block_tables"], lens, inp["scale"], maxP,
                                         partition_size=partition_size, **kw)
    assert_partials_close(tmp, es, ml, rtmp, res, rml, f"{what} partials")
    assert_attention_close(out, ref, DT[dtype], f"{what} v2 fixed")

    n = [1 + (7 * i) % 4 for i in range(len(lens))]
    splits = torch.tensor(n, dtype=torch.int32, device="cuda")
    _, _, _, out = run_v2(g, 4, splits=splits)
    assert_attention_close(out, ref, DT[dtype], f"{what} v2 splits")


# ---------------------------------------------------------- fp8 caches ---

FP8_CASES = [
    # query dtype, kv_cache_dtype, D, bs, H, Hk
    ("bf16", "fp8_e4m3", 128, 16, 32, 8),
    ("bf16", "fp8_e5m2", 128, 16, 8, 1),
    ("f16", "fp8_e4m3", 128, 8, 16, 4),
    ("f16", "fp8_e5m2", 64, 32, 12, 4),
    ("bf16", "fp8_e4m3", 256, 16, 8, 2),
    ("bf16", "fp8", 64, 8, 4, 4),
    ("f16", "fp8_e4m3", 256, 32, 16, 1),
    ("bf16", "fp8_e5m2", 128, 32, 6, 3),
]


@pytest.mark.parametrize("warps", [0, 1, 2, 4])
@pytest.mark.parametrize("dtype,kv,D,bs,H,Hk", FP8_CASES)
def test_fp8_cache_parity(dtype, kv, D, bs, H, Hk, warps):
    lens = [1, bs - 1, 16 * 5 + 3, 333, bs * 7, 1000]
    inp = workloads.make_inputs(num_heads=H, num_kv_heads=Hk, head_size=D, block_size=bs,
                                dtype=dtype, seq_lens=lens, seed=D + bs + H + Hk,
                                kv_cache_dtype=kv, k_scale=0.75, v_scale=1.5,
                                peaky_fraction=0.01, unused_slot_fill=float("nan"))
    assert inp["key_cache"].dtype == torch.uint8 and inp["x"] == 16
    pkv.set_attention_warps(warps)
    try:
        _check_all_modes(inp, dtype, f"{dtype}/{kv} D{D} bs{bs} {H}/{Hk} w{warps}")
    finally:
        pkv.set_attention_warps(0)


def test_float8_typed_caches_are_read_as_codes():
    """float8_e4m3fn / float8_e5m2 tensors select the format by themselves."""
    for kv, t in (("fp8_e4m3", torch.float8_e4m3fn), ("fp8_e5m2", torch.float8_e5m2)):
        inp = workloads.make_inputs(num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                    dtype="bf16", seq_lens=[100, 517], seed=3,
                                    kv_cache_dtype=kv, k_scale=0.5, v_scale=2.0)
        g = on_device(inp)
        out_codes = run_v1(g)
        g2 = dict(g, key_cache=g["key_cache"].view(t), value_cache=g["value_cache"].view(t),
                  kv_cache_dtype="auto")
        assert torch.equal(run_v1(g2), out_codes)


@pytest.mark.parametrize("kv", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("shift", [-40, -12, 12, 40])
def test_bf16_queries_over_fp8_keep_their_range(kv, shift):
    """Queries scaled by 2^shift (exact in bf16) with k_scale 2^-shift give the
    unscaled logits; without the per-head power-of-two scaling into f16 they
    would underflow to zero or overflow to inf."""
    inp = workloads.make_inputs(num_heads=16, num_kv_heads=2, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=[700, 33, 129], seed=5,
                                kv_cache_dtype=kv, k_scale=2.0 ** -shift, v_scale=1.0)
    inp["query"] = (inp["query"].float() * 2.0 ** shift).to(torch.bfloat16)
    g = on_device(inp)
    ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                           inp["block_tables"], inp["seq_lens_list"], inp["scale"],
                           **oracle_kwargs(inp))
    assert_attention_close(run_v1(g), ref, torch.bfloat16, f"{kv} query x 2^{shift}")


def test_fp8_rejects_fp32_queries():
    inp = workloads.make_inputs(num_heads=4, num_kv_heads=4, head_size=64, block_size=16,
                                dtype="bf16", seq_lens=[10], seed=1, kv_cache_dtype="fp8")
    g = on_device(inp)
    g["query"] = g["query"].float()
    with pytest.raises(RuntimeError, match="unsupported"):
        run_v1(g)


# ----------------------------------------------------------------- ALiBi ---

ALIBI_CASES = [
    # query dtype, kv_cache_dtype, D, bs, H, Hk
    ("bf16", "auto", 128, 16, 32, 8),
    ("f16", "auto", 64, 8, 8, 8),
    ("f32", "auto", 128, 16, 8, 2),
    ("f32", "auto", 64, 32, 4, 4),
    ("bf16", "fp8_e4m3", 128, 16, 16, 2),
    ("f16", "fp8_e5m2", 256, 8, 12, 1),
    ("bf16", "auto", 128, 16, 64, 4),
]


@pytest.mark.parametrize("warps", [0, 1, 4])
@pytest.mark.parametrize("dtype,kv,D,bs,H,Hk", ALIBI_CASES)
def test_alibi_parity(dtype, kv, D, bs, H, Hk, warps):
    lens = [1, 2 * bs + 3, 333, 1000, 3001]
    inp = workloads.make_inputs(num_heads=H, num_kv_heads=Hk, head_size=D, block_size=bs,
                                dtype=dtype, seq_lens=lens, seed=H + D, kv_cache_dtype=kv,
                                k_scale=1.25, v_scale=0.5, alibi=True,
                                unused_slot_fill=float("nan"))
    pkv.set_attention_warps(warps)
    try:
        _check_all_modes(inp, dtype, f"alibi {dtype}/{kv} D{D} bs{bs} {H}/{Hk} w{warps}")
    finally:
        pkv.set_attention_warps(0)


def test_alibi_steep_slopes_select_the_last_token():
    """Slopes of 50 per position: every weight but the last token's is below
    e^-50, so each head returns that token's value row."""
    inp = workloads.make_inputs(num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=[1, 17, 600], seed=9, alibi=True)
    inp["alibi_slopes"] = torch.full((8,), 50.0)
    inp["query"] = torch.zeros_like(inp["query"])
    g = on_device(inp)
    out = run_v1(g).float().cpu()
    vc = inp["value_cache"].float()
    for s, L in enumerate(inp["seq_lens_list"]):
        b = inp["block_rows"][s][(L - 1) // 16]
        for h in range(8):
            want = vc[b, h // 4, :, (L - 1) % 16]
            assert torch.equal(out[s, h], want.to(torch.bfloat16).float()), (s, h)


def test_alibi_slopes_must_be_float32_per_head():
    inp = workloads.make_inputs(num_heads=8, num_kv_heads=2, head_size=64, block_size=16,
                                dtype="bf16", seq_lens=[10], seed=2, alibi=True)
    g = on_device(inp)
    g["alibi_slopes"] = g["alibi_slopes"][:4]
    with pytest.raises(ValueError):
        run_v1(g)
    assert not math.isnan(float(inp["alibi_slopes"][0]))


@pytest.mark.parametrize("warps", [0, 2])
def test_fp8_copy_wait_timeout_is_reported_and_the_context_survives(warps):
    """The fp8 body's bounded waits: with the test hook every stage expects 16
    bytes that never arrive, the waits run out (20 ms), the kernel reports
    PKV_ERRF_TIMEOUT and finishes, and the next launch is correct."""
    inp = workloads.make_inputs(num_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=[64, 300], seed=51,
                                kv_cache_dtype="fp8_e4m3", k_scale=0.5, v_scale=2.0)
    g = on_device(inp)
    ref = oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                           inp["block_tables"], inp["seq_lens_list"], inp["scale"],
                           **oracle_kwargs(inp))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_attention_warps(warps)
    pkv.set_wait_limit_ns(20_000_000)
    pkv._test_set_unarrived_bytes(16)
    try:
        run_v1(g, err=err)
        torch.cuda.synchronize()
    finally:
        pkv._test_set_unarrived_bytes(0)
        pkv.set_wait_limit_ns(0)
    try:
        assert int(err.item()) & pkv.PKV_ERRF_TIMEOUT
        err.zero_()
        out = run_v1(g, err=err)
        torch.cuda.synchronize()
    finally:
        pkv.set_attention_warps(0)
    assert int(err.item()) == 0
    assert_attention_close(out, ref, torch.bfloat16, f"fp8 after timeout, warps {warps}")
