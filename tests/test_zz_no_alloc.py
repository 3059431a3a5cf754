"""The no-allocation split-KV entry point, through the C ABI.

paged_attention_v2_noalloc serves callers that cannot call cudaMalloc (an
engine that reserves all device memory up front, a plugin whose host owns the
allocator, a path where allocation would add a synchronisation): its
partition scratch is a fixed array inside the library, shared by every call.

It runs the same two kernels as paged_attention_v2_partition followed by
paged_attention_v2_reduce (which get torch-allocated scratch here) on the same
inputs, so its output must be bitwise equal to theirs, call after call; each
output is also checked against the float64 oracle at the attention
tolerance.  Between calls the array keeps the previous call's contents, so a
call that fills it with NaN partials comes before a call with more
partitions and zero-length sequences: a scratch entry the second call read
without writing it first would show up as NaN or as a bitwise difference.

This file is collected last so that a failure here never hides the other
tests; it passes alone in a fresh process as well.
"""
import ctypes

import pytest
import torch

import oracle
import paged_kv_decode_tables_gb300 as pkv
import workloads
from gpu_support import assert_attention_close, on_device, oracle_kwargs, run_v2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_decode_tables_gb300 import _build
    _build.build()


def _noalloc_call(g, out, max_parts, partition_size, splits=None):
    a = pkv._decode_args(g["query"], g["key_cache"], g["value_cache"], g["block_tables"],
                         g["seq_lens"], g["scale"], None, None, None)
    strides = (ctypes.c_int64 * 3)(*out.stride())
    return pkv.lib().paged_attention_v2_noalloc(
        out.data_ptr(), strides, max_parts, partition_size,
        None if splits is None else splits.data_ptr(), ctypes.byref(a),
        torch.cuda.current_stream().cuda_stream)


def _oracle(inp):
    return oracle.decode_v1(inp["query"], inp["key_cache"], inp["value_cache"],
                            inp["block_tables"], inp["seq_lens_list"], inp["scale"],
                            **oracle_kwargs(inp))


def _max_parts(inp, partition_size):
    return -(-inp["max_blocks_per_seq"] * inp["block_size"] // partition_size)


def _check(got, regular, inp, dtype, what):
    assert torch.equal(got, regular), (
        f"{what}: differs from the regular partition + reduce path by "
        f"{float((got.double() - regular.double()).abs().max())}")
    assert_attention_close(got, _oracle(inp), dtype, what)


def test_noalloc_matches_regular_entry_points_call_after_call():
    # call 1: fixed 512-token partitions
    inp1 = workloads.make_inputs(num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                                 dtype="bf16", seq_lens=[1, 700, 4097, 2048, 33], seed=41)
    g1 = on_device(inp1)
    maxP1 = _max_parts(inp1, 512)
    out1 = torch.full_like(g1["query"], float("nan"))
    assert _noalloc_call(g1, out1, maxP1, 512) == 0
    _, _, _, ref1 = run_v2(g1, maxP1, partition_size=512)
    torch.cuda.synchronize()
    _check(out1, ref1, inp1, torch.bfloat16, "call 1 (fixed partitions)")

    # call 2: a different batch with per-sequence split counts
    lens2 = [5000, 17, 1, 9000, 640, 2049]
    inp2 = workloads.make_inputs(num_heads=16, num_kv_heads=2, head_size=128, block_size=16,
                                 dtype="f16", seq_lens=lens2, seed=42)
    g2 = on_device(inp2)
    splits = torch.empty(len(lens2), dtype=torch.int32, device="cuda")
    pkv.compute_num_kv_splits(splits, g2["seq_lens"], num_group=1, num_head=16, num_kv_head=2,
                              max_kv_splits=16, device_core_count=148)
    out2 = torch.full_like(g2["query"], float("nan"))
    assert _noalloc_call(g2, out2, 16, 0, splits) == 0
    _, _, _, ref2 = run_v2(g2, 16, splits=splits)
    torch.cuda.synchronize()
    _check(out2, ref2, inp2, torch.float16, "call 2 (split counts)")

    # fill the scratch with NaN partials: every partition of every sequence is
    # non-empty and every value row is NaN, over more scratch than call 3 uses
    poison = workloads.make_inputs(num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                                   dtype="bf16", seq_lens=[2048] * 4, seed=44)
    gp = on_device(poison)
    gp["value_cache"].fill_(float("nan"))
    outp = torch.empty_like(gp["query"])
    maxPp = _max_parts(poison, 16)
    assert maxPp == 128
    assert _noalloc_call(gp, outp, maxPp, 16) == 0
    torch.cuda.synchronize()
    assert bool(torch.isnan(outp).all())

    # call 3: zero-length sequences and more partitions than calls 1 and 2
    lens3 = [0, 3000, 5, 0, 1500]
    inp3 = workloads.make_inputs(num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                                 dtype="bf16", seq_lens=lens3, seed=45)
    g3 = on_device(inp3)
    maxP3 = _max_parts(inp3, 64)
    assert maxP3 > max(maxP1, 16)
    # call 3's three scratch regions lie inside what the NaN call wrote
    assert 5 * 32 * maxP3 * (128 + 2) * 4 + 3 * 256 <= 4 * 32 * maxPp * 128 * 4
    out3 = torch.full_like(g3["query"], float("nan"))
    assert _noalloc_call(g3, out3, maxP3, 64) == 0
    _, _, _, ref3 = run_v2(g3, maxP3, partition_size=64)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out3).all())
    assert bool((out3[0] == 0).all()) and bool((out3[3] == 0).all())  # empty sequences
    _check(out3, ref3, inp3, torch.bfloat16, "call 3 (after NaN scratch)")


def test_noalloc_rejects_requests_beyond_its_scratch():
    cap = pkv.noalloc_scratch_bytes()
    assert cap == 32 << 20
    inp = workloads.make_inputs(num_heads=8, num_kv_heads=8, head_size=128, block_size=16,
                                dtype="bf16", seq_lens=[64] * 4, seed=43)
    g = on_device(inp)
    out = torch.zeros_like(g["query"])
    # 4 seqs x 8 heads x maxP x (128 + 2) x 4 B > 32 MiB once maxP > 2016
    st = _noalloc_call(g, out, 4096, 16)
    assert st == pkv.PKV_ERR_SCRATCH_TOO_SMALL
    assert pkv.lib().pkv_status_string(st).startswith(b"request exceeds")
    torch.cuda.synchronize()
    assert bool((out == 0).all())  # nothing was launched
