"""The no-allocation split-KV entry point, through the C ABI.

paged_attention_v2_noalloc serves callers that cannot call cudaMalloc (an
engine that reserves all device memory up front, a plugin whose host owns the
allocator, a path where allocation would add a synchronisation): its
partition scratch is a fixed array inside the library.  Two calls in a row
(different batches, fixed partitions then split counts) must each match the
regular partition + reduce entry points, which get torch-allocated scratch,
within the tests' attention tolerance.  This file is collected last so that a
failure here never hides the other tests.
"""
import ctypes

import pytest
import torch

import paged_kv_decode_tables_gb300 as pkv
import workloads
from gpu_support import attention_bound, on_device, run_v2

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


def _close(got, want, dtype):
    d = (got.double() - want.double()).abs().cpu()
    return bool((d <= attention_bound(want.double().cpu(), dtype)).all()), float(d.max())


def test_noalloc_matches_regular_entry_points_twice_in_a_row():
    # call 1: fixed 512-token partitions
    inp1 = workloads.make_inputs(num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                                 dtype="bf16", seq_lens=[1, 700, 4097, 2048, 33], seed=41)
    g1 = on_device(inp1)
    maxP1 = -(-inp1["max_blocks_per_seq"] * 16 // 512)
    out1 = torch.full_like(g1["query"], float("nan"))
    assert _noalloc_call(g1, out1, maxP1, 512) == 0
    _, _, _, ref1 = run_v2(g1, maxP1, partition_size=512)

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

    ok1, e1 = _close(out1, ref1, torch.bfloat16)
    ok2, e2 = _close(out2, ref2, torch.float16)
    assert ok1, f"call 1 differs from the regular path by {e1}"
    assert ok2, f"call 2 differs from the regular path by {e2}"


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
