"""Full-size workloads in the launch configuration bench.py times.

Metadata outputs are compared in full (bit-exact); attention outputs on
sampled sequences (first, last, shortest, longest and a few seeded picks) that
the oracle computes one by one, and on properties that hold everywhere:
every output is finite and, being a convex combination of value rows, lies
within the range of the cache's values.
"""
import pytest
import torch

import bench
import oracle
import workloads
from gpu_support import assert_attention_close, assert_partials_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_decode_tables_gb300 import _build
    _build.build()


def _samples(lens, extra=3, seed=0):
    n = len(lens)
    order = sorted(range(n), key=lambda i: lens[i])
    picks = {0, n - 1, order[0], order[-1]}
    g = torch.Generator().manual_seed(seed)
    for i in torch.randperm(n, generator=g)[:extra].tolist():
        picks.add(i)
    return sorted(picks)


def _run_step(name):
    step = bench.DecodeStep(name, seed=0, device="cuda")
    step.run()
    torch.cuda.synchronize()
    return step


def _value_range(inp):
    """Largest |value| the cache stands for (fp8: decoded code x v_scale)."""
    vc = inp["value_cache"]
    if inp["kv_cache_dtype"] != "auto":
        return float(vc.view(workloads.FP8_TORCH[inp["kv_cache_dtype"]]).float().abs().max()) * \
            inp["v_scale"]
    return float(vc.float().abs().max())


@pytest.mark.parametrize("name", ["mha_v1_fp16", "gqa_v1_bf16", "long_v2_bf16", "ragged_v2_bf16",
                                  "tiny_mha_fp32", "ragged_v2_fp8", "long_v2_fp8",
                                  "mha_v1_alibi_fp16", "gqa_v1_fp32"])
def test_full_size_workload(name):
    step = _run_step(name)
    inp, spec = step.inp, step.spec
    out = step.out
    assert bool(torch.isfinite(out).all()), "non-finite output"
    vmax = _value_range(inp)
    assert float(out.float().abs().max()) <= vmax * (1 + 2 ** -7) + 1e-3

    splits = None
    if spec.mode == "v2_splits":
        bt = inp["block_tables"].cpu()
        cu = inp["cu_num_blocks"].cpu().tolist()
        want_pi = oracle.copy_page_indices(bt, cu, cu[-1])
        assert step.page_indices.cpu().tolist() == want_pi
        splits = oracle.num_kv_splits(step.lens, 1, spec.num_heads, spec.num_kv_heads,
                                      spec.max_kv_splits, spec.device_core_count)
        assert step.splits.cpu().tolist() == splits

    seqs = _samples(step.lens)
    q, kc, vc, bt, lens = bench.oracle_sample_inputs(inp, seqs)
    kw = bench.oracle_variant_kwargs(inp)
    ref = oracle.decode_v1(q, kc, vc, bt, lens, inp["scale"], **kw)
    got = out[torch.tensor(seqs, device=out.device)]
    assert_attention_close(got, ref, DT[spec.dtype], f"{name} sampled outputs")

    if spec.mode != "v1":
        sel = torch.tensor(seqs, device=out.device)
        if spec.mode == "v2_fixed":
            maxP = step.maxP
            rtmp, res, rml = oracle.v2_partition(q, kc, vc, bt, lens, inp["scale"], maxP,
                                                 partition_size=spec.partition_size, **kw)
        else:
            maxP = step.maxP
            rtmp, res, rml = oracle.v2_partition(q, kc, vc, bt, lens, inp["scale"], maxP,
                                                 num_kv_splits=[splits[s] for s in seqs], **kw)
        assert_partials_close(step.tmp[sel], step.es[sel], step.ml[sel], rtmp, res, rml,
                              f"{name} sampled partials")


@pytest.mark.parametrize("name", ["ragged_v2_bf16", "gqa_v1_bf16", "long_v2_fp8"])
def test_end_to_end_step_equals_device_step(name):
    """The end-to-end step (one host-to-device copy of the input buffer, the
    step, the output copied back) reproduces the device-resident step bit for
    bit, after every device-side input has been overwritten."""
    step = _run_step(name)
    want = step.out.cpu()
    hin, hout = step.host_inputs()
    step.arena.fill_(0xFF)
    step.inp["block_tables"].fill_(-1)
    step.out.zero_()
    step.e2e_enqueue(hin, hout)
    torch.cuda.synchronize()
    assert torch.equal(hout, want)
    h2d, d2h = step.e2e_bytes(hin, hout)
    assert h2d == step.arena.numel() and d2h == want.numel() * want.element_size()
