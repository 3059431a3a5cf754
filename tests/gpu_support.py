"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding and compare it with the oracle under the tolerances the tests use.

Tolerances (max-abs against the float64 oracle):
* fp32 input/output: 1e-5.
* fp16 / bf16 output: ``max(2e-3, 1 ulp of the output dtype at |ref|)``.  A
  correctly rounded bf16 value already sits up to half an ulp (3.9e-3 for
  |ref| in [1, 2)) from the exact result, so a literal 2e-3 cannot hold for
  large outputs; one ulp leaves room for fp32 accumulation near a rounding
  boundary.
* fp32 split-KV partials (tmp_out): 2e-3 absolute, no ulp allowance;
  exp_sums: 1e-4 relative; max_logits: 1e-4 relative + 1e-5 absolute.
"""
import math

import torch

import paged_kv_decode_tables_gb300 as pkv

MANTISSA = {torch.float32: 23, torch.float16: 10, torch.bfloat16: 7}


def on_device(inp, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}


def attention_bound(ref: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    ref = ref.to(torch.float64)
    if dtype == torch.float32:
        return torch.full_like(ref, 1e-5)
    ulp = torch.pow(2.0, torch.floor(torch.log2(ref.abs().clamp_min(1e-30))) - MANTISSA[dtype])
    return torch.clamp(ulp, min=2e-3)


def assert_attention_close(got: torch.Tensor, ref: torch.Tensor, dtype: torch.dtype, what=""):
    got = got.detach().to("cpu", torch.float64)
    ref = ref.to(torch.float64)
    mask = ~torch.isnan(ref)  # rows the oracle did not compute are NaN
    assert bool(torch.isfinite(got[mask]).all()), f"{what}: non-finite output"
    diff = (got - ref).abs()
    bound = attention_bound(ref, dtype)
    bad = mask & (diff > bound)
    if bool(bad.any()):
        idx = bad.nonzero()[0].tolist()
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements out of tolerance; max-abs {float(diff[mask].max()):.3e}; "
            f"first {idx}: got {float(got[tuple(idx)])} ref {float(ref[tuple(idx)])}")
    return float(diff[mask].max()) if bool(mask.any()) else 0.0


def variant_kwargs(g):
    """Cache format and ALiBi arguments of an input dict (defaults: plain)."""
    return dict(kv_cache_dtype=g.get("kv_cache_dtype", "auto"), k_scale=g.get("k_scale", 1.0),
                v_scale=g.get("v_scale", 1.0), alibi_slopes=g.get("alibi_slopes"))


def oracle_kwargs(inp):
    """The same arguments for the oracle (slopes as a host list)."""
    kw = variant_kwargs(inp)
    if kw["alibi_slopes"] is not None:
        kw["alibi_slopes"] = [float(v) for v in kw["alibi_slopes"].cpu()]
    return kw


def run_v1(g, *, err=None, block_tables=None, kv_indptr=None, stream=None):
    out = torch.empty_like(g["query"])
    pkv.paged_attention_decode(out, g["query"], g["key_cache"], g["value_cache"],
                               g["block_tables"] if block_tables is None else block_tables,
                               g["seq_lens"], g["scale"], kv_indptr=kv_indptr, err_flag=err,
                               stream=stream, **variant_kwargs(g))
    return out


def run_v2(g, max_parts, *, partition_size=512, splits=None, err=None, block_tables=None,
           kv_indptr=None):
    B, H, D = g["query"].shape
    dev = g["query"].device
    tmp = torch.full((B, H, max_parts, D), float("nan"), dtype=torch.float32, device=dev)
    es = torch.full((B, H, max_parts), float("nan"), dtype=torch.float32, device=dev)
    ml = torch.full((B, H, max_parts), float("nan"), dtype=torch.float32, device=dev)
    pkv.paged_attention_v2_partition(tmp, es, ml, g["query"], g["key_cache"], g["value_cache"],
                                     g["block_tables"] if block_tables is None else block_tables,
                                     g["seq_lens"], g["scale"], partition_size=partition_size,
                                     num_kv_splits=splits, kv_indptr=kv_indptr, err_flag=err,
                                     **variant_kwargs(g))
    out = torch.empty_like(g["query"])
    pkv.paged_attention_v2_reduce(out, tmp, es, ml, g["seq_lens"], partition_size=partition_size,
                                  num_kv_splits=splits, block_size=g["block_size"], err_flag=err)
    return tmp, es, ml, out


def assert_partials_close(tmp, es, ml, rtmp, res, rml, what=""):
    tmp, es, ml = (t.detach().cpu().double() for t in (tmp, es, ml))
    empty = res == 0
    assert bool((es[empty] == 0).all()), f"{what}: empty partitions must have exp_sums 0"
    assert bool((ml[empty] == -math.inf).all()), f"{what}: empty partitions must have -inf"
    full = (~empty) & ~torch.isnan(res)
    assert bool(((es[full] - res[full]).abs() <= 1e-4 * res[full]).all()), f"{what}: exp_sums"
    assert bool(((ml[full] - rml[full]).abs() <= 1e-4 * rml[full].abs() + 1e-5).all()), \
        f"{what}: max_logits"
    d = (tmp - rtmp).abs()[full]
    assert bool((d <= 2e-3).all()), f"{what}: tmp_out max-abs {float(d.max())}"
    return float(d.max()) if d.numel() else 0.0
