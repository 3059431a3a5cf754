"""Pins of the oracle's two decode variants (no GPU): fp8 KV caches with
k_scale / v_scale, and ALiBi logit biases.

The split-KV wrapper on page "paged_attention_v2_triton.py" names both
(``alibi_slopes``, ``kv_cache_dtype``, ``k_scale``, ``v_scale``) and defines
neither; the oracle takes vLLM's reading (fp8 codes decoded and scaled) and
the ALiBi paper's definition.  The pins tie the code decoding to torch's
float8 types over all 256 codes, the fp8 path to the already-pinned plain
path on dequantized caches, and ALiBi to torch's scaled_dot_product_attention
with an additive mask, a geometric closed form and its zero-bias anchor.
"""
import math

import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.attention as oatt
import oracle.fp8 as ofp8
from test_oracle_pins import _random_paged_problem, _scatter_to_pages

TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


# ---------------------------------------------------------------- fp8 codes ---

@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_every_code_matches_torch_float8(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(TORCH_FP8[fmt]).to(torch.float64)
    got = ofp8.decode(codes, fmt)
    nan = torch.isnan(want)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(got[~nan], want[~nan])
    # signed zeros too
    assert math.copysign(1.0, float(got[0x80])) == -1.0


def test_format_landmarks():
    """Largest finite, smallest normal and smallest subnormal magnitude of each
    format, and its special codes (OCP OFP8 specification, format table)."""
    v = ofp8.code_value
    assert v(0x7E, "e4m3") == 448.0 and v(0xFE, "e4m3") == -448.0
    assert v(0x08, "e4m3") == 2.0 ** -6 and v(0x01, "e4m3") == 2.0 ** -9
    assert v(0x38, "e4m3") == 1.0 and math.isnan(v(0x7F, "e4m3")) and math.isnan(v(0xFF, "e4m3"))
    assert v(0x7B, "e5m2") == 57344.0 and v(0x04, "e5m2") == 2.0 ** -14
    assert v(0x01, "e5m2") == 2.0 ** -16 and v(0x3C, "e5m2") == 1.0
    assert v(0x7C, "e5m2") == math.inf and v(0xFC, "e5m2") == -math.inf
    assert math.isnan(v(0x7D, "e5m2"))
    assert ofp8.format_of("fp8") == "e4m3" and ofp8.format_of("auto") is None


# ------------------------------------------------------------ fp8 decoding ---

def _fp8_problem(seed, fmt, B=3, H=8, Hk=2, D=32, bs=8):
    """A paged problem whose caches hold fp8 codes (x = 16), plus the same
    caches dequantized by torch's float8 conversion (x = 16 as well)."""
    pr = _random_paged_problem(seed, B, H, Hk, D, bs, 16)
    kc_codes = pr["kc"].to(torch.float32).to(TORCH_FP8[fmt]).view(torch.uint8)
    vc_codes = pr["vc"].to(torch.float32).to(TORCH_FP8[fmt]).view(torch.uint8)
    kc_val = kc_codes.view(TORCH_FP8[fmt]).to(torch.float64)
    vc_val = vc_codes.view(TORCH_FP8[fmt]).to(torch.float64)
    return pr, kc_codes, vc_codes, kc_val, vc_val


@pytest.mark.parametrize("fmt,name", [("e4m3", "fp8"), ("e4m3", "fp8_e4m3"), ("e5m2", "fp8_e5m2")])
def test_fp8_cache_equals_the_dequantized_cache(fmt, name):
    """decode(code) * k_scale on keys and * v_scale on values, nothing else:
    the fp8 path equals the plain path on caches torch dequantized."""
    pr, kcc, vcc, kcv, vcv = _fp8_problem(11, fmt)
    ks, vs, scale = 0.375, 2.5, 0.2
    got = oracle.decode_v1(pr["q"], kcc, vcc, pr["bt"], pr["lens"], scale, kv_cache_dtype=name,
                           k_scale=ks, v_scale=vs)
    want = oracle.decode_v1(pr["q"], kcv * ks, vcv * vs, pr["bt"], pr["lens"], scale)
    assert torch.allclose(got, want, rtol=0, atol=1e-12)
    # float8-typed tensors are read as their codes
    got2 = oracle.decode_v1(pr["q"], kcc.view(TORCH_FP8[fmt]), vcc.view(TORCH_FP8[fmt]),
                            pr["bt"], pr["lens"], scale, kv_cache_dtype=name, k_scale=ks,
                            v_scale=vs)
    assert torch.equal(got, got2)


def test_fp8_v2_equals_v1():
    pr, kcc, vcc, _, _ = _fp8_problem(12, "e4m3", bs=4)
    kw = dict(kv_cache_dtype="fp8_e4m3", k_scale=0.5, v_scale=1.25)
    v1 = oracle.decode_v1(pr["q"], kcc, vcc, pr["bt"], pr["lens"], 0.3, **kw)
    maxP = -(-max(pr["lens"]) // 4)
    tmp, es, ml = oracle.v2_partition(pr["q"], kcc, vcc, pr["bt"], pr["lens"], 0.3, maxP,
                                      partition_size=4, **kw)
    v2 = oracle.v2_reduce(tmp, es, ml, pr["lens"], 4, partition_size=4)
    assert torch.allclose(v1, v2, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ ALiBi ---

def _alibi_slopes(H):
    # any distinct positive slopes will do; these are the ALiBi paper's for 8 heads
    return [2.0 ** (-8.0 * (i + 1) / H) for i in range(H)]


@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 2)])
def test_alibi_matches_sdpa_with_an_additive_mask(H, Hk):
    """The query of a length-L decode sits at position L-1; key j gets
    -slope * (L-1-j) added to its scaled score (per query head)."""
    pr = _random_paged_problem(21 + H, 3, H, Hk, 16, 4, 4)
    slopes = _alibi_slopes(H)
    scale = 0.25
    got = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], scale,
                           alibi_slopes=slopes)
    for s, L in enumerate(pr["lens"]):
        K = pr["K_log"][s].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)  # [H, L, D]
        V = pr["V_log"][s].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)
        dist = (L - 1) - torch.arange(L, dtype=torch.float64)  # query pos - key pos
        mask = torch.stack([-slopes[h] * dist for h in range(H)])[:, None, :]  # [H, 1, L]
        o = F.scaled_dot_product_attention(pr["q"][s][:, None, :], K, V, attn_mask=mask,
                                           scale=scale)
        assert torch.allclose(got[s], o[:, 0, :], rtol=0, atol=1e-12)


def test_alibi_zero_query_closed_form():
    """q = 0: the weights are geometric, p_t ~ r^(L-1-t) with r = e^-slope, so
    with v_t = t the output is (L-1) - (r/(1-r) - L r^L / (1-r^L))."""
    L, D, bs, x = 37, 8, 8, 8
    K_log = [torch.randn(L, 1, D, dtype=torch.float64)]
    V_log = [torch.arange(L, dtype=torch.float64)[:, None, None].expand(L, 1, D).clone()]
    rows = [[4, 0, 2, 3, 1]]
    kc, vc = _scatter_to_pages(K_log, V_log, rows, [L], 6, bs, x)
    bt = torch.tensor(rows, dtype=torch.int32)
    q = torch.zeros(1, 1, D, dtype=torch.float64)
    for slope in (0.0625, 0.5, 3.0):
        got = oracle.decode_v1(q, kc, vc, bt, [L], 0.7, alibi_slopes=[slope])
        r = math.exp(-slope)
        want = (L - 1) - (r / (1 - r) - L * r ** L / (1 - r ** L))
        assert abs(float(got[0, 0, 0]) - want) < 1e-11


def test_alibi_bias_is_zero_at_the_last_token():
    """q = 0 and a positive slope: the largest logit is the last token's, 0,
    so the partition holding it reports max_logits 0 and the others below."""
    pr = _random_paged_problem(5, 2, 2, 2, 8, 4, 4, lens=[13, 9])
    q = torch.zeros_like(pr["q"])
    tmp, es, ml = oracle.v2_partition(q, pr["kc"], pr["vc"], pr["bt"], pr["lens"], 1.0, 4,
                                      partition_size=4, alibi_slopes=[0.5, 0.25])
    # seq 0: 13 tokens, partitions [0,4) [4,8) [8,12) [12,13): last holds token 12
    assert float(ml[0, 0, 3]) == 0.0 and float(ml[0, 1, 3]) == 0.0
    assert float(ml[0, 0, 2]) == -0.5 * 1 and float(ml[0, 1, 0]) == -0.25 * 9
    # seq 1: 9 tokens, [8,9) holds token 8
    assert float(ml[1, 0, 2]) == 0.0


def test_alibi_v2_equals_v1():
    pr = _random_paged_problem(6, 3, 4, 2, 16, 4, 4)
    slopes = _alibi_slopes(4)
    v1 = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.25,
                          alibi_slopes=slopes)
    for P in (4, 8, 64):
        maxP = -(-max(pr["lens"]) // P)
        tmp, es, ml = oracle.v2_partition(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"],
                                          0.25, maxP, partition_size=P, alibi_slopes=slopes)
        v2 = oracle.v2_reduce(tmp, es, ml, pr["lens"], 4, partition_size=P)
        assert torch.allclose(v1, v2, rtol=0, atol=1e-12)


# ----------------------------------------------------- planted mistakes ---

def test_variant_pins_catch_planted_mistakes(monkeypatch):
    # 1. ALiBi sign flipped
    monkeypatch.setattr(oatt, "alibi_bias",
                        lambda slope, L: -float(slope) * (torch.arange(L, dtype=torch.float64) - (L - 1)))
    with pytest.raises(AssertionError):
        test_alibi_zero_query_closed_form()
    monkeypatch.undo()

    # 2. ALiBi position measured from the first token instead of the query
    monkeypatch.setattr(oatt, "alibi_bias",
                        lambda slope, L: float(slope) * torch.arange(L, dtype=torch.float64))
    with pytest.raises(AssertionError):
        test_alibi_bias_is_zero_at_the_last_token()
    monkeypatch.undo()

    # 3. slopes indexed by kv head instead of query head
    orig_v1 = oatt.decode_v1

    def v1_kv_slopes(query, key_cache, value_cache, block_tables, seq_lens, scale, **kw):
        sl = kw.pop("alibi_slopes", None)
        H, Hk = query.shape[1], key_cache.shape[1]
        if sl is not None:
            sl = [sl[h // (H // Hk)] for h in range(H)]
        return orig_v1(query, key_cache, value_cache, block_tables, seq_lens, scale,
                       alibi_slopes=sl, **kw)

    monkeypatch.setattr(oracle, "decode_v1", v1_kv_slopes)
    with pytest.raises(AssertionError):
        test_alibi_matches_sdpa_with_an_additive_mask(8, 2)
    monkeypatch.undo()

    # 4. E4M3 exponent bias off by one
    monkeypatch.setitem(ofp8.FORMATS, "e4m3", (4, 3, 8, False))
    monkeypatch.setattr(ofp8, "_TABLES", {})
    with pytest.raises(AssertionError):
        test_every_code_matches_torch_float8("e4m3")
    monkeypatch.undo()

    # 5. k_scale and v_scale swapped
    orig_gather = oatt.gather_kv

    def swapped(kc, vc, ids, L, kvh, kv_format=None, k_scale=1.0, v_scale=1.0):
        return orig_gather(kc, vc, ids, L, kvh, kv_format, v_scale, k_scale)

    monkeypatch.setattr(oatt, "gather_kv", swapped)
    with pytest.raises(AssertionError):
        test_fp8_cache_equals_the_dequantized_cache("e4m3", "fp8")
    monkeypatch.undo()
