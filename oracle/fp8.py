"""8-bit floating-point KV-cache codes -> float64: TEST INFRASTRUCTURE.

The split-KV wrapper on page "paged_attention_v2_triton.py" takes
``kv_cache_dtype`` ("auto" or an fp8 format) with ``k_scale`` / ``v_scale``
and passes them through without defining them.  Reading (vLLM's convention,
which the page says its layouts follow): an fp8 cache stores one byte per
element, ``x = 16`` elements per key group, and the value an element stands
for is ``decode(code) * k_scale`` for keys and ``decode(code) * v_scale`` for
values.  ``"fp8"`` means E4M3.

The two formats are the OCP 8-bit floating point ones (OCP "8-bit Floating
Point Specification (OFP8)", 2023):

* E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
  ``S.1111.111`` is NaN, so the largest finite magnitude is 448.
* E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits; IEEE-style
  infinities (``S.11111.00``) and NaNs (``S.11111.mm``, mm != 0).

Both have subnormals at exponent field 0: ``m * 2^(1 - bias - mantissa_bits)``.
"""
from __future__ import annotations

import math

import torch

__all__ = ["FORMATS", "format_of", "code_value", "decode"]

# name -> (exponent bits, mantissa bits, bias, has infinities)
FORMATS = {
    "e4m3": (4, 3, 7, False),
    "e5m2": (5, 2, 15, True),
}


def format_of(kv_cache_dtype: str):
    """``None`` for "auto" (caches hold the query's dtype), else "e4m3"/"e5m2"."""
    names = {"auto": None, "fp8": "e4m3", "fp8_e4m3": "e4m3", "fp8_e5m2": "e5m2"}
    if kv_cache_dtype not in names:
        raise ValueError(f"unknown kv_cache_dtype {kv_cache_dtype!r}")
    return names[kv_cache_dtype]


def code_value(code: int, fmt: str) -> float:
    """The real number one 8-bit code stands for (NaN for the NaN codes)."""
    ebits, mbits, bias, has_inf = FORMATS[fmt]
    code = int(code) & 0xFF
    sign = -1.0 if code >> 7 else 1.0
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    e_max = (1 << ebits) - 1
    if has_inf and e == e_max:
        return sign * math.inf if m == 0 else math.nan
    if not has_inf and e == e_max and m == (1 << mbits) - 1:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** (1 - bias - mbits)
    return sign * (1.0 + m / (1 << mbits)) * 2.0 ** (e - bias)


def _table(fmt: str) -> torch.Tensor:
    return torch.tensor([code_value(c, fmt) for c in range(256)], dtype=torch.float64)


_TABLES = {}


def decode(codes: torch.Tensor, fmt: str) -> torch.Tensor:
    """Element-wise float64 values of a uint8 tensor of ``fmt`` codes."""
    if codes.dtype != torch.uint8:
        raise ValueError("fp8 codes must be a uint8 tensor")
    if fmt not in _TABLES:
        _TABLES[fmt] = _table(fmt)
    return _TABLES[fmt][codes.to(torch.int64)]
