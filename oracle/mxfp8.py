"""Oracle: FP8 codecs and MXFP8 group quantisation (test infrastructure only).

The pages fix only the shape of the scheme: 32-element groups along a GEMM's contraction
dimension, one E8M0 shared scale per group, FP8 e4m3 / e5m2 elements (blockwise MoE backward
page, first paragraph and gate_up_weight_scales / down_weight_scales; dense matmul backward page,
float8_dtype default "float8_e5m2").  The scale rule is the OCP Microscaling (MX) v1.0 one:

    shared_exp = floor(log2(amax)) - emax_elem        emax_elem = 8 (e4m3), 15 (e5m2)
    scale byte = clamp(shared_exp + 127, 0, 254)      E8M0, value 2^(byte - 127)
    element    = RNE(v / 2^(byte - 127)) in the FP8 format, saturating to +-max finite

with floor(log2(amax)) read off the binary exponent of amax (exact, no log), amax = 0 (or a
subnormal amax) giving byte 0.  The sign is kept: a negative value (or -0) that rounds to zero
gives -0 (code 0x80), as torch's float8 dtypes (the matmul page's float8_dtype) convert.  NaN / Inf
inputs are outside the contract.

Bit-exact by construction: the decode tables come from the format definitions; encoding is the
nearest table value with ties going to the even code.
"""
from __future__ import annotations

import numpy as np

E4M3, E5M2 = 0, 1
_SPEC = {  # exponent bits, mantissa bits, bias, emax_elem, largest finite code (positive)
    E4M3: (4, 3, 7, 8, 0x7E),
    E5M2: (5, 2, 15, 15, 0x7B),
}


def fp8_decode_table(fmt: int) -> np.ndarray:
    """Value of each of the 256 codes (NaN / Inf codes map to NaN / Inf)."""
    ebits, mbits, bias, _, _ = _SPEC[fmt]
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> mbits) & ((1 << ebits) - 1)
        m = c & ((1 << mbits) - 1)
        if fmt == E4M3 and e == 15 and m == 7:
            out[c] = np.nan
        elif fmt == E5M2 and e == 31:
            out[c] = sign * np.inf if m == 0 else np.nan
        elif e == 0:
            out[c] = sign * m * 2.0 ** (1 - bias - mbits)
        else:
            out[c] = sign * (1.0 + m / 2.0 ** mbits) * 2.0 ** (e - bias)
    return out


def fp8_max(fmt: int) -> float:
    return float(fp8_decode_table(fmt)[_SPEC[fmt][4]])


def fp8_encode(y: np.ndarray, fmt: int) -> np.ndarray:
    """Round-to-nearest-even into the FP8 format, saturating to +-max; the sign bit is kept (a
    negative value rounding to zero gives -0)."""
    y = np.asarray(y, dtype=np.float64)
    table = fp8_decode_table(fmt)
    maxc = _SPEC[fmt][4]
    pos = table[: maxc + 1]                      # codes 0..maxc, strictly increasing values
    a = np.minimum(np.abs(y), pos[-1])
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, maxc)   # first value >= a
    lo = np.clip(hi - 1, 0, maxc)
    d_hi = pos[hi] - a
    d_lo = a - pos[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = np.signbit(y).astype(np.uint8) << 7
    return (mag | sign).astype(np.uint8)


def fp8_to_float(codes: np.ndarray, fmt: int) -> np.ndarray:
    return fp8_decode_table(fmt)[np.asarray(codes, dtype=np.uint8)]


def e8m0_byte(amax: np.ndarray, fmt: int) -> np.ndarray:
    """Shared-scale byte from the group amax (see module docstring)."""
    amax = np.asarray(amax, dtype=np.float64)
    emax_elem = _SPEC[fmt][3]
    _, ex = np.frexp(amax)                      # amax = m * 2**ex, m in [0.5, 1)
    floor_log2 = ex.astype(np.int64) - 1
    byte = np.where(amax > 0, floor_log2 - emax_elem + 127, 0)
    return np.clip(byte, 0, 254).astype(np.uint8)


def mx_quantize(v: np.ndarray, fmt: int, axis: int = -1):
    """Quantise `v` in groups of 32 consecutive elements along `axis`.

    Returns (codes uint8 with v's shape, scale bytes uint8 with that axis divided by 32).
    The length along `axis` must be a multiple of 32 (callers pad with zeros).
    """
    v = np.moveaxis(np.asarray(v, dtype=np.float64), axis, -1)
    n = v.shape[-1]
    assert n % 32 == 0, "group axis must be a multiple of 32"
    g = v.reshape(v.shape[:-1] + (n // 32, 32))
    byte = e8m0_byte(np.max(np.abs(g), axis=-1), fmt)
    scale = np.ldexp(1.0, byte.astype(np.int64) - 127)
    codes = fp8_encode(g / scale[..., None], fmt).reshape(v.shape)
    return np.moveaxis(codes, -1, axis), np.moveaxis(byte, -1, axis)


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, fmt: int, axis: int = -1) -> np.ndarray:
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1)
    vals = fp8_to_float(c, fmt)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    out = vals * np.repeat(scale, 32, axis=-1)
    return np.moveaxis(out, -1, axis)


def mx_roundtrip(v: np.ndarray, fmt: int, axis: int = -1) -> np.ndarray:
    """dequantize(quantize(v)) along `axis`: the value an MXFP8 GEMM operand carries."""
    q, s = mx_quantize(v, fmt, axis)
    return mx_dequantize(q, s, fmt, axis)


def mx_roundtrip_torch(v: np.ndarray, fmt: int, axis: int = -1) -> np.ndarray:
    """mx_roundtrip of a 2-D array of float32 numbers with torch's CPU float8 cast as the element
    rounding, for operands of a quarter of a billion elements (the full-size parity tests), where the
    table search above takes minutes.

    The same rule, step by step: the group amax (a tree of pairwise maxima), the scale byte from its
    binary exponent, the scaled value (a division by a power of two, exact in float32 wherever the
    result can round to a nonzero code) clamped to +-max finite, then round-to-nearest-even into the
    format by the cast, which keeps the sign of zero; the dequantised value (an FP8 value times a power
    of two) is exact in float32 for float32 inputs.  The oracle quantises only float32 numbers (bf16
    inputs, intermediates rounded to float32 first); other inputs raise.  Pinned equal to
    mx_roundtrip (tests/test_oracle_mxfp8.py)."""
    import torch
    a = np.asarray(v, dtype=np.float64)
    assert a.ndim == 2 and axis in (0, 1, -1), "2-D operands, groups along one of the two axes"
    t64 = torch.from_numpy(np.ascontiguousarray(a))
    t = t64.to(torch.float32)
    if not torch.equal(t.to(torch.float64), t64):
        raise ValueError("mx_roundtrip_torch quantises float32 numbers only")
    R, C = t.shape
    if axis == 0:
        assert R % 32 == 0, "group axis must be a multiple of 32"
        g = t.view(R // 32, 32, C)        # group index, element of the group, column
        gdim = 1
    else:
        assert C % 32 == 0, "group axis must be a multiple of 32"
        g = t.view(R, C // 32, 32)
        gdim = 2
    m = g.abs()
    width = 32
    while width > 1:                     # amax of each group by halving
        width //= 2
        m = torch.maximum(m.narrow(gdim, 0, width), m.narrow(gdim, width, width))
    amax = m.squeeze(gdim)
    byte = e8m0_byte(amax.to(torch.float64).numpy(), fmt).astype(np.int64)
    scale = torch.from_numpy(np.ldexp(1.0, byte - 127)).to(torch.float32).unsqueeze(gdim)
    maxv = fp8_max(fmt)
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    y = (g / scale).clamp_(-maxv, maxv).to(dt).to(torch.float32) * scale
    return y.reshape(R, C).to(torch.float64).numpy()
