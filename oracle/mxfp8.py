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
