"""Pins for oracle.mxfp8: torch's own float8 casts, hand-worked examples, round trips."""
import os

import numpy as np
import pytest
import torch

from oracle import mxfp8 as mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_scale_examples.txt")
TORCH_FMT = {mx.E4M3: torch.float8_e4m3fn, mx.E5M2: torch.float8_e5m2}
FMT = {"e4m3": mx.E4M3, "e5m2": mx.E5M2}


@pytest.mark.parametrize("fmt", [mx.E4M3, mx.E5M2])
def test_decode_table_matches_torch(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(TORCH_FMT[fmt]).to(torch.float64).numpy()
    ours = mx.fp8_decode_table(fmt)
    finite = np.isfinite(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[finite], ref[finite])
    assert mx.fp8_max(fmt) == {mx.E4M3: 448.0, mx.E5M2: 57344.0}[fmt]


@pytest.mark.parametrize("fmt", [mx.E4M3, mx.E5M2])
def test_encode_matches_torch_rne_on_all_bf16_patterns(fmt):
    """torch's CPU float8 cast is round-to-nearest-even; compare on every in-range bf16 value."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).to(torch.float64)
    vmax = mx.fp8_max(fmt)
    for shift in (0, -6, 6, -12):
        w = v * 2.0 ** shift
        ok = torch.isfinite(w) & (w.abs() <= vmax)
        w = w[ok]
        ref = w.to(TORCH_FMT[fmt]).view(torch.uint8).numpy().copy()   # signed zeros included
        ours = mx.fp8_encode(w.numpy(), fmt)
        assert np.array_equal(ours, ref), f"shift {shift}"


@pytest.mark.parametrize("fmt", [mx.E4M3, mx.E5M2])
def test_encode_saturates(fmt):
    vmax = mx.fp8_max(fmt)
    c = mx.fp8_encode(np.array([vmax * 1.01, -vmax * 4, 1e30]), fmt)
    assert list(mx.fp8_to_float(c, fmt)) == [vmax, -vmax, vmax]


def _read_golden():
    scales, groups = [], []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "scale":
            scales.append((FMT[f[1]], float(f[2]), int(f[3])))
        else:
            arrow = f.index("->")
            vals = [float(t) for t in f[2:arrow]]
            byte = int(f[arrow + 1])
            codes = [int(t, 16) for t in f[arrow + 2:]]
            groups.append((FMT[f[1]], vals, byte, codes))
    return scales, groups


def test_golden_scale_bytes():
    scales, _ = _read_golden()
    assert len(scales) >= 10
    for fmt, amax, byte in scales:
        amax32 = np.float32(amax).astype(np.float64)
        assert int(mx.e8m0_byte(np.array([amax32]), fmt)[0]) == byte, (fmt, amax)


def test_golden_groups():
    _, groups = _read_golden()
    assert len(groups) >= 4
    for fmt, vals, byte, codes in groups:
        v = np.zeros(32)
        v[: len(vals)] = vals
        q, s = mx.mx_quantize(v[None, :], fmt, axis=1)
        assert int(s[0, 0]) == byte
        assert [int(c) for c in q[0, : len(codes)]] == codes
        assert np.all(q[0, len(codes):] == 0)


@pytest.mark.parametrize("fmt", [mx.E4M3, mx.E5M2])
def test_roundtrip_identity_on_representable_groups(fmt):
    """Groups built from FP8 values times a power of two, with the group max in the top binade,
    are reproduced exactly."""
    rng = np.random.default_rng(3)
    table = mx.fp8_decode_table(fmt)
    emax = {mx.E4M3: 8, mx.E5M2: 15}[fmt]
    finite = np.nonzero(np.isfinite(table))[0]
    vals = table[rng.choice(finite, size=(64, 32))]
    vals = np.clip(vals, -2.0 ** emax * 1.5, 2.0 ** emax * 1.5)
    vals[:, 0] = 2.0 ** emax                       # amax in [2^emax, 2^(emax+1))
    vals = vals * np.ldexp(1.0, rng.integers(-20, 20, size=(64, 1)))
    back = mx.mx_roundtrip(vals, fmt, axis=1)
    assert np.array_equal(back, vals)


@pytest.mark.parametrize("fmt", [mx.E4M3, mx.E5M2])
def test_group_max_lands_in_top_binade(fmt):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((200, 32)) * np.ldexp(1.0, rng.integers(-30, 30, size=(200, 1)))
    q, s = mx.mx_quantize(v, fmt, axis=1)
    emax = {mx.E4M3: 8, mx.E5M2: 15}[fmt]
    amax = np.max(np.abs(v), axis=1)
    scaled = amax / np.ldexp(1.0, s.astype(np.int64)[:, 0] - 127)
    assert np.all((scaled >= 2.0 ** emax) & (scaled < 2.0 ** (emax + 1)))
    # every element is within a quarter of 2^emax (in scaled units) of its input: half an ulp of
    # the top binade for e5m2, and the saturation gap 2^(emax+1) - max for both formats
    back = mx.mx_dequantize(q, s, fmt, axis=1)
    tol = 0.25 * 2.0 ** emax * np.ldexp(1.0, s.astype(np.int64)[:, 0] - 127)
    assert np.all(np.abs(back - v) <= tol[:, None])


def test_quantize_axis_and_padding_shapes():
    v = np.arange(64 * 3, dtype=np.float64).reshape(64, 3)
    q, s = mx.mx_quantize(v, mx.E5M2, axis=0)
    assert q.shape == (64, 3) and s.shape == (2, 3)
    with pytest.raises(AssertionError):
        mx.mx_quantize(np.ones((3, 33)), mx.E5M2, axis=1)


def _same_values(a, b):
    """Equal as numbers and in the sign of every zero."""
    return np.array_equal(a, b) and np.array_equal(np.signbit(a), np.signbit(b))


@pytest.mark.parametrize("fmt", [mx.E4M3, mx.E5M2])
@pytest.mark.parametrize("axis", [0, 1])
def test_torch_cast_roundtrip_equals_the_definition(fmt, axis):
    """mx_roundtrip_torch (the fast form the full-size tests use) gives bit for bit what mx_roundtrip
    gives: float32 values spread over 2^-140 .. 2^+100 within a group, zeros of both signs, groups of
    a single huge or tiny value, ties of the element rounding."""
    rng = np.random.default_rng(3)
    shape = (256, 192)
    mant = rng.standard_normal(shape)
    expo = rng.integers(-140, 100, size=shape)
    v = np.asarray(np.ldexp(mant, expo), dtype=np.float32).astype(np.float64)
    v[rng.random(shape) < 0.05] = 0.0
    v[rng.random(shape) < 0.05] = -0.0
    v[:32, :32] = 0.0
    v[0, 0] = float(np.float32(3.0e38)) if axis == 1 else v[0, 0]
    # ties: values exactly halfway between two FP8 neighbours once scaled (group amax 2^emax)
    emax = {mx.E4M3: 8, mx.E5M2: 15}[fmt]
    mbits = {mx.E4M3: 3, mx.E5M2: 2}[fmt]
    ties = (1.0 + (2 * np.arange(31) + 1) / 2.0 ** (mbits + 1)) * 2.0 ** (emax - 3)
    if axis == 1:
        v[40, :32] = np.concatenate([[2.0 ** emax], ties])
        v[41, :32] = -v[40, :32]
    else:
        v[:32, 40] = np.concatenate([[2.0 ** emax], ties])
        v[:32, 41] = -v[:32, 40]
    assert _same_values(mx.mx_roundtrip_torch(v, fmt, axis), mx.mx_roundtrip(v, fmt, axis))


@pytest.mark.parametrize("fmt", [mx.E4M3, mx.E5M2])
def test_torch_cast_roundtrip_on_all_bf16_patterns(fmt):
    """Every finite bf16 value, in groups of 32 consecutive patterns, through both round trips."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).to(torch.float64).numpy()
    v = np.where(np.isfinite(v), v, 0.0).reshape(-1, 32)
    for shift in (0, -20, 20):
        w = np.ldexp(v, shift)
        w = np.where(w.astype(np.float32).astype(np.float64) == w, w, 0.0)   # float32 numbers only
        assert _same_values(mx.mx_roundtrip_torch(w, fmt, 1), mx.mx_roundtrip(w, fmt, 1)), shift
        assert _same_values(mx.mx_roundtrip_torch(w.T.copy(), fmt, 0), mx.mx_roundtrip(w.T.copy(), fmt, 0)), shift


def test_torch_cast_roundtrip_refuses_values_beyond_float32():
    with pytest.raises(ValueError):
        mx.mx_roundtrip_torch(np.full((1, 32), 1e300), mx.E5M2, 1)
