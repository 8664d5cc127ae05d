"""Per-GEMM parity of the store GEMMs on their own operands.  MXFP8: the quantised operands the GPU
wrote to the workspace -- dh row-wise (dx_expanded's A), dh^T, x_g^T (dW1's), a'^T, dout_g^T (dW2's),
each with its tiled scales -- and the weights quantised by the oracle (the GPU's own weight codes are
pinned bit-exact to those elsewhere) are dequantised exactly; BF16: the operand rows (or transposed
copies) as written.  They are contracted in float64, expert by expert over its tile rows.  Both sides
read the same values, so quantisation near-ties cannot enter: what remains is the tensor core's
accumulation and the bf16 rounding of the GEMM outputs.  Compared: G2's dx_expanded (the workspace's
DX_EXP rows, padding rows included), G4's dW1 and G3's dW2, and G1's epilogue outputs (dh, ds, and
for MXFP8 the codes and scales of dh, dh^T and a'^T) from dA_raw on the rows the GPU gathered."""
import numpy as np
import pytest
import torch

from helpers import np64, rel_fro, run_gpu, tiled_sf_to_plain
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_MXFP8, make_moe_inputs,
                                                   small_moe, with_ids)
from oracle import mxfp8 as omx

pytestmark = pytest.mark.gpu

# bf16 output rounding (half an ulp is at most 2^-9 relative) dominates the difference from the float64
# result (about 1.7e-3 relative Frobenius).  Against that result rounded to bf16 the two differ only
# where the tensor core's sum lands on the other side of a rounding boundary: the last bit of a small
# share of the elements (measured: 0.002% over a few hundred rows, 0.5-0.7% over the 65k rows of the
# imbalanced workload's hottest expert).  Elementwise, |gpu - ref| stays within one bf16 ulp of ref
# plus an accumulation term 2^-18 * sum_k |a_k b_k| (which only matters where the sum cancels; the
# largest ratio measured is 0.5, the rounding itself).
L1_TOL = 2e-3
FLIP_SHARE = 0.01
ACC_EPS = 2.0 ** -18


def _ragged_ids(T, K, E, seed):
    rng = np.random.default_rng(seed)
    p = np.ones(E)
    p[0] = 0.0          # an empty expert
    p[E - 1] = 12.0     # a hot one: a contraction of several hundred rows
    p /= p.sum()
    ids = np.stack([rng.choice(E, size=K, replace=False, p=p) for _ in range(T)])
    return torch.from_numpy(ids.astype(np.int32))


def _deq(op, name, rows, cols, fmt):
    """Codes [rows, cols] of region `name` and its tiled scales (groups along cols), dequantised."""
    q = op.region(name).cpu().numpy().reshape(rows, cols)
    sf = tiled_sf_to_plain(op.region(name + "_SF").cpu().numpy(), rows, cols)
    return omx.mx_dequantize(q, sf, fmt, axis=-1)


def _ordered(a: np.ndarray) -> np.ndarray:
    """bf16 values as integers in the order of the values (adjacent bf16 numbers differ by one)."""
    b = torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)
    return np.where(b < 0, -32768 - b, b)


def _check(name, got, ref, mag):
    """`mag` = sum_k |a_k b_k| of each element (|A| |B|^T)."""
    err = rel_fro(got, ref)
    share = float(np.count_nonzero(_ordered(got) != _ordered(ref))) / ref.size
    ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(ref), 1e-300))).astype(np.int64) - 7)
    excess = float(np.max(np.abs(got - ref) / (ulp + ACC_EPS * mag + 1e-300)))
    msg = f"{name}: relative Frobenius {err:.3e}, {share:.3%} off the rounded result, excess {excess:.2f}"
    assert err <= L1_TOL and share <= FLIP_SHARE and excess <= 1.0, msg
    return err, share, excess


@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
def test_mxfp8_store_gemms_on_their_own_operands(affinity):
    cfg = small_moe("mx_l1", T=700, H=384, I=256, E=6, K=2, B=256, seed=36, precision=PREC_MXFP8,
                    affinity=affinity)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(700, 2, 6, seed=8))
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    P, H, I, fa = op.tile_rows, cfg.H, cfg.I, cfg.fp8_act
    toff = op.region("TILE_OFFSETS").view(torch.int32).cpu().numpy()
    used = int(toff[cfg.E])
    dh = _deq(op, "DH", P, 2 * I, fa)[:used]
    dh_t = _deq(op, "DH_T", 2 * I, P, fa)[:, :used]
    x_t = _deq(op, "X_GT", H, P, fa)[:, :used]
    ap_t = _deq(op, "AP_T", I, P, fa)[:, :used]
    dout_t = _deq(op, "DOUT_GT", H, P, fa)[:, :used]
    W1q, W1s = omx.mx_quantize(inp.W1.double().numpy(), cfg.fp8_w, axis=-1)   # [E, H, 2I], groups along 2I
    W1 = omx.mx_dequantize(W1q, W1s, cfg.fp8_w, axis=-1)
    dx_exp = np64(op.region("DX_EXP").view(torch.bfloat16).reshape(P, H))[:used]
    ref = {n: (np.zeros(shape), np.zeros(shape)) for n, shape in
           (("dx", (used, H)), ("dW1", (cfg.E, H, 2 * I)), ("dW2", (cfg.E, I, H)))}

    def put(n, idx, A, B):   # the contraction A B^T and its magnitude |A| |B|^T
        ref[n][0][idx] = A @ B.T
        ref[n][1][idx] = np.abs(A) @ np.abs(B).T

    for e in range(cfg.E):
        a, b = int(toff[e]), int(toff[e + 1])
        if a == b:
            continue
        put("dx", slice(a, b), dh[a:b], W1[e])               # G2: dh W1_e^T over the expert's tile rows
        put("dW1", e, x_t[:, a:b], dh_t[:, a:b])             # G4: x_g^T dh over its rows
        put("dW2", e, ap_t[:, a:b], dout_t[:, a:b])          # G3: a'^T dout_g over its rows
    assert np.count_nonzero(ref["dW1"][0][0]) == 0 and np.count_nonzero(np64(got["dW1"])[0]) == 0   # empty expert
    errs = {"G2_dx_expanded": _check("dx_expanded", dx_exp, *ref["dx"]),
            "G4_dW1": _check("dW1", np64(got["dW1"]), *ref["dW1"]),
            "G3_dW2": _check("dW2", np64(got["dW2"]), *ref["dW2"])}
    print({k: (f"{a:.2e}", f"{b:.3%}", f"{c:.2f}") for k, (a, b, c) in errs.items()})


def _deq_block(op, name, R, C, r0, nr, c0, nc, fmt):
    """Rows r0.. (nr) and columns c0.. (nc, a multiple of 32 from a multiple of 32) of region `name`
    ([R, C] codes, tiled scales with groups along C), dequantised; only that block leaves the GPU."""
    q = op.region(name).view(R, C)[r0:r0 + nr, c0:c0 + nc].cpu().numpy()
    r = torch.arange(r0, r0 + nr, device="cuda")[:, None]
    g = torch.arange(c0 // 32, (c0 + nc) // 32, device="cuda")[None, :]
    off = ((r // 128) * (C // 128) + (g * 32) // 128) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    sf = op.region(name + "_SF")[off].cpu().numpy()
    return omx.mx_dequantize(q, sf, fmt, axis=-1)


def test_mxfp8_store_gemms_on_their_own_operands_hot_expert_full_size():
    """The imbalanced workload at full size: the hottest expert's contraction over all its tile rows
    (about 65k) for one 128 x 256 output tile of dW1 (across the gate/up boundary) and of dW2, and 256
    of its dx_expanded rows over the whole hidden dimension."""
    from moe_expert_layer_routing_gb300.inputs import CONFIGS
    cfg = CONFIGS["imbalanced_mxfp8"]
    inp = make_moe_inputs(cfg, device="cuda")
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    P, H, I, fa = op.tile_rows, cfg.H, cfg.I, cfg.fp8_act
    toff = op.region("TILE_OFFSETS").view(torch.int32).cpu().numpy()
    e = int(np.argmax(np.diff(toff)))
    a, b = int(toff[e]), int(toff[e + 1])
    assert b - a > 32768, "the hot expert holds the longest contraction"
    h0, j0, i0, c0 = 1920, I - 128, 640, 2048
    x_t = _deq_block(op, "X_GT", H, P, h0, 128, a, b - a, fa)
    dh_t = _deq_block(op, "DH_T", 2 * I, P, j0, 256, a, b - a, fa)
    ap_t = _deq_block(op, "AP_T", I, P, i0, 128, a, b - a, fa)
    dout_t = _deq_block(op, "DOUT_GT", H, P, c0, 256, a, b - a, fa)
    r0 = a + (b - a) // 2 // 128 * 128
    dh = _deq_block(op, "DH", P, 2 * I, r0, 256, 0, 2 * I, fa)
    W1q, W1s = omx.mx_quantize(inp.W1[e].double().cpu().numpy(), cfg.fp8_w, axis=-1)   # [H, 2I]
    W1e = omx.mx_dequantize(W1q, W1s, cfg.fp8_w, axis=-1)
    dx_exp = np64(op.region("DX_EXP").view(torch.bfloat16).reshape(P, H)[r0:r0 + 256])
    def contract(A, B):
        return A @ B.T, np.abs(A) @ np.abs(B).T

    errs = {"G4_dW1": _check("dW1 tile", np64(got["dW1"][e, h0:h0 + 128, j0:j0 + 256]), *contract(x_t, dh_t)),
            "G3_dW2": _check("dW2 tile", np64(got["dW2"][e, i0:i0 + 128, c0:c0 + 256]), *contract(ap_t, dout_t)),
            "G2_dx_expanded": _check("dx_expanded rows", dx_exp, *contract(dh, W1e))}
    print(f"expert {e}, {b - a} tile rows:",
          {k: (f"{u:.2e}", f"{v:.3%}", f"{w:.2f}") for k, (u, v, w) in errs.items()})


@pytest.mark.parametrize("mn", [1, 0])
@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
def test_bf16_store_gemms_on_their_own_operands(affinity, mn, set_option):
    """BF16: the GEMMs' operands as the GPU wrote them -- row-major x_g, dh, a' and dout_g read through
    the MN-major layout (MN_OPERANDS = 1), or their transposed copies (0) -- contracted in float64 and
    compared with dx_expanded, dW1 and dW2 the same way as the MXFP8 ones."""
    from moe_expert_layer_routing_gb300.inputs import PREC_BF16
    set_option("MN_OPERANDS", mn)
    cfg = small_moe("bf16_l1", T=700, H=384, I=256, E=6, K=2, B=256, seed=37, precision=PREC_BF16,
                    affinity=affinity)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(700, 2, 6, seed=9))
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    P, H, I = op.tile_rows, cfg.H, cfg.I
    toff = op.region("TILE_OFFSETS").view(torch.int32).cpu().numpy()
    used = int(toff[cfg.E])

    def rows(name, cols):   # [used, cols] token rows: the row-major region, or the transposed copy
        r = op.region(name).view(torch.bfloat16)
        return np64(r.reshape(P, cols)[:used] if mn else r.reshape(cols, P)[:, :used].T)

    dh = np64(op.region("DH").view(torch.bfloat16).reshape(P, 2 * I))[:used]
    dh_w = dh if mn else rows("DH_T", 2 * I)     # the dW1 GEMM's B operand
    x = rows("X_GT", H)
    ap = rows("AP_T", I)
    # the dW2 GEMM's B operand: dout_g itself with MN-major operands (s moved to a' for affinity on
    # H), else the transposed copy (s-scaled for affinity on H)
    dout = np64(op.region("DOUT_G").view(torch.bfloat16).reshape(P, H))[:used] if mn else rows("DOUT_GT", H)
    W1 = np64(inp.W1)
    dx_exp = np64(op.region("DX_EXP").view(torch.bfloat16).reshape(P, H))[:used]
    ref = {n: (np.zeros(shape), np.zeros(shape)) for n, shape in
           (("dx", (used, H)), ("dW1", (cfg.E, H, 2 * I)), ("dW2", (cfg.E, I, H)))}

    def put(n, idx, A, B):
        ref[n][0][idx] = A @ B.T
        ref[n][1][idx] = np.abs(A) @ np.abs(B).T

    for e in range(cfg.E):
        a, b = int(toff[e]), int(toff[e + 1])
        if a == b:
            continue
        put("dx", slice(a, b), dh[a:b], W1[e])
        put("dW1", e, x[a:b].T, dh_w[a:b].T)
        put("dW2", e, ap[a:b].T, dout[a:b].T)
    errs = {"G2_dx_expanded": _check("dx_expanded", dx_exp, *ref["dx"]),
            "G4_dW1": _check("dW1", np64(got["dW1"]), *ref["dW1"]),
            "G3_dW2": _check("dW2", np64(got["dW2"]), *ref["dW2"])}
    print({k: (f"{a:.2e}", f"{b:.3%}", f"{c:.2f}") for k, (a, b, c) in errs.items()})


# ---------------------------------------------------------------------------------------------------
# G1: dA_raw = dout_g W2_e^T on the dout rows the GPU gathered (and quantised), then the dSwiGLU
# epilogue written out in float64 on the same checkpoint values
# ---------------------------------------------------------------------------------------------------

def _fp8_ordered(c: np.ndarray) -> np.ndarray:
    """FP8 codes (sign-magnitude bytes) as integers in the order of their values."""
    c = c.astype(np.int64)
    return np.where(c < 0x80, c, 0x80 - c)


def _g1_reference(inp, op, mx):
    """Per used tile row: the float64 dA_raw from the GPU's own A operand and the weights (quantised by
    the oracle for MXFP8), its magnitude sum |dout_g| |W2_e|^T, and the row's gate, up and s."""
    from helpers import oracle_h, oracle_meta
    cfg = inp.cfg
    P, H, I = op.tile_rows, cfg.H, cfg.I
    toff = op.region("TILE_OFFSETS").view(torch.int32).cpu().numpy()
    used = int(toff[cfg.E])
    flat = op.region("TILE_ROW_FLAT").view(torch.int32).cpu().numpy()[:used]
    valid = flat >= 0
    t, k = np.where(valid, flat // cfg.K, 0), np.where(valid, flat % cfg.K, 0)
    if mx:
        g = _deq(op, "DOUT_G", P, H, cfg.fp8_act)[:used]
        W2q, W2s = omx.mx_quantize(inp.W2.double().numpy(), cfg.fp8_w, axis=-1)   # [E, I, H], groups along H
        W2 = omx.mx_dequantize(W2q, W2s, cfg.fp8_w, axis=-1)
    else:
        g = np64(op.region("DOUT_G").view(torch.bfloat16).reshape(P, H))[:used]
        W2 = np64(inp.W2)
    dA_raw, mag = np.zeros((used, I)), np.zeros((used, I))
    for e in range(cfg.E):
        a, b = int(toff[e]), int(toff[e + 1])
        dA_raw[a:b] = g[a:b] @ W2[e].T
        mag[a:b] = np.abs(g[a:b]) @ np.abs(W2[e]).T
    h = oracle_h(inp, oracle_meta(inp))[t, k] * valid[:, None]
    s = inp.s.double().numpy()[t, k] * valid
    return dict(used=used, valid=valid, t=t, k=k, dA_raw=dA_raw, mag=mag, gate=h[:, :I], up=h[:, I:], s=s)


def _dswiglu(ref):
    """dh = [dgate | dup] in float64, and the factors that multiply dA_raw in each (for error terms)."""
    from oracle import moe as om
    gate, up, s = ref["gate"], ref["up"], ref["s"][:, None]
    cg, cu = s * up * om.dsilu(gate), s * om.silu(gate)
    return np.concatenate([cg * ref["dA_raw"], cu * ref["dA_raw"]], 1), np.concatenate([cg, cu], 1)


@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
def test_bf16_g1_epilogue_on_its_own_operands(affinity):
    """BF16 G1: dh within one bf16 ulp of the float64 dSwiGLU of the float64 dA_raw (plus the
    accumulation term and 2^-20 relative for the epilogue's fp32 SiLU), ds within 2^-16 of
    sum |dA_raw a| per slot."""
    from moe_expert_layer_routing_gb300.inputs import PREC_BF16
    from oracle import moe as om
    cfg = small_moe("g1_l1", T=700, H=384, I=256, E=6, K=2, B=256, seed=38, precision=PREC_BF16,
                    affinity=affinity)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(700, 2, 6, seed=10))
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    ref = _g1_reference(inp, op, mx=False)
    used, I = ref["used"], cfg.I
    dh_ref, coef = _dswiglu(ref)
    dh = np64(op.region("DH").view(torch.bfloat16).reshape(op.tile_rows, 2 * I))[:used]
    ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(dh_ref), 1e-300))).astype(np.int64) - 7)
    bound = ulp + ACC_EPS * np.abs(coef) * np.concatenate([ref["mag"]] * 2, 1) + 2.0 ** -20 * np.abs(dh_ref)
    excess = float(np.max(np.abs(dh - dh_ref) / bound))
    share = float(np.count_nonzero(_ordered(dh) != _ordered(dh_ref))) / dh.size
    assert excess <= 1.0 and share <= FLIP_SHARE, (excess, share)
    # ds[t, k] = <dA_raw, a> over the slot's row
    a = om.silu(ref["gate"]) * ref["up"]
    v = ref["valid"]
    ds_ref = np.zeros((cfg.T, cfg.K))
    ds_mag = np.zeros((cfg.T, cfg.K))
    ds_ref[ref["t"][v], ref["k"][v]] = np.sum(ref["dA_raw"] * a, 1)[v]
    ds_mag[ref["t"][v], ref["k"][v]] = (np.sum(np.abs(ref["dA_raw"] * a), 1) * 2.0 ** -16
                                        + ACC_EPS * np.sum(ref["mag"] * np.abs(a), 1))[v]
    ds = np64(got["ds"])
    ds_excess = float(np.max(np.abs(ds - ds_ref) / (ds_mag + 1e-300)))
    assert ds_excess <= 1.0, ds_excess
    print(f"dh: excess {excess:.2f}, {share:.3%} off the rounded result; ds: excess {ds_excess:.3f}")


@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
def test_mxfp8_g1_epilogue_on_its_own_operands(affinity):
    """MXFP8 G1: the float64 dh, and a' = (s) SiLU(gate) up, quantised by the oracle -- row-wise for dh
    (G2's operand), along 32 tile rows for dh^T and a'^T (G4's and G3's) -- against the GPU's codes and
    scales: scale bytes equal but for a few groups whose amax sits at a power of two, codes equal but
    for a small share one step apart (the GPU's fp32 value and the float64 one on the two sides of a
    rounding boundary)."""
    from oracle import moe as om
    cfg = small_moe("g1_l1_mx", T=700, H=384, I=256, E=6, K=2, B=256, seed=39, precision=PREC_MXFP8,
                    affinity=affinity)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(700, 2, 6, seed=11))
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    ref = _g1_reference(inp, op, mx=True)
    used, I, P, fa = ref["used"], cfg.I, op.tile_rows, cfg.fp8_act
    dh_ref, _ = _dswiglu(ref)
    a_ref = om.silu(ref["gate"]) * ref["up"] * (ref["s"][:, None] if affinity == AFFINITY_ON_I else 1.0)
    out = {}
    for name, vals, R, C, axis in (("DH", dh_ref, P, 2 * I, 1), ("DH_T", dh_ref, 2 * I, P, 0),
                                   ("AP_T", a_ref, I, P, 0)):
        q_ref, s_ref = omx.mx_quantize(vals, fa, axis=axis)        # [used, C'] codes, scales along axis
        q = op.region(name).cpu().numpy().reshape(R, C)
        sf = tiled_sf_to_plain(op.region(name + "_SF").cpu().numpy(), R, C)
        if axis == 0:   # transposed outputs: [features, tile rows]
            q, sf = q[:, :used].T, sf[:, :used // 32].T
        else:
            q, sf = q[:used], sf[:used]
        same_sf = sf == s_ref
        sf_share = 1.0 - float(np.count_nonzero(same_sf)) / same_sf.size
        same_group = np.repeat(same_sf, 32, axis=axis)
        d = np.abs(_fp8_ordered(q) - _fp8_ordered(q_ref))[same_group]
        steps, share = int(d.max()), float(np.count_nonzero(d)) / d.size
        out[name] = (f"{sf_share:.3%} scales, {share:.3%} codes, max {steps} step")
        assert sf_share <= 0.01 and steps <= 1 and share <= FLIP_SHARE, (name, out[name])
    print(out)
