"""GPU parity of the MoE backward (BF16 and MXFP8) and the dense linear backward against the oracle,
at sizes the oracle finishes in seconds: several 128-row tiles, ragged expert loads, empty experts,
single-row experts, invalid ids, both affinity modes, biases, both N-tile widths."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from helpers import (BF16_TOL, MXFP8_TOL, compare_outputs, np64, oracle_bwd, oracle_h, oracle_meta,
                     rel_fro, run_gpu, tiled_sf_to_plain)
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, CONFIGS, PREC_MXFP8,
                                                   make_linear_inputs, make_moe_inputs, small_moe, with_ids,
                                                   LinearConfig)
from oracle import linear as olin
from oracle import mxfp8 as omx

pytestmark = pytest.mark.gpu


def _ragged_ids(T, K, E, seed, empty=(0,), single=(1,), hot=None):
    rng = np.random.default_rng(seed)
    allowed = [e for e in range(E) if e not in empty and e not in single]
    p = np.ones(len(allowed))
    if hot is not None:
        p[allowed.index(hot)] = 20.0
    p /= p.sum()
    ids = np.stack([rng.choice(allowed, size=K, replace=False, p=p) for _ in range(T)])
    for i, e in enumerate(single):
        ids[i, K - 1] = e
    return torch.from_numpy(ids.astype(np.int32))


def _check(inp, tol):
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0, f"device status {int(got['status'].item())}"
    ref = oracle_bwd(inp)
    return compare_outputs(got, ref, tol)


def test_tiny_bf16_config():
    _check(make_moe_inputs(CONFIGS["tiny_bf16"]), BF16_TOL)


@pytest.mark.parametrize("mn", [1, 0])
@pytest.mark.parametrize("affinity", [AFFINITY_ON_H, AFFINITY_ON_I])
@pytest.mark.parametrize("I", [384, 256])
def test_bf16_bias_ragged(affinity, I, mn, set_option):
    """BF16 with biases over ragged experts, 128- and 256-column G1 tiles; the dW1 GEMM reading dh as an
    MN-major operand (db1 from the dA epilogue's butterfly column sums) or through dh^T (db1 from the
    transposes)."""
    set_option("MN_OPERANDS", mn)
    cfg = small_moe("ragged_bias", T=300, H=256, I=I, E=8, K=3, B=256, seed=21, bias=True, affinity=affinity)
    inp = make_moe_inputs(cfg)
    inp = with_ids(inp, _ragged_ids(300, 3, 8, seed=5, hot=2))
    _check(inp, BF16_TOL)


@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
@pytest.mark.parametrize("I", [384, 256])
def test_mxfp8_bias_ragged(affinity, I):
    """MXFP8 with biases: db1 and db2 (sums of the unquantised dh and s*dout) and the <dout, b2> term of
    ds, over ragged experts (an empty one, a single-row one, a hot one), 192- and 128-column G1 tiles."""
    cfg = small_moe("mx_bias", T=300, H=256, I=I, E=8, K=3, B=256, seed=24, bias=True, precision=PREC_MXFP8,
                    affinity=affinity)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(300, 3, 8, seed=6, hot=2))
    errs = _check(inp, MXFP8_TOL)
    assert {"db1", "db2"} <= set(errs)


def test_bf16_single_expert_top1():
    cfg = small_moe("dense_like", T=200, H=384, I=128, E=1, K=1, B=128, seed=22)
    _check(make_moe_inputs(cfg), BF16_TOL)


def test_bf16_many_tiles_wide_hidden():
    cfg = small_moe("wide", T=700, H=640, I=256, E=6, K=2, B=512, seed=23)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(700, 2, 6, seed=7, empty=(3,), single=(), hot=0))
    _check(inp, BF16_TOL)


def test_bf16_invalid_ids_are_reported_and_skipped():
    cfg = small_moe("bad_ids", T=128, H=128, I=128, E=4, K=2, B=128, seed=24)
    inp = make_moe_inputs(cfg)
    ids = inp.ids.clone()
    ids[5, 0] = 4
    ids[9, 1] = -3
    inp = with_ids(inp, ids)
    op, got = run_gpu(inp)
    import moe_expert_layer_routing_gb300 as mb
    assert int(got["status"].item()) == mb.STATUS_BAD_EXPERT_ID
    ref = oracle_bwd(inp)
    compare_outputs(got, ref, BF16_TOL)
    assert float(got["ds"][5, 0]) == 0.0 and float(got["ds"][9, 1]) == 0.0


@pytest.mark.parametrize("gather", [1, 0])
def test_bf16_intermediates_match_oracle(gather, set_option):
    """dh and the gathered operands in the workspace match the oracle's own values (G1 gathering its
    dout rows itself, or reading the gathered copy)."""
    set_option("G1_GATHER", gather)
    inp = make_moe_inputs(CONFIGS["tiny_bf16"])
    op, got = run_gpu(inp)
    meta = oracle_meta(inp)
    cfg = inp.cfg
    h = oracle_h(inp, meta)
    P = op.tile_rows
    used = int(op.region("TILE_OFFSETS").view(torch.int32)[cfg.E].item())   # rows of the used tiles
    flat = op.region("TILE_ROW_FLAT").view(torch.int32).cpu().numpy()[:used]
    valid = flat >= 0
    t, k = flat[valid] // cfg.K, flat[valid] % cfg.K
    if gather:   # no gathered copy: G1 reads dout's rows
        assert op.region("DOUT_G").numel() == 0
    else:
        dout_g = op.region("DOUT_G").view(torch.bfloat16).reshape(P, cfg.H).cpu()[:used]
        assert torch.equal(dout_g[torch.from_numpy(valid)], inp.dout[torch.from_numpy(t)])
        assert torch.all(dout_g[torch.from_numpy(~valid)] == 0)
    # BF16: the dW1 GEMM reads x's gathered rows MN-major (held in the X_GT region), padding rows zero
    x_rows = op.region("X_GT").view(torch.bfloat16).reshape(P, cfg.H).cpu()[:used]
    assert torch.equal(x_rows[torch.from_numpy(valid)], inp.x[torch.from_numpy(t)])
    assert torch.all(x_rows[torch.from_numpy(~valid)] == 0)
    # dh from the oracle's formulas
    from oracle import moe as om
    x, dout, W2, s = map(om._f64, (inp.x, inp.dout, inp.W2, inp.s))
    ids = inp.ids.numpy()
    e = ids[t, k]
    g = dout[t]
    dA_raw = np.einsum("rh,rih->ri", g, W2[e])
    gate, up = h[t, k, :cfg.I], h[t, k, cfg.I:]
    dA = s[t, k][:, None] * dA_raw
    dh_ref = np.concatenate([dA * up * om.dsilu(gate), dA * om.silu(gate)], 1)
    dh = np64(op.region("DH").view(torch.bfloat16).reshape(P, 2 * cfg.I))[:used]
    assert rel_fro(dh[valid], dh_ref) < BF16_TOL
    assert np.all(dh[~valid] == 0)
    assert op.region("DH_T").numel() == 0  # BF16: the dW1 GEMM reads dh itself (MN-major), no dh^T


# ----------------------------------------------------------------------------------------------
# MXFP8
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
def test_mxfp8_small(affinity):
    cfg = small_moe("mx_small", T=256, H=256, I=256, E=4, K=2, B=256, seed=31, precision=PREC_MXFP8,
                    affinity=affinity)
    _check(make_moe_inputs(cfg), MXFP8_TOL)


def test_mxfp8_ragged_many_tiles():
    cfg = small_moe("mx_ragged", T=900, H=384, I=384, E=8, K=3, B=512, seed=32, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(900, 3, 8, seed=9, empty=(0, 6), single=(1,), hot=3))
    _check(inp, MXFP8_TOL)


@pytest.mark.parametrize("gather", [1, 0])
def test_mxfp8_quantised_operands_match_oracle_codes(gather, set_option):
    """G1's dout operand is quantised bit-exactly: per token (the rows G1 gathers) or as the gathered
    copy, with the gathered tiled scales either way."""
    set_option("G1_GATHER", gather)
    cfg = small_moe("mx_codes", T=256, H=256, I=256, E=4, K=2, B=256, seed=33, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = make_moe_inputs(cfg)
    op, got = run_gpu(inp)
    P = op.tile_rows
    used = int(op.region("TILE_OFFSETS").view(torch.int32)[cfg.E].item())
    flat = op.region("TILE_ROW_FLAT").view(torch.int32).cpu().numpy()[:used]
    valid = flat >= 0
    t = flat // cfg.K
    rows = np.where(valid[:, None], inp.dout.double().numpy()[np.where(valid, t, 0)], 0.0)
    rq, rs = omx.mx_quantize(rows, cfg.fp8_act, axis=1)
    sf = tiled_sf_to_plain(op.region("DOUT_G_SF").cpu().numpy(), P, cfg.H)[:used]
    assert np.array_equal(sf, rs)
    if gather:
        tq, _ = omx.mx_quantize(inp.dout.double().numpy(), cfg.fp8_act, axis=1)
        assert op.region("DOUT_G").numel() == 0
        assert np.array_equal(op.region("DOUT_Q").cpu().numpy().reshape(cfg.T, cfg.H), tq)
    else:
        q = op.region("DOUT_G").cpu().numpy().reshape(P, cfg.H)[:used]
        assert np.array_equal(q, rq)


@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
def test_mxfp8_transposed_operands_match_oracle_codes(affinity):
    """The token-quantised transposed operands of the weight-gradient GEMMs (x_g^T for dW1, dout_g^T
    for dW2, s-scaled in fp32 for affinity on H) are bit-exact: codes and scales of groups of 32 tile
    rows, against the oracle's quantisation along the row axis."""
    cfg = small_moe("mx_tcodes", T=300, H=384, I=256, E=5, K=2, B=256, seed=34, precision=PREC_MXFP8,
                    affinity=affinity)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(300, 2, 5, seed=4, empty=(0,), single=(1,), hot=2))
    op, got = run_gpu(inp)
    P = op.tile_rows
    used = int(op.region("TILE_OFFSETS").view(torch.int32)[cfg.E].item())
    flat = op.region("TILE_ROW_FLAT").view(torch.int32).cpu().numpy()[:used]
    valid = flat >= 0
    t, k = np.where(valid, flat // cfg.K, 0), np.where(valid, flat % cfg.K, 0)
    xrows = np.where(valid[:, None], inp.x.double().numpy()[t], 0.0)
    drows = np.where(valid[:, None], inp.dout.double().numpy()[t], 0.0)
    if affinity == AFFINITY_ON_H:  # s * dout rounded to fp32, as the kernel computes it
        drows = (drows * inp.s.double().numpy()[t, k][:, None]).astype(np.float32).astype(np.float64)
    for name, rows in (("X_GT", xrows), ("DOUT_GT", drows)):
        rq, rs = omx.mx_quantize(rows, cfg.fp8_act, axis=0)
        q = op.region(name).cpu().numpy().reshape(cfg.H, P)[:, :used].T
        sf = tiled_sf_to_plain(op.region(name + "_SF").cpu().numpy(), cfg.H, P)[:, :used // 32].T
        assert np.array_equal(q, rq), name
        assert np.array_equal(sf, rs), name


def test_linear_bwd_small_both_precisions():
    import moe_expert_layer_routing_gb300 as mb
    inp = make_linear_inputs(LinearConfig("lin_small", M=256, N=384, K=512, seed=41))
    for prec, tol, fn in ((mb.PREC_MXFP8, MXFP8_TOL, olin.linear_backward_mxfp8),
                          (mb.PREC_BF16, BF16_TOL, olin.linear_backward)):
        got = mb.linear_bwd(inp.dY.cuda(), inp.W.cuda(), inp.X.cuda(), precision=prec)
        torch.cuda.synchronize()
        ref = fn(inp.dY, inp.W, inp.X)
        assert rel_fro(np64(got["dX"]), ref["dX"]) < tol
        assert rel_fro(np64(got["dW"]), ref["dW"]) < tol


@pytest.mark.parametrize("mn", [1, 0])
def test_linear_bwd_bf16_operand_layouts(mn, set_option):
    """BF16 linear backward reading dY, W and X themselves as MN-major operands (no copies), or through
    transposed copies; odd tile counts and 128-column tiles."""
    import moe_expert_layer_routing_gb300 as mb
    set_option("MN_OPERANDS", mn)
    inp = make_linear_inputs(LinearConfig("lin_mn", M=384, N=256, K=640, seed=43))
    got = mb.linear_bwd(inp.dY.cuda(), inp.W.cuda(), inp.X.cuda(), precision=mb.PREC_BF16)
    torch.cuda.synchronize()
    ref = olin.linear_backward(inp.dY, inp.W, inp.X)
    assert rel_fro(np64(got["dX"]), ref["dX"]) < BF16_TOL
    assert rel_fro(np64(got["dW"]), ref["dW"]) < BF16_TOL


def test_linear_bwd_outputs_16_byte_aligned():
    """Outputs in caller buffers that are 16- but not 32-byte aligned (the public contract), through
    the direct-store epilogue (K = 384: 128-column tiles): identical to aligned outputs."""
    import moe_expert_layer_routing_gb300 as mb
    inp = make_linear_inputs(LinearConfig("lin_align", M=256, N=256, K=384, seed=43))
    dY, W, X = inp.dY.cuda(), inp.W.cuda(), inp.X.cuda()
    ref = mb.linear_bwd(dY, W, X, precision=mb.PREC_MXFP8)
    op = mb.LinearBwd(256, 256, 384, mb.PREC_MXFP8, device="cuda")
    views = []
    for rows in (256, 256):
        buf = torch.zeros(rows * 384 + 32, dtype=torch.bfloat16, device="cuda")
        off = ((32 - buf.data_ptr() % 32) % 32 + 16) // 2   # elements to 16 bytes past a 32-byte boundary
        views.append(buf[off:off + rows * 384].view(rows, 384))
    op.dX, op.dW = views
    assert op.dX.data_ptr() % 32 == 16 and op.dW.data_ptr() % 32 == 16
    op.run(dY, W, X)
    torch.cuda.synchronize()
    assert torch.equal(op.dX, ref["dX"]) and torch.equal(op.dW, ref["dW"])


def test_linear_bwd_dense_4096_config():
    """The dense MXFP8 workload at full size (oracle float64 matmuls of 4096^3)."""
    import moe_expert_layer_routing_gb300 as mb
    inp = make_linear_inputs(CONFIGS["dense_mxfp8_4096"], device="cuda")
    got = mb.linear_bwd(inp.dY, inp.W, inp.X, precision=mb.PREC_MXFP8)
    torch.cuda.synchronize()
    ref = olin.linear_backward_mxfp8(inp.dY.cpu(), inp.W.cpu(), inp.X.cpu())
    assert rel_fro(np64(got["dX"]), ref["dX"]) < MXFP8_TOL
    assert rel_fro(np64(got["dW"]), ref["dW"]) < MXFP8_TOL


@pytest.mark.parametrize("mx", [False, True])
def test_accumulate_adds_weight_and_bias_gradients(mx):
    """accumulate=1: dW1, dW2 (and db1, db2) are added to their previous contents, here twice in a
    row onto a random start; dx and ds are overwritten.  Tolerance: the path's bar plus the bf16
    rounding of the accumulated sums (measured against the size of the added gradients)."""
    import moe_expert_layer_routing_gb300 as mb
    from helpers import to_device
    if mx:
        cfg = small_moe("acc_mx", T=300, H=256, I=256, E=4, K=2, B=256, seed=41, precision=PREC_MXFP8,
                        affinity=AFFINITY_ON_I, bias=True)
    else:
        cfg = small_moe("acc_bf16", T=300, H=256, I=384, E=6, K=2, B=128, seed=42, bias=True)
    inp = make_moe_inputs(cfg)
    ref = oracle_bwd(inp)
    d = to_device(inp)
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size, precision=cfg.precision,
                   affinity=cfg.affinity, has_bias=cfg.bias, accumulate=True)
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, b2=d.b2 if cfg.bias else None)
    if mx:
        W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)
        W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
    else:
        kw.update(W1=d.W1, W2=d.W2)
    op.bind(**kw)
    g = torch.Generator().manual_seed(5)
    names = ["dW1", "dW2"] + (["db1", "db2"] if cfg.bias else [])
    init = {}
    for n in names:
        t = getattr(op, n)
        scale = float(np.std(ref[n])) if np.std(ref[n]) > 0 else 1.0
        init[n] = (torch.randn(t.shape, generator=g) * scale).to(t.dtype)
        t.copy_(init[n].cuda())
    op.run()
    op.run()
    torch.cuda.synchronize()
    assert int(op.status.item()) == 0
    tol = (MXFP8_TOL if mx else BF16_TOL) + 4e-3
    for n in names:
        got = np64(getattr(op, n)) - init[n].double().numpy()
        assert rel_fro(got, 2 * ref[n]) < tol, n
    assert rel_fro(np64(op.dx), ref["dx"]) < (MXFP8_TOL if mx else BF16_TOL)
