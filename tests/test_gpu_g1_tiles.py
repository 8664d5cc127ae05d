"""GPU parity of the dSwiGLU GEMM (dA = dout_g W2_e^T with its epilogue) at both of its MXFP8 tile
widths: 192 columns (the default where I is a multiple of 192; W2's scales re-tiled into two atoms
per tile) and 128 (library option G1_TILE_N = 128), against the oracle on the same inputs, over ragged expert
loads, both activation formats, both affinity modes and the GeGLU / interleaved variant; and the two
widths agree on the quantised dh operand."""
import numpy as np
import pytest
import torch

from helpers import MXFP8_TOL, compare_outputs, oracle_bwd, oracle_h, oracle_meta, run_gpu, to_device
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, FP8_E4M3, FP8_E5M2, PREC_MXFP8,
                                                   make_moe_inputs, small_moe, with_ids)
from oracle import moe as om

pytestmark = pytest.mark.gpu


def _ragged_ids(T, K, E, seed):
    """Expert 0 empty, expert 1 a single row, expert 2 hot."""
    rng = np.random.default_rng(seed)
    p = np.ones(E - 2)
    p[0] = 12.0
    p /= p.sum()
    ids = np.stack([rng.choice(np.arange(2, E), size=K, replace=False, p=p) for _ in range(T)])
    ids[0, K - 1] = 1
    return torch.from_numpy(ids.astype(np.int32))


@pytest.mark.parametrize("warps", [16, 8])
@pytest.mark.parametrize("bn", [192, 128])
@pytest.mark.parametrize("I", [384, 768])
@pytest.mark.parametrize("fmt_act,aff", [(FP8_E5M2, AFFINITY_ON_I), (FP8_E4M3, AFFINITY_ON_H)])
def test_mxfp8_g1_tile_widths(set_option, bn, I, fmt_act, aff, warps):
    """Both G1 tile widths with eight epilogue warps or sixteen (two groups taking alternate chunks)."""
    set_option("G1_TILE_N", bn)
    set_option("G1_WARPS", warps)
    cfg = small_moe("g1w", T=520, H=256, I=I, E=6, K=2, B=256, seed=91, precision=PREC_MXFP8, affinity=aff,
                    fp8_act=fmt_act)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(520, 2, 6, seed=11))
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    compare_outputs(got, oracle_bwd(inp), MXFP8_TOL)


@pytest.mark.parametrize("warps", [16, 8])
def test_mxfp8_g1_variant_at_192(set_option, warps):
    """GeGLU with the interleaved gate/up layout through the 192-column tiles."""
    import moe_expert_layer_routing_gb300 as mb
    set_option("G1_TILE_N", 192)
    set_option("G1_WARPS", warps)
    cfg = small_moe("g1v", T=400, H=256, I=384, E=5, K=2, B=128, seed=92, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(400, 2, 5, seed=12))
    d = to_device(inp)
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size, precision=PREC_MXFP8,
                   affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, glu=mb.GLU_GEGLU,
                   gate_up_layout=mb.GATE_UP_INTERLEAVED)
    W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)
    W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
    op.bind(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q,
            W2_sf=W2_sf).run()
    torch.cuda.synchronize()
    got = op.outputs()
    assert int(got["status"].item()) == 0
    h = oracle_h(inp, oracle_meta(inp))
    ref = om.moe_backward_mxfp8(inp.x, inp.dout, inp.W1, inp.W2, inp.s, inp.ids.numpy(), h, affinity=cfg.affinity,
                                fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, activation="geglu", gate_up="interleaved")
    compare_outputs(got, ref, MXFP8_TOL)


@pytest.mark.parametrize("warps", [16, 8])
def test_g1_widths_agree_on_dh(set_option, warps):
    """The quantised dh of the two tile widths: each output element's contraction is the same, so the
    codes and scales agree except where fp32 accumulation order moves a value across a rounding
    boundary (none expected; at most a handful allowed)."""
    cfg = small_moe("g1agree", T=384, H=512, I=768, E=4, K=2, B=128, seed=93, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = make_moe_inputs(cfg)
    outs = {}
    set_option("G1_WARPS", warps)
    for bn in (192, 128):
        set_option("G1_TILE_N", bn)
        op, got = run_gpu(inp)
        assert int(got["status"].item()) == 0
        used = int(op.region("TILE_OFFSETS").view(torch.int32)[cfg.E].item())
        dh = op.region("DH").cpu().numpy().reshape(op.tile_rows, 2 * cfg.I)[:used]
        outs[bn] = (dh.copy(), got["ds"].double().cpu().numpy())
    diff = np.count_nonzero(outs[192][0] != outs[128][0])
    assert diff <= outs[128][0].size * 1e-4, diff
    ds192, ds128 = outs[192][1], outs[128][1]   # partial sums per tile width: summation order differs
    np.testing.assert_allclose(ds192, ds128, rtol=1e-4, atol=1e-5 * np.abs(ds128).max())


def test_g1_eight_and_sixteen_epilogue_warps_are_bit_identical(set_option):
    """The two epilogue layouts compute every element the same way (only the ds partials are summed in
    another grouping): dx, dW1, dW2 bit-identical, ds to fp32 rounding."""
    import torch
    cfg = small_moe("g1warps", T=600, H=512, I=384, E=6, K=2, B=256, seed=94, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I, bias=True)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(600, 2, 6, seed=13))
    outs = {}
    for warps in (16, 8):
        set_option("G1_WARPS", warps)
        _, got = run_gpu(inp)
        assert int(got["status"].item()) == 0
        outs[warps] = {k: v.clone() for k, v in got.items() if v is not None}
    for n in ("dx", "dW1", "dW2", "db1", "db2"):
        assert torch.equal(outs[16][n], outs[8][n]), n
    torch.testing.assert_close(outs[16]["ds"], outs[8]["ds"], rtol=1e-5, atol=1e-6)
