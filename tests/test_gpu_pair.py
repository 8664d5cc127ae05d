"""GPU parity of the CTA-pair GEMMs (cta_group::2, 256 x 256 per pair) and of the single-CTA GEMMs
they replace, on the same problems: shapes where every store GEMM (dW2, dx_expanded, dW1) can pair,
experts with an odd number of 128-row tiles (the last tile's partner idles), an empty expert (zero
contraction), a single-row expert; the dense linear backward with an odd tile count; and the
recomputed pre-activations (checkpoint epilogue)."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, np64, oracle_bwd, rel_fro, run_gpu
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   LinearConfig, make_linear_inputs, make_moe_inputs, small_moe,
                                                   with_ids)
from oracle import linear as olin

pytestmark = pytest.mark.gpu


def _ids(T, K, E, seed):
    """Expert 0 empty, expert 1 a single row, expert 2 hot (an odd tile count is likely), rest uniform."""
    rng = np.random.default_rng(seed)
    allowed = list(range(2, E))
    p = np.ones(len(allowed))
    p[0] = 9.0
    p /= p.sum()
    ids = np.stack([rng.choice(allowed, size=K, replace=False, p=p) for _ in range(T)])
    ids[0, K - 1] = 1
    return torch.from_numpy(ids.astype(np.int32))


# PAIR_GEMMS: 2 pairs for both precisions (the MXFP8 default is the single-CTA kernel), 0 none
@pytest.mark.parametrize("pair", [2, 0])
@pytest.mark.parametrize("prec,aff", [(PREC_BF16, AFFINITY_ON_H), (PREC_MXFP8, AFFINITY_ON_I)])
def test_moe_bwd_pair_and_single_cta(pair, prec, aff, set_option):
    set_option("PAIR_GEMMS", pair)
    cfg = small_moe("pair", T=700, H=512, I=256, E=6, K=2, B=256, seed=51, precision=prec, affinity=aff)
    inp = with_ids(make_moe_inputs(cfg), _ids(700, 2, 6, seed=9))
    counts = np.bincount(inp.ids.numpy().reshape(-1), minlength=6)
    tiles = (counts + 127) // 128
    assert counts[0] == 0 and counts[1] == 1 and np.any(tiles % 2 == 1)
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    compare_outputs(got, oracle_bwd(inp), MXFP8_TOL if prec == PREC_MXFP8 else BF16_TOL)


@pytest.mark.parametrize("pair", [2, 0])
def test_linear_bwd_odd_tiles_pair_and_single_cta(pair, set_option):
    import moe_expert_layer_routing_gb300 as mb
    set_option("PAIR_GEMMS", pair)
    inp = make_linear_inputs(LinearConfig("lin_odd", M=384, N=512, K=768, seed=52))
    for prec, tol, fn in ((mb.PREC_MXFP8, MXFP8_TOL, olin.linear_backward_mxfp8),
                          (mb.PREC_BF16, BF16_TOL, olin.linear_backward)):
        got = mb.linear_bwd(inp.dY.cuda(), inp.W.cuda(), inp.X.cuda(), precision=prec)
        torch.cuda.synchronize()
        ref = fn(inp.dY, inp.W, inp.X)
        assert rel_fro(np64(got["dX"]), ref["dX"]) < tol
        assert rel_fro(np64(got["dW"]), ref["dW"]) < tol


@pytest.mark.parametrize("bn", [256, 128])
def test_pair_and_single_cta_give_the_same_gradients_to_rounding(bn, set_option):
    """The two GEMM paths differ only in the order of the fp32 sums: their bf16 outputs agree to a
    few bf16 ulps relative to the gradient's size."""
    set_option("PAIR_TILE_N", bn)
    cfg = small_moe("pair_eq", T=512, H=512, I=256, E=4, K=2, B=128, seed=53, precision=PREC_MXFP8)
    inp = make_moe_inputs(cfg)
    outs = []
    for pair in (2, 0):
        set_option("PAIR_GEMMS", pair)
        _, got = run_gpu(inp)
        outs.append({k: np64(v) for k, v in got.items() if v is not None and k != "status"})
    for n in ("dx", "dW1", "dW2", "ds"):
        a, b = outs[0][n], outs[1][n]
        assert np.linalg.norm(a - b) <= 4e-3 * np.linalg.norm(b), n


@pytest.mark.parametrize("mn", [1, 0])
@pytest.mark.parametrize("pair", [2, 0])
def test_bf16_128_column_weight_gradient_tiles(pair, mn, set_option):
    """BF16 weight-gradient GEMMs at 128 columns — pair tiles of 128 (one 64-column box of an MN-major
    B per CTA) or single-CTA tiles of 128 (two boxes) — with MN-major and with transposed operands."""
    set_option("PAIR_GEMMS", pair)
    set_option("MN_OPERANDS", mn)
    if pair:
        set_option("PAIR_TILE_N", 128)
    else:
        set_option("G3_TILE_N", 128)
        set_option("G4_TILE_N", 128)
    cfg = small_moe("wgrad128", T=700, H=512, I=256, E=6, K=2, B=256, seed=54, precision=PREC_BF16,
                    affinity=AFFINITY_ON_H)
    inp = with_ids(make_moe_inputs(cfg), _ids(700, 2, 6, seed=10))
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    compare_outputs(got, oracle_bwd(inp), BF16_TOL)
