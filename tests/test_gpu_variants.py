"""GPU parity of the layer variants: GeGLU (act = GELU with the exact normal CDF) and the interleaved
gate/up layout of W1 (gate_i at column 2i, up_i at 2i+1; dW1 and db1 follow), BF16 and MXFP8, against
the oracle on the same inputs; and the recomputed pre-activations with an interleaved W1."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, oracle_h, oracle_meta, to_device
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe, with_ids)
from oracle import moe as om

pytestmark = pytest.mark.gpu

VARIANTS = [("geglu", "concat"), ("swiglu", "interleaved"), ("geglu", "interleaved")]


def _ragged_ids(T, K, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(np.arange(1, E))[:K] for _ in range(T)])  # expert 0 empty
    return torch.from_numpy(ids.astype(np.int32))


def _gpu(inp, glu, layout, **extra):
    import moe_expert_layer_routing_gb300 as mb
    cfg = inp.cfg
    d = to_device(inp)
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size, precision=cfg.precision,
                   affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, has_bias=cfg.bias,
                   glu=mb.GLU_GEGLU if glu == "geglu" else mb.GLU_SWIGLU,
                   gate_up_layout=mb.GATE_UP_INTERLEAVED if layout == "interleaved" else mb.GATE_UP_CONCAT,
                   act_src=extra.pop("act_src", mb.ACT_CHECKPOINT))
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, b2=d.b2 if cfg.bias else None)
    if "W1t" not in extra:
        kw["ckpt"] = d.ckpt
    if cfg.precision == PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)   # groups along 2I in W1's own layout
        W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
        if "W1t" in extra:
            kw["W1t_q"], kw["W1t_sf"] = mb.quantize_weights(extra.pop("W1t").cuda(), cfg.fp8_w)
    else:
        kw.update(W1=d.W1, W2=d.W2)
        if "W1t" in extra:
            kw["W1t"] = extra.pop("W1t").cuda()
    op.bind(**kw).run()
    torch.cuda.synchronize()
    return op.outputs()


def _oracle(inp, h, glu, layout):
    cfg = inp.cfg
    ids = inp.ids.numpy()
    if cfg.precision == PREC_MXFP8:
        return om.moe_backward_mxfp8(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, affinity=cfg.affinity,
                                     fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, activation=glu, gate_up=layout)
    return om.moe_backward(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, b2=inp.b2, with_bias=cfg.bias,
                           activation=glu, gate_up=layout)


@pytest.mark.parametrize("glu,layout", VARIANTS)
def test_bf16_variants_with_bias(glu, layout):
    cfg = small_moe("var_bf16", T=300, H=256, I=384, E=5, K=2, B=256, seed=71, bias=True, affinity=AFFINITY_ON_H)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(300, 2, 5, seed=2))
    got = _gpu(inp, glu, layout)
    assert int(got["status"].item()) == 0
    compare_outputs(got, _oracle(inp, oracle_h(inp, oracle_meta(inp)), glu, layout), BF16_TOL)


@pytest.mark.parametrize("glu,layout", VARIANTS)
def test_mxfp8_variants(glu, layout):
    cfg = small_moe("var_mx", T=320, H=256, I=256, E=5, K=2, B=128, seed=72, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(320, 2, 5, seed=3))
    got = _gpu(inp, glu, layout)
    assert int(got["status"].item()) == 0
    compare_outputs(got, _oracle(inp, oracle_h(inp, oracle_meta(inp)), glu, layout), MXFP8_TOL)


@pytest.mark.parametrize("prec,tol", [(PREC_BF16, BF16_TOL), (PREC_MXFP8, MXFP8_TOL)])
def test_recompute_with_interleaved_w1(prec, tol):
    """W1 interleaved for the backward GEMMs; W1t (the recomputation operand) is [gate | up]."""
    import moe_expert_layer_routing_gb300 as mb
    cfg = small_moe("var_rec", T=256, H=256, I=256, E=4, K=2, B=128, seed=73, precision=prec,
                    affinity=AFFINITY_ON_I)
    inp = make_moe_inputs(cfg)
    gc, uc = om.gate_up_columns(cfg.I, "interleaved")
    order = torch.from_numpy(np.concatenate([gc, uc]))
    W1t = inp.W1[:, :, order].transpose(1, 2).contiguous()            # [E, 2I, H], rows [gate | up]
    got = _gpu(inp, "geglu", "interleaved", act_src=mb.ACT_RECOMPUTE, W1t=W1t)
    assert int(got["status"].item()) == 0
    h = om.recompute_h(inp.x, inp.W1[:, :, order], inp.ids.numpy(), mxfp8=prec == PREC_MXFP8,
                       fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w)
    compare_outputs(got, _oracle(inp, h, "geglu", "interleaved"), tol)
