"""GPU parity with [BW]'s optional checkpoints of the dW_down factors: intermediate_checkpoint_T
(a), scaled_intermediate_checkpoint_T (s*a, affinity on I) and down_proj_act_checkpoint (s*dout,
affinity on H), bf16 in the block layout, against the oracle given the same saved values."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, oracle_h, oracle_meta, to_device
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe)
from oracle import moe as om

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


def _slots(meta, T, K, B):
    """Block-layout slot of every (t, k) (-1 if unrouted)."""
    eo, bo = meta["expert_offsets"], meta["block_offsets"]
    E = len(eo) - 1
    er = np.repeat(np.arange(E), np.diff(eo))
    r = np.arange(int(eo[E]))
    slot = np.full(T * K, -1, dtype=np.int64)
    slot[meta["s_scatter_idx"]] = bo[er] * B + (r - eo[er])
    return slot.reshape(T, K)


def _feature_major(vals, slot, Nb, B):
    """[T,K,F] -> [Nb,F,B] (feature-major per block, like the gate/up checkpoint)."""
    F = vals.shape[2]
    out = np.zeros((Nb, F, B))
    t, k = np.nonzero(slot >= 0)
    sl = slot[t, k]
    out[sl // B, :, sl % B] = vals[t, k]
    return out


def _slot_major(vals, slot, Nb, B):
    """[T,K,F] -> [Nb,B,F] (one row per slot)."""
    F = vals.shape[2]
    out = np.zeros((Nb * B, F))
    t, k = np.nonzero(slot >= 0)
    out[slot[t, k]] = vals[t, k]
    return out.reshape(Nb, B, F)


CASES = [(PREC_BF16, AFFINITY_ON_H, ("inter", "sdout")), (PREC_BF16, AFFINITY_ON_H, ("inter",)),
         (PREC_BF16, AFFINITY_ON_H, ("sdout",)), (PREC_BF16, AFFINITY_ON_I, ("inter",)),
         (PREC_BF16, AFFINITY_ON_I, ("scaled",)), (PREC_MXFP8, AFFINITY_ON_I, ("scaled",)),
         (PREC_MXFP8, AFFINITY_ON_I, ("inter",)), (PREC_MXFP8, AFFINITY_ON_H, ("inter", "sdout"))]


@pytest.mark.parametrize("mn", [1, 0])
@pytest.mark.parametrize("prec,aff,saved", CASES)
def test_saved_dw_down_factors(prec, aff, saved, mn, set_option):
    """BF16 with and without MN-major weight-gradient operands (with them, a saved factor replaces the
    operand it stands for, and s moves to a' for affinity on H only when no saved s*dout carries it)."""
    import moe_expert_layer_routing_gb300 as mb
    if prec == PREC_MXFP8 and mn == 0:
        pytest.skip("MXFP8 builds the transposed operands either way")
    set_option("MN_OPERANDS", mn)
    bias = prec == PREC_BF16 and "sdout" in saved
    cfg = small_moe("saved", T=300, H=256, I=256, E=5, K=2, B=256, seed=81, precision=prec, affinity=aff, bias=bias)
    inp = make_moe_inputs(cfg)
    meta = oracle_meta(inp)
    h = oracle_h(inp, meta)
    T, K, I, B = cfg.T, cfg.K, cfg.I, cfg.block_size
    Nb = mb.num_blocks_bound(T, K, cfg.E, B)
    slot = _slots(meta, T, K, B)
    s = inp.s.double().numpy()
    a = np.asarray(_bf16(om.silu(h[..., :I]) * h[..., I:]).double())          # saved a (bf16)
    sa = np.asarray(_bf16(s[..., None] * a).double())                          # saved s*a (bf16)
    sd = np.asarray(_bf16(s[..., None] * inp.dout.double().numpy()[:, None, :]).double())  # saved s*dout
    d = to_device(inp)
    op = mb.MoeBwd(T=T, H=cfg.H, I=I, E=cfg.E, K=K, block_size=B, precision=prec, affinity=aff, fp8_act=cfg.fp8_act,
                   fp8_w=cfg.fp8_w, has_bias=bias)
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, b2=d.b2 if bias else None)
    if prec == PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)
        W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
    else:
        kw.update(W1=d.W1, W2=d.W2)
    inter = sdout = None
    if "inter" in saved:
        kw["intermediate_ckpt"] = _bf16(_feature_major(a, slot, Nb, B)).cuda()
        inter = om._to_f32(s[..., None] * a) if aff == AFFINITY_ON_I else a
    if "scaled" in saved:
        kw["scaled_intermediate_ckpt"] = _bf16(_feature_major(sa, slot, Nb, B)).cuda()
        inter = sa
    if "sdout" in saved:
        kw["down_proj_act_ckpt"] = _bf16(_slot_major(sd, slot, Nb, B)).cuda()
        sdout = sd
    op.bind(**kw).run()
    torch.cuda.synchronize()
    got = op.outputs()
    assert int(got["status"].item()) == 0
    ids = inp.ids.numpy()
    if prec == PREC_MXFP8:
        ref = om.moe_backward_mxfp8(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, affinity=aff, fp8_act=cfg.fp8_act,
                                    fp8_w=cfg.fp8_w, inter=inter, sdout=sdout)
        compare_outputs(got, ref, MXFP8_TOL)
    else:
        ref = om.moe_backward(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, b2=inp.b2 if bias else None,
                              with_bias=bias, affinity=aff, inter=inter, sdout=sdout)
        compare_outputs(got, ref, BF16_TOL)


def test_saved_factors_are_used():
    """A saved factor that differs from the recomputed one changes dW2 the way the oracle says."""
    import moe_expert_layer_routing_gb300 as mb
    cfg = small_moe("saved_used", T=256, H=256, I=256, E=4, K=2, B=128, seed=82, affinity=AFFINITY_ON_H)
    inp = make_moe_inputs(cfg)
    meta = oracle_meta(inp)
    h = oracle_h(inp, meta)
    T, K, I, B = cfg.T, cfg.K, cfg.I, cfg.block_size
    Nb = mb.num_blocks_bound(T, K, cfg.E, B)
    slot = _slots(meta, T, K, B)
    a2 = np.asarray(_bf16(2.0 * om.silu(h[..., :I]) * h[..., I:]).double())   # twice the true a
    d = to_device(inp)
    op = mb.MoeBwd(T=T, H=cfg.H, I=I, E=cfg.E, K=K, block_size=B, affinity=AFFINITY_ON_H)
    op.bind(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, W1=d.W1, W2=d.W2,
            intermediate_ckpt=_bf16(_feature_major(a2, slot, Nb, B)).cuda()).run()
    torch.cuda.synchronize()
    got = op.outputs()
    ref = om.moe_backward(inp.x, inp.dout, inp.W1, inp.W2, inp.s, inp.ids.numpy(), h, affinity=0, inter=a2)
    compare_outputs(got, ref, BF16_TOL)


GATE_ACT_CASES = [(PREC_BF16, AFFINITY_ON_H, "swiglu", "concat", 256, 1.0),
                  (PREC_BF16, AFFINITY_ON_I, "geglu", "interleaved", 256, 2.0),
                  (PREC_MXFP8, AFFINITY_ON_I, "swiglu", "concat", 384, 1.0),
                  (PREC_MXFP8, AFFINITY_ON_H, "geglu", "interleaved", 256, 2.0),
                  (PREC_MXFP8, AFFINITY_ON_I, "swiglu", "concat", 256, 2.0)]


@pytest.mark.parametrize("prec,aff,glu,layout,I,c", GATE_ACT_CASES)
def test_saved_gate_act(prec, aff, glu, layout, I, c):
    """[BW] gate_act_checkpoint_T: a saved act(gate) (c = 1: the forward's own, rounded to bf16; c = 2:
    a value the recomputation would not give) enters ds, a' and dup; the oracle gets the same values."""
    import moe_expert_layer_routing_gb300 as mb
    bias = prec == PREC_BF16
    cfg = small_moe("gact", T=300, H=256, I=I, E=5, K=2, B=256, seed=84, precision=prec, affinity=aff, bias=bias)
    inp = make_moe_inputs(cfg)
    meta = oracle_meta(inp)
    h = oracle_h(inp, meta)
    T, K, B = cfg.T, cfg.K, cfg.block_size
    Nb = mb.num_blocks_bound(T, K, cfg.E, B)
    slot = _slots(meta, T, K, B)
    ga = np.asarray(_bf16(c * om.ACTIVATIONS[glu][0](h[..., :I])).double())
    d = to_device(inp)
    op = mb.MoeBwd(T=T, H=cfg.H, I=I, E=cfg.E, K=K, block_size=B, precision=prec, affinity=aff, fp8_act=cfg.fp8_act,
                   fp8_w=cfg.fp8_w, has_bias=bias, glu=mb.GLU_GEGLU if glu == "geglu" else mb.GLU_SWIGLU,
                   gate_up_layout=mb.GATE_UP_INTERLEAVED if layout == "interleaved" else mb.GATE_UP_CONCAT)
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, b2=d.b2 if bias else None,
              gate_act_ckpt=_bf16(_feature_major(ga, slot, Nb, B)).cuda())
    if prec == PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)
        W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
    else:
        kw.update(W1=d.W1, W2=d.W2)
    op.bind(**kw).run()
    torch.cuda.synchronize()
    got = op.outputs()
    assert int(got["status"].item()) == 0
    ids = inp.ids.numpy()
    if prec == PREC_MXFP8:
        ref = om.moe_backward_mxfp8(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, affinity=aff, fp8_act=cfg.fp8_act,
                                    fp8_w=cfg.fp8_w, activation=glu, gate_up=layout, gate_act=ga)
        compare_outputs(got, ref, MXFP8_TOL)
    else:
        ref = om.moe_backward(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, b2=inp.b2, with_bias=True,
                              affinity=aff, activation=glu, gate_up=layout, gate_act=ga)
        compare_outputs(got, ref, BF16_TOL)
