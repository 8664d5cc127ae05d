"""GPU parity of the recomputed gate/up pre-activations (act_src RECOMPUTE): the forward grouped GEMM
h = x_g W1_e + b1_e that moe_bwd runs in place of reading the [N,2,I,B] checkpoint, and the whole
backward built on it, against the oracle's recompute_h and backward on the same inputs."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, np64, oracle_meta, to_device
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe, with_ids)
from oracle import moe as om
from oracle import route_meta as orm

pytestmark = pytest.mark.gpu


def _ragged_ids(T, K, E, seed):
    """Expert 0 empty, expert 1 a single row, expert 2 hot; the rest uniform."""
    rng = np.random.default_rng(seed)
    allowed = list(range(2, E))
    p = np.ones(len(allowed))
    p[0] = 12.0
    p /= p.sum()
    ids = np.stack([rng.choice(allowed, size=K, replace=False, p=p) for _ in range(T)])
    ids[0, K - 1] = 1
    return torch.from_numpy(ids.astype(np.int32))


def _bf16_ulp(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def _run(inp, precision, has_bias, use_b1):
    import moe_expert_layer_routing_gb300 as mb
    cfg = inp.cfg
    d = to_device(inp)
    W1t = d.W1.transpose(1, 2).contiguous()                 # [E, 2I, H]
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size, precision=precision,
                   affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, has_bias=has_bias,
                   act_src=mb.ACT_RECOMPUTE)
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, b2=d.b2 if has_bias else None, b1=d.b1 if use_b1 else None)
    if precision == PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)
        W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
        W1t_q, W1t_sf = mb.quantize_weights(W1t, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf, W1t_q=W1t_q, W1t_sf=W1t_sf)
    else:
        kw.update(W1=d.W1, W2=d.W2, W1t=W1t)
    op.bind(**kw).run()
    torch.cuda.synchronize()
    return op, op.outputs()


def _check(inp, precision, has_bias, use_b1, tol):
    cfg = inp.cfg
    mx = precision == PREC_MXFP8
    op, got = _run(inp, precision, has_bias, use_b1)
    assert int(got["status"].item()) == 0
    ids = inp.ids.numpy()
    b1 = inp.b1 if use_b1 else None
    h = om.recompute_h(inp.x, inp.W1, ids, b1=b1, mxfp8=mx, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w)
    # 1. the recomputed checkpoint, read back from the workspace through the block layout
    meta = oracle_meta(inp)
    Nb = op.region("GATE_UP_CKPT").numel() // (2 * cfg.I * cfg.block_size * 2)
    ck = op.region("GATE_UP_CKPT").view(torch.bfloat16).reshape(Nb, 2, cfg.I, cfg.block_size)
    got_h = orm.checkpoint_rows(np64(ck), meta, cfg.T, cfg.K)
    routed = (ids >= 0) & (ids < cfg.E)
    diff = np.abs(got_h - h)[routed]
    # bound: one bf16 ulp of the result plus the fp32 dot-product error H * 2^-23 * sum |x| |W1_e|
    # (truncating accumulation; 1.25x covers the quantised operands' magnitudes under MXFP8)
    x64, W64 = np64(inp.x), np64(inp.W1)
    mag = np.zeros_like(h)
    for e in range(cfg.E):
        t, k = np.nonzero(ids == e)
        mag[t, k] = np.abs(x64[t]) @ np.abs(W64[e])
    bound = _bf16_ulp(h[routed]) + cfg.H * 2.0 ** -23 * 1.25 * mag[routed]
    assert np.all(diff <= bound), (float(np.max(diff / bound)), float(np.max(diff)), float(np.mean(diff > 0)))
    assert np.mean(diff > 0) < 0.05, float(np.mean(diff > 0))
    # 2. the backward on those pre-activations
    if mx:
        ref = om.moe_backward_mxfp8(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, affinity=cfg.affinity,
                                    fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w)
    else:
        ref = om.moe_backward(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, b2=inp.b2 if has_bias else None,
                              with_bias=has_bias)
    return compare_outputs(got, ref, tol)


@pytest.mark.parametrize("affinity", [AFFINITY_ON_H, AFFINITY_ON_I])
def test_recompute_bf16_bias_ragged(affinity):
    cfg = small_moe("rec_bf16", T=300, H=256, I=384, E=8, K=3, B=256, seed=41, bias=True, affinity=affinity)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(300, 3, 8, seed=6))
    _check(inp, PREC_BF16, has_bias=True, use_b1=True, tol=BF16_TOL)


def test_recompute_bf16_no_bias_single_expert():
    cfg = small_moe("rec_e1", T=200, H=384, I=128, E=1, K=1, B=128, seed=42)
    _check(make_moe_inputs(cfg), PREC_BF16, has_bias=False, use_b1=False, tol=BF16_TOL)


@pytest.mark.parametrize("B,pair", [(128, 1), (512, 1), (512, 2)])
def test_recompute_mxfp8_with_gate_up_bias(B, pair, set_option):
    # PAIR_GEMMS = 2 runs the recomputation GEMM on CTA pairs (the MXFP8 default is one CTA per tile)
    set_option("PAIR_GEMMS", pair)
    # b1 enters the recomputation only (bias gradients are BF16-only); inputs drawn with biases
    cfg = small_moe("rec_mx", T=320, H=512, I=256, E=6, K=2, B=B, seed=43, bias=True, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = with_ids(make_moe_inputs(cfg), _ragged_ids(320, 2, 6, seed=8))
    _check(inp, PREC_MXFP8, has_bias=False, use_b1=True, tol=MXFP8_TOL)


def test_recompute_matches_checkpoint_path_given_the_same_h():
    """The same problem run twice, once reading a checkpoint that holds the oracle's recomputed h and
    once recomputing it: the gradients agree to the rounding of h (both against the oracle)."""
    import moe_expert_layer_routing_gb300 as mb
    cfg = small_moe("rec_same", T=256, H=256, I=256, E=4, K=2, B=128, seed=44)
    inp = make_moe_inputs(cfg)
    ids = inp.ids.numpy()
    h = om.recompute_h(inp.x, inp.W1, ids)
    meta = oracle_meta(inp)
    ck = np.zeros(tuple(inp.ckpt.shape))
    # scatter h into the block layout: grouped row r of expert e -> slot block_offsets[e]*B + r - offsets[e]
    eo, bo, B = meta["expert_offsets"], meta["block_offsets"], cfg.block_size
    expert_of_row = np.repeat(np.arange(cfg.E), np.diff(eo))
    r = np.arange(int(eo[cfg.E]))
    slot = bo[expert_of_row] * B + (r - eo[expert_of_row])
    hf = h.reshape(cfg.T * cfg.K, 2 * cfg.I)[meta["s_scatter_idx"]]
    ck[slot // B, 0, :, slot % B] = hf[:, :cfg.I]
    ck[slot // B, 1, :, slot % B] = hf[:, cfg.I:]
    inp_ck = replace(inp, ckpt=torch.from_numpy(ck).to(torch.bfloat16))
    d = to_device(inp_ck)
    a = mb.moe_bwd(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, E=cfg.E, I=cfg.I, block_size=cfg.block_size,
                   W1=d.W1, W2=d.W2)
    b = mb.moe_bwd(x=d.x, dout=d.dout, s=d.s, ids=d.ids, E=cfg.E, I=cfg.I, block_size=cfg.block_size, W1=d.W1,
                   W2=d.W2, W1t=d.W1.transpose(1, 2).contiguous())
    torch.cuda.synchronize()
    ref = om.moe_backward(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h)
    compare_outputs(a, ref, BF16_TOL)
    compare_outputs(b, ref, BF16_TOL)
    for n in ("dx", "dW1", "dW2", "ds"):
        assert np.linalg.norm(np64(a[n]) - np64(b[n])) <= 2e-3 * np.linalg.norm(ref[n]), n
