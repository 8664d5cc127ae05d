"""prep's gathered operands at sizes where every persistent prep CTA walks several work items (more
128-column chunk items, or whole tiles with biases, than two CTAs per SM), so the gathers of one
item overlap the quantisation of the previous one and the tokens of each next tile come from the
prefetch: the row-major dout_g copy (G1's A operand) and the weight-gradient GEMMs' operands — for
MXFP8 (and BF16 without MN-major operands) the transposed x_g^T and dout_g^T with their scales, for
BF16 by default x's gathered rows (the dW2 GEMM then reads dout_g itself) — bit-exact against the
oracle's gather and quantisation (dout s-scaled in fp32 for affinity on H)."""
import numpy as np
import pytest
import torch

from helpers import run_gpu, tiled_sf_to_plain
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe)
from oracle import mxfp8 as omx

pytestmark = pytest.mark.gpu

# (T, H, bias): without biases an item is one 128-column chunk of a tile (about 200 tiles x 4 chunks
# here); with biases a whole tile (about 500 tiles)
SHAPES = [(6000, 512, False), (16000, 256, True)]


def _bf16_bits(a: torch.Tensor) -> np.ndarray:
    return a.contiguous().view(torch.int16).numpy()


@pytest.mark.parametrize("mn", [1, 0])
@pytest.mark.parametrize("prec", [PREC_MXFP8, PREC_BF16])
@pytest.mark.parametrize("affinity", [AFFINITY_ON_I, AFFINITY_ON_H])
@pytest.mark.parametrize("T,H,bias", SHAPES)
def test_prep_operands_many_items(prec, affinity, T, H, bias, mn, set_option):
    if prec == PREC_MXFP8 and mn == 0:
        pytest.skip("MXFP8 builds the transposed operands either way")
    set_option("MN_OPERANDS", mn)
    cfg = small_moe("prep_items", T=T, H=H, I=256, E=8, K=4, B=256, seed=101 + T % 7, precision=prec,
                    affinity=affinity, bias=bias)
    inp = make_moe_inputs(cfg)
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    P = op.tile_rows
    used = int(op.region("TILE_OFFSETS").view(torch.int32)[cfg.E].item())
    items = used // 128 * (1 if bias else H // 128)
    assert items > 2 * torch.cuda.get_device_properties(0).multi_processor_count, "a work item per CTA at most"
    flat = op.region("TILE_ROW_FLAT").view(torch.int32).cpu().numpy()[:used]
    valid = flat >= 0
    t, k = np.where(valid, flat // cfg.K, 0), np.where(valid, flat % cfg.K, 0)
    vt = torch.from_numpy(valid)[:, None]
    tt = torch.from_numpy(t.astype(np.int64))
    xrows = torch.where(vt, inp.x[tt], torch.zeros((), dtype=inp.x.dtype))       # bf16, padding zero
    drows = torch.where(vt, inp.dout[tt], torch.zeros((), dtype=inp.dout.dtype))
    if affinity == AFFINITY_ON_H:  # s * dout in fp32 (the kernel's product), then quantised / rounded
        sd = drows.float() * torch.where(vt, inp.s[tt, torch.from_numpy(k.astype(np.int64))][:, None],
                                         torch.zeros(()))
    else:
        sd = drows.float()
    if prec == PREC_MXFP8:
        rq, rs = omx.mx_quantize(drows.double().numpy(), cfg.fp8_act, axis=1)
        assert np.array_equal(op.region("DOUT_G").cpu().numpy().reshape(P, H)[:used], rq)
        assert np.array_equal(tiled_sf_to_plain(op.region("DOUT_G_SF").cpu().numpy(), P, H)[:used], rs)
        for name, rows in (("X_GT", xrows.double().numpy()), ("DOUT_GT", sd.double().numpy())):
            tq, ts = omx.mx_quantize(rows, cfg.fp8_act, axis=0)
            q = op.region(name).cpu().numpy().reshape(H, P)[:, :used].T
            sf = tiled_sf_to_plain(op.region(name + "_SF").cpu().numpy(), H, P)[:, :used // 32].T
            assert np.array_equal(q, tq), name
            assert np.array_equal(sf, ts), name
    else:
        g = op.region("DOUT_G").cpu().view(torch.bfloat16).reshape(P, H)[:used]
        assert np.array_equal(_bf16_bits(g), _bf16_bits(drows))
        checks = [("X_GT", xrows)]
        if not mn:  # MN-major: the dW2 GEMM reads dout_g itself (s moves to a' for affinity on H)
            checks.append(("DOUT_GT", sd.to(torch.bfloat16)))
        for name, rows in checks:
            r = op.region(name).cpu().view(torch.bfloat16)
            got_rows = r.reshape(P, H)[:used] if mn else r.reshape(H, P)[:, :used].T
            assert np.array_equal(_bf16_bits(got_rows), _bf16_bits(rows)), name
