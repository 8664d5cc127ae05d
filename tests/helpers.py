"""Shared test helpers: error metrics, scale-layout conversion, running the library and the oracle
on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, PREC_MXFP8, MoeInputs)
from oracle import moe as om
from oracle import mxfp8 as omx
from oracle import route_meta as orm

BF16_TOL = 1e-2     # relative Frobenius bar of the BF16 path against the float64 oracle
MXFP8_TOL = 2e-3    # relative Frobenius bar of the MXFP8 path against the oracle on the same quantisation


def rel_fro(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    if den == 0:
        return float(num)
    return float(num / den)


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def tiled_sf_to_plain(sf: np.ndarray, R: int, C: int) -> np.ndarray:
    """Scale bytes of an [R, C] matrix (groups along C) from the tiled MMA layout to [R, C/32]:
    atom ((r/128), (c/128)) row-major, inside it byte (r%32)*16 + ((r%128)/32)*4 + (c/32)%4."""
    sf = np.asarray(sf).reshape(-1)
    r = np.arange(R)[:, None]
    g = np.arange(C // 32)[None, :]
    c = g * 32
    off = ((r // 128) * (C // 128) + c // 128) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    return sf[off]


def oracle_meta(inp: MoeInputs) -> dict:
    cfg = inp.cfg
    return orm.route_meta(inp.ids.cpu().numpy(), cfg.E, cfg.block_size)


def oracle_h(inp: MoeInputs, meta: dict) -> np.ndarray:
    cfg = inp.cfg
    return orm.checkpoint_rows(inp.ckpt.cpu().to(torch.float64).numpy(), meta, cfg.T, cfg.K)


def oracle_bwd(inp: MoeInputs, meta=None):
    cfg = inp.cfg
    meta = meta or oracle_meta(inp)
    h = oracle_h(inp, meta)
    ids = inp.ids.cpu().numpy()
    if cfg.precision == PREC_MXFP8:
        return om.moe_backward_mxfp8(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, affinity=cfg.affinity,
                                     fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, b2=inp.b2, with_bias=cfg.bias)
    return om.moe_backward(inp.x, inp.dout, inp.W1, inp.W2, inp.s, ids, h, b2=inp.b2, with_bias=cfg.bias)


def to_device(inp: MoeInputs, device="cuda") -> MoeInputs:
    from dataclasses import replace
    mv = lambda t: None if t is None else t.to(device).contiguous()  # noqa: E731
    return replace(inp, x=mv(inp.x), dout=mv(inp.dout), W1=mv(inp.W1), W2=mv(inp.W2), b1=mv(inp.b1),
                   b2=mv(inp.b2), s=mv(inp.s), ids=mv(inp.ids), ckpt=mv(inp.ckpt))


def run_gpu(inp: MoeInputs):
    """moe_bwd through the C ABI on cuda:0; returns (op, outputs) after a device synchronise."""
    import moe_expert_layer_routing_gb300 as mb
    cfg = inp.cfg
    d = to_device(inp)
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size,
                   precision=cfg.precision, affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w,
                   has_bias=cfg.bias)
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, b2=d.b2 if cfg.bias else None)
    if cfg.precision == PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)
        W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
    else:
        kw.update(W1=d.W1, W2=d.W2)
    op.bind(**kw).run()
    torch.cuda.synchronize()
    return op, op.outputs()


def compare_outputs(got: dict, ref: dict, tol: float, names=("dx", "dW1", "dW2", "ds", "db1", "db2")):
    errs = {}
    for n in names:
        if ref.get(n) is None or got.get(n) is None:
            continue
        errs[n] = rel_fro(np64(got[n]), ref[n])
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"relative Frobenius errors above {tol}: {bad} (all: {errs})"
    return errs
