"""GPU parity of the routing options of the blockwise backward: variable top-K (-1 marks an unused
slot), [BW] `num_valid_tokens` (only the leading tokens are routed) and the [T*E] masked affinity
gradient, both precisions, against the oracle on the same inputs."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, np64, oracle_bwd, rel_fro, to_device
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe, with_ids)
from oracle import moe as om

pytestmark = pytest.mark.gpu


def _run(inp, num_valid=None, masked=True):
    import moe_expert_layer_routing_gb300 as mb
    cfg = inp.cfg
    d = to_device(inp)
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size, precision=cfg.precision,
                   affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, has_bias=cfg.bias, ds_masked=masked)
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, b2=d.b2 if cfg.bias else None)
    if num_valid is not None:
        kw["num_valid_tokens"] = torch.tensor([num_valid], dtype=torch.int32, device="cuda")
    if cfg.precision == PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(d.W1, cfg.fp8_w)
        W2_q, W2_sf = mb.quantize_weights(d.W2, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
    else:
        kw.update(W1=d.W1, W2=d.W2)
    op.bind(**kw).run()
    torch.cuda.synchronize()
    return op.outputs()


def _varlen_ids(T, K, E, seed):
    """Each token keeps 1..K distinct experts; the remaining slots are -1, at varying positions."""
    rng = np.random.default_rng(seed)
    ids = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        n = rng.integers(1, K + 1)
        pos = rng.permutation(K)[:n]
        ids[t, pos] = rng.permutation(E)[:n]
    return torch.from_numpy(ids)


@pytest.mark.parametrize("prec,aff,tol", [(PREC_BF16, AFFINITY_ON_H, BF16_TOL), (PREC_MXFP8, AFFINITY_ON_I, MXFP8_TOL)])
def test_variable_top_k(prec, aff, tol):
    cfg = small_moe("varlen", T=400, H=256, I=256, E=6, K=4, B=256, seed=61, precision=prec, affinity=aff)
    inp = with_ids(make_moe_inputs(cfg), _varlen_ids(400, 4, 6, seed=3))
    got = _run(inp)
    assert int(got["status"].item()) == 0          # -1 slots are not errors
    ref = oracle_bwd(inp)
    compare_outputs(got, ref, tol)
    ids = inp.ids.numpy()
    assert np.all(np64(got["ds"])[ids < 0] == 0)
    m = om.ds_masked(ref["ds"], ids, cfg.E)
    assert rel_fro(np64(got["ds_masked"]), m) <= tol
    assert np.all(np64(got["ds_masked"])[m == 0] == 0)


@pytest.mark.parametrize("prec,tol", [(PREC_BF16, BF16_TOL), (PREC_MXFP8, MXFP8_TOL)])
@pytest.mark.parametrize("nv", [0, 1, 237, 10_000])
def test_num_valid_tokens(prec, tol, nv):
    import moe_expert_layer_routing_gb300 as mb
    cfg = small_moe("nvalid", T=300, H=256, I=256, E=5, K=2, B=128, seed=62, precision=prec,
                    affinity=AFFINITY_ON_I if prec == PREC_MXFP8 else AFFINITY_ON_H)
    inp = make_moe_inputs(cfg)
    got = _run(inp, num_valid=nv)
    assert int(got["status"].item()) == 0
    n = max(0, min(nv, cfg.T))
    ref_inp = with_ids(inp, torch.from_numpy(om.valid_token_ids(inp.ids.numpy(), nv)))
    ref = oracle_bwd(ref_inp)
    if n > 0:
        compare_outputs(got, ref, tol)
    else:
        for name in ("dW1", "dW2"):
            assert torch.count_nonzero(got[name]) == 0
    assert torch.count_nonzero(got["dx"][n:]) == 0 and torch.count_nonzero(got["ds"][n:]) == 0
    dm = got["ds_masked"].reshape(cfg.T, cfg.E)
    assert torch.count_nonzero(dm[n:]) == 0
    if n > 0:
        assert rel_fro(np64(got["ds_masked"]), om.ds_masked(ref["ds"], ref_inp.ids.numpy(), cfg.E)) <= tol


def test_out_of_range_ids_still_reported():
    import moe_expert_layer_routing_gb300 as mb
    cfg = small_moe("badid", T=128, H=128, I=128, E=4, K=2, B=128, seed=63)
    inp = make_moe_inputs(cfg)
    ids = inp.ids.clone()
    ids[3, 1] = -1   # unused slot: fine
    ids[7, 0] = -2   # invalid
    got = _run(with_ids(inp, ids))
    assert int(got["status"].item()) == mb.STATUS_BAD_EXPERT_ID
