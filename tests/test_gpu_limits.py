"""The library at its documented size limits: E = 1024 experts (most of them empty or holding a
single row), top-K = 64, and block_size = 1024 -- routing metadata bit-exact against the oracle and
the whole backward within the path's tolerance, in both precisions."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, oracle_bwd, run_gpu
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe, with_ids)
from oracle import route_meta as orm

pytestmark = pytest.mark.gpu


def _ids(T, K, E, seed, bad=0):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, size=K, replace=False) for _ in range(T)]).astype(np.int32)
    if bad:
        idx = rng.choice(T * K, size=bad, replace=False)
        ids.reshape(-1)[idx] = np.where(np.arange(bad) % 2 == 0, E, -1)
    return ids


@pytest.mark.parametrize("T,K,E,B,bad", [(3000, 8, 1024, 128, 0), (1500, 64, 1024, 256, 0),
                                         (2000, 4, 1024, 1024, 7)])
def test_route_meta_at_the_limits(T, K, E, B, bad):
    import moe_expert_layer_routing_gb300 as mb
    ids = _ids(T, K, E, seed=T + K, bad=bad)
    got = mb.route_meta(torch.from_numpy(ids).cuda(), E, B)
    torch.cuda.synchronize()
    ref = orm.route_meta(ids, E, B)
    nv = int(ref["expert_offsets"][-1])
    g = {k: v.cpu().numpy() for k, v in got.items() if not k.startswith("_")}
    for name in ("expert_offsets", "s_reverse_scatter_idx", "token_position_to_id", "block_to_expert",
                 "block_offsets"):
        assert np.array_equal(g[name], ref[name]), name
    for name in ("x_gather_idx", "s_scatter_idx"):
        assert np.array_equal(g[name][:nv], ref[name]), name
    assert int(g["num_blocks"][0]) == ref["num_blocks"]
    assert int(g["status"][0]) == (mb.STATUS_BAD_EXPERT_ID if ref["n_bad"] else 0)


@pytest.mark.parametrize("prec,tol", [(PREC_BF16, BF16_TOL), (PREC_MXFP8, MXFP8_TOL)])
@pytest.mark.parametrize("case", ["E1024", "K64", "B1024"])
def test_moe_bwd_at_the_limits(case, prec, tol):
    """E = 1024 with 512 tokens at top-8 (about four rows an expert, many empty); top-64 of 128 experts;
    1024-row blocks over ragged experts."""
    shapes = {"E1024": dict(T=512, E=1024, K=8, B=128), "K64": dict(T=96, E=128, K=64, B=128),
              "B1024": dict(T=1500, E=4, K=2, B=1024)}[case]
    cfg = small_moe(f"limit_{case}", H=128, I=128, seed=71, precision=prec,
                    affinity=AFFINITY_ON_I if prec == PREC_MXFP8 else AFFINITY_ON_H, **shapes)
    inp = make_moe_inputs(cfg)
    if case == "B1024":   # ragged: one expert takes most rows
        rng = np.random.default_rng(5)
        p = np.array([0.1, 0.6, 0.25, 0.05])
        ids = np.stack([rng.choice(4, size=2, replace=False, p=p) for _ in range(cfg.T)]).astype(np.int32)
        inp = with_ids(inp, torch.from_numpy(ids))
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    counts = np.bincount(inp.ids.numpy().reshape(-1), minlength=cfg.E)
    empty = np.nonzero(counts == 0)[0]
    for e in empty[:4]:
        assert torch.count_nonzero(got["dW1"][int(e)]).item() == 0
        assert torch.count_nonzero(got["dW2"][int(e)]).item() == 0
    errs = compare_outputs(got, oracle_bwd(inp), tol)
    print(case, prec, {k: f"{v:.2e}" for k, v in errs.items()}, f"{len(empty)} empty experts")


@pytest.mark.parametrize("prec", [PREC_BF16, PREC_MXFP8])
def test_zero_tokens(prec):
    """T = 0: the routing metadata is all zero offsets and no blocks; the backward zeroes the weight
    gradients (or leaves them as they are with accumulate), with the token-sized arrays empty."""
    import moe_expert_layer_routing_gb300 as mb
    H, I, E, K, B = 128, 128, 4, 2, 128
    ids = torch.empty(0, K, dtype=torch.int32, device="cuda")
    meta = mb.route_meta(ids, E, B)
    torch.cuda.synchronize()
    assert torch.count_nonzero(meta["expert_offsets"]) == 0 and torch.count_nonzero(meta["block_offsets"]) == 0
    assert int(meta["num_blocks"][0]) == 0 and int(meta["status"][0]) == 0
    g = torch.Generator(device="cuda").manual_seed(5)
    W1 = (torch.randn(E, H, 2 * I, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, I, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    kw = dict(x=torch.empty(0, H, dtype=torch.bfloat16, device="cuda"),
              dout=torch.empty(0, H, dtype=torch.bfloat16, device="cuda"),
              s=torch.empty(0, K, dtype=torch.float32, device="cuda"), ids=ids,
              ckpt=torch.empty(0, 2, I, B, dtype=torch.bfloat16, device="cuda"))
    if prec == PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(W1)
        W2_q, W2_sf = mb.quantize_weights(W2)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
    else:
        kw.update(W1=W1, W2=W2)
    for accumulate in (False, True):
        op = mb.MoeBwd(T=0, H=H, I=I, E=E, K=K, block_size=B, precision=prec, accumulate=accumulate)
        op.dW1.fill_(1.0)
        op.dW2.fill_(1.0)
        op.bind(**kw).run()
        torch.cuda.synchronize()
        got = op.outputs()
        assert int(got["status"].item()) == 0
        want = 1.0 if accumulate else 0.0
        assert bool((got["dW1"] == want).all()) and bool((got["dW2"] == want).all())
        assert got["dx"].numel() == 0 and got["ds"].numel() == 0


@pytest.mark.parametrize("prec", [PREC_BF16, PREC_MXFP8])
def test_linear_bwd_empty_contractions(prec):
    """M = 0 (no rows): dW = dY^T X is an empty sum, all zeros; N = 0 (no output features): dX = dY W is
    all zeros.  The empty operands are not read."""
    import moe_expert_layer_routing_gb300 as mb
    for M, N, K in ((0, 256, 384), (256, 0, 384)):
        op = mb.LinearBwd(M, N, K, prec, device="cuda")
        op.dX.fill_(3.0)
        op.dW.fill_(3.0)
        dY = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        W = torch.randn(N, K, device="cuda").to(torch.bfloat16)
        X = torch.randn(M, K, device="cuda").to(torch.bfloat16)
        op.run(dY, W, X)
        torch.cuda.synchronize()
        assert bool((op.dX == 0).all()) and bool((op.dW == 0).all())
