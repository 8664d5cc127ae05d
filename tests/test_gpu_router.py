"""GPU parity of moe_router_bwd against the float64 oracle (fp32 arithmetic on the GPU)."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, np64, oracle_bwd, rel_fro, run_gpu
from moe_expert_layer_routing_gb300.inputs import CONFIGS, make_moe_inputs
from oracle import router as orr

pytestmark = pytest.mark.gpu

# fp32 softmax over E terms and sums over K: relative error ~ (E + K) * 2^-24 ~ 1e-5 for E = 128
ROUTER_TOL = 3e-5


def _case(T, E, K, seed):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32) * 2
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    g = rng.standard_normal((T, K)).astype(np.float32)
    return logits, ids, g


@pytest.mark.parametrize("mode,renorm", [(0, False), (1, False), (1, True), (2, False)])
@pytest.mark.parametrize("T,E,K", [(1000, 128, 8), (37, 40, 3), (5, 1024, 64)])
def test_router_bwd(mode, renorm, T, E, K):
    import moe_expert_layer_routing_gb300 as mb
    logits, ids, g = _case(T, E, K, seed=T + E)
    scores = orr.router_forward(mode, logits, ids, renorm).astype(np.float32)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    got = mb.router_bwd(mode, c(ids), c(g), E, logits=c(logits), scores=c(scores), renorm=renorm)
    torch.cuda.synchronize()
    ref = orr.router_backward(mode, ids, g, E, logits=logits.astype(np.float64), renorm=renorm)
    assert rel_fro(np64(got), ref) < ROUTER_TOL


def test_chain_from_moe_ds_to_router_logits():
    """moe_bwd's ds fed to the router backward of the router that produced the routing (top-K over a
    softmax of all experts, renormalised): against the oracle chain."""
    import moe_expert_layer_routing_gb300 as mb
    inp = make_moe_inputs(CONFIGS["tiny_bf16"])
    op, got = run_gpu(inp)
    ref_ds = oracle_bwd(inp)["ds"]
    logits = inp.extra["logits"]
    dl = mb.router_bwd(1, inp.ids.cuda(), got["ds"], inp.cfg.E, logits=logits.cuda(), scores=inp.s.cuda(),
                       renorm=True)
    torch.cuda.synchronize()
    ref = orr.router_backward(1, inp.ids.numpy(), ref_ds, inp.cfg.E, logits=logits.double().numpy(), renorm=True)
    assert rel_fro(np64(dl), ref) < BF16_TOL
