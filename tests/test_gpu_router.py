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


def _scores(mode, logits, ids, renorm, E):
    """The forward's scores of each row over its slots with ids in [0, E) (0 for the others)."""
    s = np.zeros(ids.shape)
    for t in range(ids.shape[0]):
        ok = (ids[t] >= 0) & (ids[t] < E)
        if ok.any():
            s[t, ok] = orr.router_forward(mode, logits[t:t + 1], ids[t:t + 1, ok], renorm)[0]
    return s


@pytest.mark.parametrize("mode,renorm", [(0, False), (1, False), (1, True), (2, False)])
@pytest.mark.parametrize("T,E,K,odd", [(1000, 128, 8, False), (37, 40, 3, False), (5, 1024, 64, False),
                                        (300, 132, 32, True), (65, 520, 5, True), (40, 130, 4, True),
                                        (50, 1028, 2, False), (301, 256, 16, True), (77, 512, 8, True),
                                        (33, 68, 2, True), (129, 256, 8, True), (50, 32, 8, True)])
def test_router_bwd(mode, renorm, T, E, K, odd):
    """One-pass kernel with a token per 8 lanes (E a multiple of 4 up to 256, K <= 8: E = 32, 40, 68,
    128, 256 -- a partial column group at 68, odd token counts), per half-warp (up to 512, K <= 16:
    E = 256 with K = 16, E = 512) or per warp (up to 1024, K <= 32: E = 132 with K = 32, E = 520), and
    the general one (K = 64, E = 130, E = 1028); `odd` rows repeat an id (the slots' gradients add) and
    carry ids outside [0, E)."""
    import moe_expert_layer_routing_gb300 as mb
    logits, ids, g = _case(T, E, K, seed=T + E)
    if odd:
        ids[::3, K - 1] = ids[::3, 0]        # repeated id
        ids[1::7, K - 1] = -1                # unused slot
        ids[2::11, 0] = E                    # out of range
    scores = _scores(mode, logits, ids, renorm, E).astype(np.float32)
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
