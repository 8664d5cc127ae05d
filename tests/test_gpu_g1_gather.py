"""G1 (dA = dout_g W2_e^T with the dSwiGLU epilogue) gathering its dout rows itself with 16-byte
asynchronous copies into the swizzled stage, against G1 reading the gathered copy written by the
gather pass: the A operand holds the same values, so every output is bit-identical -- both
precisions, every G1 tile width, ragged experts (padding rows), an empty and a single-row expert, a
hot expert over many tiles, several k-blocks per tile -- and matches the oracle."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, oracle_bwd, run_gpu
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe, with_ids)

pytestmark = pytest.mark.gpu


def _ids(T, K, E, seed):
    rng = np.random.default_rng(seed)
    p = np.ones(E - 2)
    p[0] = 12.0
    p /= p.sum()
    ids = np.stack([rng.choice(np.arange(2, E), size=K, replace=False, p=p) for _ in range(T)])
    ids[0, K - 1] = 1
    return torch.from_numpy(ids.astype(np.int32))


@pytest.mark.parametrize("prec,aff,bias,bn,I", [(PREC_BF16, AFFINITY_ON_H, True, 256, 512),
                                                (PREC_BF16, AFFINITY_ON_H, False, 128, 384),
                                                (PREC_MXFP8, AFFINITY_ON_I, False, 192, 384),
                                                (PREC_MXFP8, AFFINITY_ON_H, False, 128, 256)])
def test_gathered_and_copied_dout_rows_give_identical_outputs(prec, aff, bias, bn, I, set_option):
    set_option("G1_TILE_N", bn)
    cfg = small_moe("g1_gather", T=700, H=512, I=I, E=6, K=2, B=256, seed=81, precision=prec, affinity=aff,
                    bias=bias)
    inp = with_ids(make_moe_inputs(cfg), _ids(700, 2, 6, seed=6))
    outs = {}
    for gather in (1, 0):
        set_option("G1_GATHER", gather)
        _, got = run_gpu(inp)
        assert int(got["status"].item()) == 0
        outs[gather] = {k: v.clone() for k, v in got.items() if v is not None}
    for n in ("dx", "dW1", "dW2", "ds", "db1", "db2"):
        if n in outs[0]:
            assert torch.equal(outs[1][n], outs[0][n]), n
    compare_outputs(outs[1], oracle_bwd(inp), MXFP8_TOL if prec == PREC_MXFP8 else BF16_TOL)
