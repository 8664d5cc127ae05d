"""GPU parity at the full sizes of the three MoE workloads, in the launch configuration bench.py
times: all outputs are produced on the GPU, then sampled experts (empty, lightest, median, heaviest)
are checked on dW1/dW2(/db1/db2) and sampled tokens on dx/ds against the float64 oracle run on the
exact sub-problem (oracle.sample).  An expert above 8192 rows (the imbalanced workload's hottest,
about 59k rows: the longest contraction of the weight-gradient GEMMs) is checked over all its rows on
a range of 128 intermediate features: 256 columns of dW1 and 128 rows of dW2, each over the whole
hidden dimension; the MXFP8 oracle quantises with the torch-cast form of its round trip there."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, np64, rel_fro, run_gpu
from moe_expert_layer_routing_gb300.inputs import CONFIGS, PREC_MXFP8, make_moe_inputs
from oracle import moe as om
from oracle import mxfp8 as omx
from oracle import sample as osm

pytestmark = pytest.mark.gpu


HOT_ROWS = 8192      # experts above this many rows are checked on a feature range
HOT_FEATURES = 128


def _oracle(cfg, sub, weights_only=False):
    if cfg.precision == PREC_MXFP8:
        return om.moe_backward_mxfp8(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"],
                                     affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w,
                                     tokens=[] if weights_only else None, quant=omx.mx_roundtrip_torch)
    return om.moe_backward(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"],
                           b2=sub["b2"], with_bias=cfg.bias)


def _pick_tokens(ids, n, max_experts, seed):
    rng = np.random.default_rng(seed)
    chosen, experts = [], set()
    for t in rng.permutation(ids.shape[0]):
        new = experts | set(int(e) for e in ids[t])
        if len(new) <= max_experts:
            chosen.append(int(t))
            experts = new
        if len(chosen) == n:
            break
    return chosen


@pytest.mark.parametrize("name", ["finegrained_bf16", "manyexpert_mxfp8", "imbalanced_mxfp8"])
def test_full_size_sampled(name):
    cfg = CONFIGS[name]
    tol = MXFP8_TOL if cfg.precision == PREC_MXFP8 else BF16_TOL
    inp = make_moe_inputs(cfg, device="cuda")
    op, got = run_gpu(inp)
    assert int(got["status"].item()) == 0
    ids = inp.ids.cpu().numpy()
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    nz = np.nonzero(counts)[0]
    by_load = nz[np.argsort(counts[nz], kind="stable")]
    sample = {int(by_load[0]), int(by_load[len(by_load) // 2]), int(by_load[-1])}
    cpu = {k: (None if getattr(inp, k) is None else getattr(inp, k).cpu())
           for k in ("x", "dout", "W1", "W2", "ckpt", "b2")}
    s_np = inp.s.cpu().numpy()
    dW1, dW2 = got["dW1"], got["dW2"]
    errs = {}
    for e in sorted(sample):
        if counts[e] > HOT_ROWS:   # all its rows, a range of features in the middle of I
            i0 = (cfg.I // 2) // 32 * 32
            sub = osm.subproblem(cpu["x"], cpu["dout"], cpu["W1"], cpu["W2"], s_np, ids, cpu["ckpt"],
                                 cfg.block_size, experts=[e], b2=cpu["b2"], features=(i0, HOT_FEATURES))
            ref = _oracle(cfg, sub, weights_only=True)
            cols = torch.as_tensor(sub["columns"]).cuda()
            tag = f"[{e}, {counts[e]} rows, features {i0}..{i0 + HOT_FEATURES - 1}]"
            errs["dW1" + tag] = rel_fro(np64(dW1[e][:, cols]), ref["dW1"][0])
            errs["dW2" + tag] = rel_fro(np64(dW2[e][i0:i0 + HOT_FEATURES]), ref["dW2"][0])
            if cfg.bias:
                errs["db1" + tag] = rel_fro(np64(got["db1"][e][cols]), ref["db1"][0])
                errs["db2" + tag] = rel_fro(np64(got["db2"][e]), ref["db2"][0])
            del sub, ref
            continue
        sub = osm.subproblem(cpu["x"], cpu["dout"], cpu["W1"], cpu["W2"], s_np, ids, cpu["ckpt"], cfg.block_size,
                             experts=[e], b2=cpu["b2"])
        ref = _oracle(cfg, sub)
        errs[f"dW1[{e}]"] = rel_fro(np64(dW1[e]), ref["dW1"][0])
        errs[f"dW2[{e}]"] = rel_fro(np64(dW2[e]), ref["dW2"][0])
        if cfg.bias:
            errs[f"db1[{e}]"] = rel_fro(np64(got["db1"][e]), ref["db1"][0])
            errs[f"db2[{e}]"] = rel_fro(np64(got["db2"][e]), ref["db2"][0])
    empty = np.nonzero(counts == 0)[0]
    for e in empty[:2]:
        assert torch.count_nonzero(dW1[int(e)]).item() == 0 and torch.count_nonzero(dW2[int(e)]).item() == 0
    toks = _pick_tokens(ids, 8, 24 if cfg.precision == PREC_MXFP8 else 64, seed=5)
    sub = osm.subproblem(cpu["x"], cpu["dout"], cpu["W1"], cpu["W2"], s_np, ids, cpu["ckpt"], cfg.block_size,
                         tokens=toks, b2=cpu["b2"])
    ref = _oracle(cfg, sub)
    errs["dx[tokens]"] = rel_fro(np64(got["dx"][torch.as_tensor(sub["tokens"]).cuda()]), ref["dx"])
    errs["ds[tokens]"] = rel_fro(np64(got["ds"][torch.as_tensor(sub["tokens"]).cuda()]), ref["ds"])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    print(f"{name}: relative Frobenius errors {errs}")
    assert not bad, f"{name}: {bad} (all {errs})"
    for n in ("dx", "dW1", "dW2", "ds"):
        assert torch.isfinite(got[n].float()).all()
