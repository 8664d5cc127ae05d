"""moe_bwd driven by routing metadata from the caller ([BW] token_position_to_id, block_to_expert;
[SM] expert_frequency_offset, s_scatter_idx): metadata written by moe_route_meta, and metadata built
by the oracle's plain grouping, give outputs bit-identical to the call that computes the routing
itself (both precisions, an empty expert, a single-row expert, a hot expert) and meet the parity
bars; with num_valid_tokens too.  Metadata that is not a routing of the ids is reported in the
status word (MOE_STATUS_BAD_ROUTE_META) and stays within bounds: bad offsets leave an empty routing
(zero weight gradients)."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, compare_outputs, oracle_bwd, to_device
from moe_expert_layer_routing_gb300.inputs import (AFFINITY_ON_H, AFFINITY_ON_I, PREC_BF16, PREC_MXFP8,
                                                   make_moe_inputs, small_moe, with_ids)
from oracle import route_meta as orm

pytestmark = pytest.mark.gpu

OUT = ("dx", "dW1", "dW2", "ds", "db1", "db2")


def _ids(T, K, E, seed):
    """Expert 0 empty, expert 1 a single row, expert 2 hot, the rest uniform."""
    rng = np.random.default_rng(seed)
    p = np.ones(E - 2)
    p[0] = 10.0
    p /= p.sum()
    ids = np.stack([rng.choice(np.arange(2, E), size=K, replace=False, p=p) for _ in range(T)])
    ids[0, K - 1] = 1
    return torch.from_numpy(ids.astype(np.int32))


def _run(inp, route_meta=None, num_valid=None):
    import moe_expert_layer_routing_gb300 as mb
    cfg = inp.cfg
    d = to_device(inp)
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size, precision=cfg.precision,
                   affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, has_bias=cfg.bias)
    kw = dict(x=d.x, dout=d.dout, s=d.s, ids=d.ids, ckpt=d.ckpt, b2=d.b2 if cfg.bias else None, route_meta=route_meta)
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
    return {k: (v.clone() if v is not None else None) for k, v in op.outputs().items()}


def _oracle_meta(ids: np.ndarray, E, B):
    """The oracle's grouping as the int32 device tensors moe_bwd takes (s_scatter_idx padded to T*K)."""
    m = orm.route_meta(ids, E, B)
    TK = ids.size
    ss = np.full(TK, -1, dtype=np.int64)
    ss[: m["s_scatter_idx"].size] = m["s_scatter_idx"]
    dev = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int32)).cuda()  # noqa: E731
    return dict(expert_offsets=dev(m["expert_offsets"]), s_scatter_idx=dev(ss), block_offsets=dev(m["block_offsets"]),
                token_position_to_id=dev(m["token_position_to_id"]), block_to_expert=dev(m["block_to_expert"]))


CASES = [(PREC_BF16, AFFINITY_ON_H, True, BF16_TOL), (PREC_MXFP8, AFFINITY_ON_I, False, MXFP8_TOL)]


@pytest.mark.parametrize("prec,aff,bias,tol", CASES)
def test_library_and_oracle_metadata_reproduce_the_internal_routing(prec, aff, bias, tol):
    import moe_expert_layer_routing_gb300 as mb
    cfg = small_moe("meta_in", T=600, H=256, I=256, E=6, K=2, B=256, seed=71, precision=prec, affinity=aff, bias=bias)
    inp = with_ids(make_moe_inputs(cfg), _ids(600, 2, 6, seed=4))
    base = _run(inp)
    assert int(base["status"].item()) == 0
    lib_meta = mb.route_meta(inp.ids.cuda(), cfg.E, cfg.block_size)
    for meta in (lib_meta, {k: lib_meta[k] for k in ("expert_offsets", "s_scatter_idx", "block_offsets")},
                 _oracle_meta(inp.ids.numpy(), cfg.E, cfg.block_size)):
        got = _run(inp, route_meta=meta)
        assert int(got["status"].item()) == 0
        for n in OUT:
            if base[n] is not None:
                assert torch.equal(got[n], base[n]), n
    compare_outputs(got, oracle_bwd(inp), tol)


def test_metadata_with_num_valid_tokens():
    """Only the leading 350 tokens routed: the oracle's grouping of those tokens' slots drives the call."""
    cfg = small_moe("meta_nv", T=500, H=256, I=256, E=5, K=2, B=128, seed=72, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = make_moe_inputs(cfg)
    base = _run(inp, num_valid=350)
    ids = inp.ids.numpy().copy()
    ids[350:] = -1
    got = _run(inp, route_meta=_oracle_meta(ids, cfg.E, cfg.block_size), num_valid=350)
    assert int(got["status"].item()) == 0 and int(base["status"].item()) == 0
    for n in ("dx", "dW1", "dW2", "ds"):
        assert torch.equal(got[n], base[n]), n


def _corrupt(meta, how, E):
    m = {k: v.clone() for k, v in meta.items() if k in ("expert_offsets", "s_scatter_idx", "block_offsets",
                                                        "token_position_to_id", "block_to_expert")}
    eo = m["expert_offsets"].cpu()
    if how == "offsets_decrease":
        m["expert_offsets"][3] = int(eo[2]) - 1
    elif how == "offsets_past_rows":
        m["expert_offsets"][E] = int(eo[E]) + 5
    elif how == "offsets_not_from_zero":
        m["expert_offsets"][0] = 1
    elif how == "too_few_blocks":
        bo = m["block_offsets"].cpu()
        m["block_offsets"][3:] = bo[3:] - 1        # expert 2 (hot) loses a block
    elif how == "blocks_past_bound":
        m["block_offsets"][E] = 1 << 30
    elif how == "duplicate_row":
        m["s_scatter_idx"][int(eo[3]) + 1] = m["s_scatter_idx"][int(eo[3])]
    elif how == "row_of_other_expert":
        a, b = int(eo[2]), int(eo[3])
        m["s_scatter_idx"][a], m["s_scatter_idx"][b] = m["s_scatter_idx"][b].clone(), m["s_scatter_idx"][a].clone()
    elif how == "flat_out_of_range":
        m["s_scatter_idx"][int(eo[4])] = 1 << 30
    elif how == "slot_missing":
        m["expert_offsets"][E] = int(eo[E]) - 1
    elif how == "token_table":
        bo = m["block_offsets"].cpu()
        m["token_position_to_id"][int(bo[2]) * 256 + 3] += 1
    elif how == "block_table":
        m["block_to_expert"][int(m["block_offsets"][2])] = 5
    return m


@pytest.mark.parametrize("how,empty", [("offsets_decrease", True), ("offsets_past_rows", True),
                                       ("offsets_not_from_zero", True), ("too_few_blocks", True),
                                       ("blocks_past_bound", True), ("duplicate_row", False),
                                       ("row_of_other_expert", False), ("flat_out_of_range", False),
                                       ("slot_missing", False), ("token_table", False), ("block_table", False)])
def test_bad_metadata_is_reported(how, empty):
    import moe_expert_layer_routing_gb300 as mb
    cfg = small_moe("meta_bad", T=600, H=256, I=256, E=6, K=2, B=256, seed=73, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    inp = with_ids(make_moe_inputs(cfg), _ids(600, 2, 6, seed=5))
    meta = mb.route_meta(inp.ids.cuda(), cfg.E, cfg.block_size)
    got = _run(inp, route_meta=_corrupt(meta, how, cfg.E))
    status = int(got["status"].item())
    assert status & mb.STATUS_BAD_ROUTE_META, (how, status)
    for n in ("dx", "dW1", "dW2", "ds"):
        assert torch.isfinite(got[n].float()).all(), n
    if empty:   # every row dropped: nothing accumulates
        assert torch.count_nonzero(got["dW1"]).item() == 0 and torch.count_nonzero(got["dx"]).item() == 0
    again = _run(inp, route_meta=meta)          # the context is fine and the good metadata still works
    assert int(again["status"].item()) == 0
