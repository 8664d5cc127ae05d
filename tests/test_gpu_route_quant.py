"""GPU parity: routing metadata and the MXFP8 quantiser, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from helpers import tiled_sf_to_plain
from oracle import mxfp8 as omx
from oracle import route_meta as orm

pytestmark = pytest.mark.gpu


def _lib():
    import moe_expert_layer_routing_gb300 as mb
    return mb


def _routing(T, K, E, seed, empty=(), single=(), bad=0):
    rng = np.random.default_rng(seed)
    allowed = [e for e in range(E) if e not in empty]
    ids = np.stack([rng.choice(allowed, size=K, replace=False) for _ in range(T)])
    for i, e in enumerate(single):          # expert e gets exactly one row
        ids[ids == e] = allowed[0] if allowed[0] != e else allowed[1]
        ids[i, 0] = e
    if bad:
        idx = rng.choice(T * K, size=bad, replace=False)
        ids.reshape(-1)[idx] = np.where(np.arange(bad) % 2 == 0, E, -1)
    return ids.astype(np.int32)


CASES = [
    (256, 2, 4, 128, dict(seed=0)),
    (1000, 3, 8, 256, dict(seed=1, empty=(0, 5), single=(1,))),
    (4097, 8, 64, 128, dict(seed=2)),
    (5, 2, 16, 1024, dict(seed=3)),
    (333, 1, 1, 512, dict(seed=4)),
    (700, 4, 32, 128, dict(seed=5, bad=9)),
    (16384, 8, 64, 128, dict(seed=6)),
]


@pytest.mark.parametrize("T,K,E,B,kw", CASES)
def test_route_meta_bit_exact(T, K, E, B, kw):
    mb = _lib()
    ids = _routing(T, K, E, **kw)
    got = mb.route_meta(torch.from_numpy(ids).cuda(), E, B)
    torch.cuda.synchronize()
    ref = orm.route_meta(ids, E, B)
    nv = int(ref["expert_offsets"][-1])
    g = {k: v.cpu().numpy() for k, v in got.items() if not k.startswith("_")}
    assert np.array_equal(g["expert_offsets"], ref["expert_offsets"])
    assert np.array_equal(g["x_gather_idx"][:nv], ref["x_gather_idx"])
    assert np.array_equal(g["s_scatter_idx"][:nv], ref["s_scatter_idx"])
    assert np.array_equal(g["s_reverse_scatter_idx"], ref["s_reverse_scatter_idx"])
    assert np.array_equal(g["token_position_to_id"], ref["token_position_to_id"])
    assert np.array_equal(g["block_to_expert"], ref["block_to_expert"])
    assert np.array_equal(g["block_offsets"], ref["block_offsets"])
    assert int(g["num_blocks"][0]) == ref["num_blocks"]
    assert int(g["status"][0]) == (mb.STATUS_BAD_EXPERT_ID if ref["n_bad"] else 0)


def _wide_bf16(rows, cols, seed):
    """bf16 values whose magnitude varies by 2^+-40 across rows and columns, with zero rows,
    subnormal-range and large entries."""
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(rows, cols, generator=g)
    v = v * torch.exp2(torch.randint(-40, 40, (rows, 1), generator=g).float())
    v = v * torch.exp2(torch.randint(-6, 6, (1, cols), generator=g).float())
    v[::7] = 0.0
    v[3, :5] = torch.tensor([1e-38, -2e-39, 3.0e38, -1.5e37, 0.0])
    return v.to(torch.bfloat16)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("gather", [False, True])
def test_quantize_rowwise_bit_exact(fmt, layout, gather):
    mb = _lib()
    x = _wide_bf16(256, 384, seed=10 + fmt)
    idx = None
    src = x
    if gather:
        idx = torch.randint(-1, 256, (384,), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
        src = torch.where((idx >= 0)[:, None], x[idx.clamp(min=0).long()], torch.zeros((), dtype=torch.bfloat16))
    q, sf = mb.mxfp8_quantize(x.cuda(), mb.QUANT_ROWWISE, fmt, None if idx is None else idx.cuda(), layout)
    torch.cuda.synchronize()
    rq, rs = omx.mx_quantize(src.double().numpy(), fmt, axis=1)
    assert np.array_equal(q.cpu().numpy(), rq)
    s = sf.cpu().numpy()
    s = tiled_sf_to_plain(s, rq.shape[0], rq.shape[1]) if layout == 1 else s.reshape(rq.shape[0], -1)
    assert np.array_equal(s, rs)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("gather", [False, True])
def test_quantize_colwise_bit_exact(fmt, layout, gather):
    mb = _lib()
    x = _wide_bf16(384, 256, seed=20 + fmt)
    idx = None
    src = x
    if gather:
        idx = torch.randint(-1, 384, (512,), generator=torch.Generator().manual_seed(4), dtype=torch.int32)
        src = torch.where((idx >= 0)[:, None], x[idx.clamp(min=0).long()], torch.zeros((), dtype=torch.bfloat16))
    q, sf = mb.mxfp8_quantize(x.cuda(), mb.QUANT_COLWISE, fmt, None if idx is None else idx.cuda(), layout)
    torch.cuda.synchronize()
    rq, rs = omx.mx_quantize(src.double().numpy().T, fmt, axis=1)   # transposed, groups along rows of src
    assert np.array_equal(q.cpu().numpy(), rq)
    s = sf.cpu().numpy()
    s = tiled_sf_to_plain(s, rq.shape[0], rq.shape[1]) if layout == 1 else s.reshape(rq.shape[0], -1)
    assert np.array_equal(s, rs)


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_colwise_16_byte_aligned_output(fmt):
    """The codes go to a caller buffer that is 16- but not 32-byte aligned (the public contract):
    same bytes as into an aligned buffer, and the oracle's."""
    mb = _lib()
    x = _wide_bf16(416, 128, seed=30 + fmt)
    q_al, sf_al = mb.mxfp8_quantize(x.cuda(), mb.QUANT_COLWISE, fmt, None, 0)
    buf = torch.zeros(128 * 416 + 64, dtype=torch.uint8, device="cuda")
    base = buf.data_ptr()
    off = (32 - base % 32) % 32 + 16          # 16 bytes past a 32-byte boundary
    sf = torch.zeros(128 * 416 // 32, dtype=torch.uint8, device="cuda")
    xd = x.cuda()
    rc = mb.lib().mxfp8_quantize(xd.data_ptr(), 416, 416, 128, 128, None, mb.QUANT_COLWISE, fmt, base + off,
                                 sf.data_ptr(), 0, None)
    assert rc == 0
    torch.cuda.synchronize()
    q = buf[off:off + 128 * 416].view(128, 416)
    assert torch.equal(q, q_al) and torch.equal(sf, sf_al)
    rq, _ = omx.mx_quantize(x.double().numpy().T, fmt, axis=1)
    assert np.array_equal(q.cpu().numpy(), rq)
