"""Dense linear backward on the GPU: the MXFP8 operands its one quantisation launch writes (dY
row-wise for dX, the transposed W^T, dY^T and X^T for the two GEMMs, all with tiled scales) bit-exact
against the oracle's quantiser on inputs spread over 80 binades with zeros; the two GEMMs on the
library's second stream give the same bits as one after the other, are joined back into the caller's
stream, and run inside a captured CUDA graph."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, MXFP8_TOL, np64, rel_fro, tiled_sf_to_plain
from moe_expert_layer_routing_gb300.inputs import FP8_E4M3, FP8_E5M2, LinearConfig, make_linear_inputs
from oracle import linear as olin
from oracle import mxfp8 as omx

pytestmark = pytest.mark.gpu


def _spread(r, c, gen):
    """bf16 values whose magnitudes span 2^-40 .. 2^40, about 1% exact zeros."""
    v = torch.randn(r, c, generator=gen) * torch.pow(2.0, torch.randint(-40, 41, (r, c), generator=gen).float())
    v[torch.rand(r, c, generator=gen) < 0.01] = 0.0
    return v.to(torch.bfloat16)


def _regions(ws: np.ndarray, M, N, K):
    """The MXFP8 operand regions of linear_bwd's workspace, in its order (each start 256-byte aligned):
    dY codes [M,N] and scales, W^T [K,N], dY^T [N,M], X^T [K,M], each followed by its scales."""
    sizes = [M * N, M * N // 32, K * N, K * N // 32, N * M, N * M // 32, K * M, K * M // 32]
    out, off = [], 0
    for n in sizes:
        out.append(ws[off:off + n])
        off = (off + n + 255) // 256 * 256
    return out


@pytest.mark.parametrize("fmt", [FP8_E5M2, FP8_E4M3])
def test_linear_mxfp8_operands_bit_exact(fmt):
    import moe_expert_layer_routing_gb300 as mb
    M, N, K = 384, 256, 640   # three, two and five 128-tiles: every source has several tiles of each kind
    gen = torch.Generator().manual_seed(61 + fmt)
    dY, W, X = _spread(M, N, gen), _spread(N, K, gen), _spread(M, K, gen)
    op = mb.LinearBwd(M, N, K, mb.PREC_MXFP8, fmt, device="cuda").run(dY.cuda(), W.cuda(), X.cuda())
    torch.cuda.synchronize()
    reg = _regions(op.workspace.cpu().numpy(), M, N, K)
    q, s = omx.mx_quantize(dY.double().numpy(), fmt, axis=1)      # dX's A: groups along N
    assert np.array_equal(reg[0].reshape(M, N), q)
    assert np.array_equal(tiled_sf_to_plain(reg[1], M, N), s)
    # transposed operands: groups along the source rows (W's N for dX; dY's and X's M for dW)
    for name, src, iq in (("W^T", W, 2), ("dY^T", dY, 4), ("X^T", X, 6)):
        R, C = src.shape
        q, s = omx.mx_quantize(src.double().numpy(), fmt, axis=0)   # [R, C] codes, [R/32, C] scales
        assert np.array_equal(reg[iq].reshape(C, R), q.T), name
        assert np.array_equal(tiled_sf_to_plain(reg[iq + 1], C, R), s.T), name


@pytest.mark.parametrize("prec", [1, 0])
def test_linear_concurrent_gemms_match_serial_on_a_side_stream(prec, set_option):
    """dW's GEMM on the library's second stream beside dX's: the same bits as both on the caller's
    stream; work the caller enqueues after the call on its own (non-default) stream sees both
    results (three calls in a row, each followed by copies of the outputs on that stream)."""
    import moe_expert_layer_routing_gb300 as mb
    inp = make_linear_inputs(LinearConfig("lin_conc", M=512, N=384, K=768, seed=47))
    dY, W, X = inp.dY.cuda(), inp.W.cuda(), inp.X.cuda()
    set_option("LINEAR_CONCURRENT", 0)
    ref = mb.linear_bwd(dY, W, X, precision=prec)
    torch.cuda.synchronize()
    set_option("LINEAR_CONCURRENT", 1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    copies = []
    with torch.cuda.stream(s):
        for _ in range(3):
            got = mb.linear_bwd(dY, W, X, precision=prec, stream=s)
            copies.append((got["dX"].clone(), got["dW"].clone()))
    s.synchronize()
    for dXc, dWc in copies:
        assert torch.equal(dXc, ref["dX"]) and torch.equal(dWc, ref["dW"])
    fn, tol = (olin.linear_backward_mxfp8, MXFP8_TOL) if prec == 1 else (olin.linear_backward, BF16_TOL)
    want = fn(inp.dY, inp.W, inp.X)
    assert rel_fro(np64(ref["dX"]), want["dX"]) < tol and rel_fro(np64(ref["dW"]), want["dW"]) < tol


def test_linear_bwd_captured_in_a_cuda_graph(set_option):
    """The fork onto the second stream and the join back are captured with the call: replaying the
    graph reproduces the eager outputs."""
    import moe_expert_layer_routing_gb300 as mb
    set_option("LINEAR_CONCURRENT", 1)
    inp = make_linear_inputs(LinearConfig("lin_graph", M=256, N=384, K=512, seed=53))
    dY, W, X = inp.dY.cuda(), inp.W.cuda(), inp.X.cuda()
    op = mb.LinearBwd(256, 384, 512, mb.PREC_MXFP8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        op.run(dY, W, X, stream=s)   # eager first: the library's stream and events exist before capture
    s.synchronize()
    want_dX, want_dW = op.dX.clone(), op.dW.clone()
    op.dX.zero_()
    op.dW.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        op.run(dY, W, X)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(op.dX, want_dX) and torch.equal(op.dW, want_dW)
