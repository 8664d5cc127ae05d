"""Pins for oracle.linear: torch autograd of Y = X @ W^T on MX-exact inputs, inner-product identity."""
import numpy as np
import torch

from oracle import linear as ol
from oracle import mxfp8 as mx


def _exact_inputs(M=64, N=96, K=32, seed=0):
    """Integers in [-3, 3] are exactly representable by MX e5m2 along either axis (every group's
    scale is 2^-14 or 2^-15 and 1, 2, 3 times it are e5m2 values)."""
    rng = np.random.default_rng(seed)
    return (rng.integers(-3, 4, (M, N)).astype(np.float64), rng.integers(-3, 4, (N, K)).astype(np.float64),
            rng.integers(-3, 4, (M, K)).astype(np.float64))


def test_exact_inputs_match_torch_autograd():
    dY, W, X = _exact_inputs()
    for v, ax in ((dY, 0), (dY, 1), (W, 0), (X, 0)):
        assert np.array_equal(mx.mx_roundtrip(v, mx.E5M2, axis=ax), v)
    tX = torch.tensor(X, requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    Y = tX @ tW.T
    (Y * torch.tensor(dY)).sum().backward()
    g = ol.linear_backward_mxfp8(dY, W, X)
    assert np.array_equal(g["dX"], tX.grad.numpy())
    assert np.array_equal(g["dW"], tW.grad.numpy())
    g2 = ol.linear_backward(dY, W, X)
    assert np.array_equal(g2["dX"], tX.grad.numpy()) and np.array_equal(g2["dW"], tW.grad.numpy())


def test_inner_product_identity():
    """<dX, X> = <dY, Y> = <dW, W> for Y = X W^T (exact integer inputs)."""
    dY, W, X = _exact_inputs(seed=1)
    g = ol.linear_backward_mxfp8(dY, W, X)
    Y = X @ W.T
    v = np.sum(dY * Y)
    assert np.sum(g["dX"] * X) == v and np.sum(g["dW"] * W) == v


def test_quantisation_axes():
    """Scaling row m of dY by 2^j scales row m of dX exactly (dX groups along N); scaling
    column k of X by 2^j scales column k of dW exactly (dW groups along M)."""
    rng = np.random.default_rng(2)
    dY, W, X = rng.standard_normal((64, 64)), rng.standard_normal((64, 32)) * 0.02, rng.standard_normal((64, 32))
    base = ol.linear_backward_mxfp8(dY, W, X)
    sc = np.ldexp(1.0, rng.integers(-8, 8, 64))
    assert np.array_equal(ol.linear_backward_mxfp8(dY * sc[:, None], W, X)["dX"], base["dX"] * sc[:, None])
    sk = np.ldexp(1.0, rng.integers(-8, 8, 32))
    assert np.array_equal(ol.linear_backward_mxfp8(dY, W, X * sk[None, :])["dW"], base["dW"] * sk[None, :])
    err = np.linalg.norm(base["dX"] - dY @ W) / np.linalg.norm(dY @ W)
    assert 1e-3 < err < 0.15
