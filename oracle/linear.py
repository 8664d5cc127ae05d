"""Oracle: dense linear backward, BF16 and MXFP8 (test infrastructure only).

"Matmul MXFP8 Backward Kernel API Reference", "Forward pass convention": Y = X @ W^T with X [M,K],
W [N,K], Y [M,N].  The backward is two matmuls,

    dX = dY @ W        [M,K], contraction over N
    dW = dY^T @ X      [N,K], contraction over M

In the MXFP8 form each operand is quantised in 32-element groups along that matmul's contraction
dimension (float8_dtype, default float8_e5m2, for every operand) and the products are accumulated
exactly here (float64); the page's output_dtype default is bfloat16.
"""
from __future__ import annotations

import numpy as np

from . import mxfp8 as mx
from .moe import _f64


def linear_backward(dY, W, X):
    dY, W, X = map(_f64, (dY, W, X))
    return dict(dX=dY @ W, dW=dY.T @ X)


def linear_backward_mxfp8(dY, W, X, fmt=mx.E5M2):
    dY, W, X = map(_f64, (dY, W, X))
    dYq_n = mx.mx_roundtrip(dY, fmt, axis=1)    # dX: groups along N (rows of dY)
    Wq_n = mx.mx_roundtrip(W, fmt, axis=0)      #     groups along N (columns of W)
    dYq_m = mx.mx_roundtrip(dY, fmt, axis=0)    # dW: groups along M (columns of dY)
    Xq_m = mx.mx_roundtrip(X, fmt, axis=0)      #     groups along M (columns of X)
    return dict(dX=dYq_n @ Wq_n, dW=dYq_m.T @ Xq_m)
