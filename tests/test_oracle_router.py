"""Pins for oracle.router: finite differences of the forward, torch float64 autograd, and the
closed forms the sonic-moe router kernels state (s (g - <g,s>) on the selected logits; p (dp - <dp,p>))."""
import numpy as np
import pytest
import torch

from oracle import router as orr


def _problem(T=7, E=9, K=3, seed=0):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E))
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    g = rng.standard_normal((T, K))
    return logits, ids, g


@pytest.mark.parametrize("mode,renorm", [(0, False), (1, False), (1, True), (2, False)])
def test_finite_differences(mode, renorm):
    logits, ids, g = _problem()
    got = orr.router_backward(mode, ids, g, logits.shape[1], logits=logits, renorm=renorm)
    eps = 1e-6
    num = np.zeros_like(logits)
    for idx in np.ndindex(logits.shape):
        lp, lm = logits.copy(), logits.copy()
        lp[idx] += eps
        lm[idx] -= eps
        num[idx] = (np.sum(g * orr.router_forward(mode, lp, ids, renorm)) -
                    np.sum(g * orr.router_forward(mode, lm, ids, renorm))) / (2 * eps)
    assert np.max(np.abs(num - got)) < 1e-8


@pytest.mark.parametrize("mode,renorm", [(0, False), (1, False), (1, True), (2, False)])
def test_torch_autograd(mode, renorm):
    logits, ids, g = _problem(T=64, E=32, K=8, seed=1)
    L = torch.tensor(logits, requires_grad=True)
    I = torch.tensor(ids)
    if mode == 2:
        s = torch.gather(L, 1, I)
    elif mode == 0:
        s = torch.softmax(torch.gather(L, 1, I), dim=1)
    else:
        s = torch.gather(torch.softmax(L, dim=1), 1, I)
        if renorm:
            s = s / s.sum(dim=1, keepdim=True)
    (s * torch.tensor(g)).sum().backward()
    got = orr.router_backward(mode, ids, g, 32, logits=logits, renorm=renorm)
    assert np.allclose(got, L.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_closed_forms_of_the_page():
    logits, ids, g = _problem(T=10, E=12, K=4, seed=2)
    s = orr.router_forward(0, logits, ids)
    got = orr.router_backward(0, ids, g, 12, logits=logits)
    for t in range(10):
        dot = np.sum(g[t] * s[t])
        assert np.allclose(got[t, ids[t]], s[t] * (g[t] - dot), rtol=1e-12, atol=1e-14)
        mask = np.ones(12, bool)
        mask[ids[t]] = False
        assert np.all(got[t, mask] == 0)
    # top-K over softmax without renormalisation: p * (dp - <dp_sel, p_sel>) for every logit
    got = orr.router_backward(1, ids, g, 12, logits=logits)
    for t in range(10):
        p = np.exp(logits[t] - logits[t].max())
        p /= p.sum()
        dp = np.zeros(12)
        dp[ids[t]] = g[t]
        assert np.allclose(got[t], p * (dp - np.sum(g[t] * p[ids[t]])), rtol=1e-12, atol=1e-14)


def test_invalid_ids_contribute_nothing():
    logits, ids, g = _problem(T=3, E=6, K=2, seed=3)
    ids2 = ids.copy()
    ids2[1, 1] = 6
    a = orr.router_backward(2, ids2, g, 6)
    assert a[1].sum() == g[1, 0]
