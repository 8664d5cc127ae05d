"""Oracle: router backward, from the routing scores' gradient ds to the router logits (test
infrastructure only).

sonic-moe functional/backward.py, `_topk_softmax_bwd` (softmax over the selected top-K logits, or
top-K over a softmax of all E logits with optional renormalisation of the kept probabilities) and
`_topk_bwd` (scores are the selected logits themselves).  Written here as explicit Jacobian
products of each forward, per token, in float64:

  softmax over top-K    s = softmax(l[idx])                   ds/dl[idx_j] = s_k (delta_kj - s_j)
  top-K over softmax    p = softmax(l) over all E, r = p[idx], s = r / sum(r) if renormalised else r
                        dp_i/dl_j = p_i (delta_ij - p_j);  ds_k/dr_j = (delta_kj - s_k) / sum(r)
  plain top-K           s = l[idx]                            ds_k/dl[idx_k] = 1

Gradients of every logit are returned ([T, E]); logits never selected get zero in the first and
last forms and -p_i * <dp_sel, p_sel> in the second.  Ids outside [0, E) contribute nothing.
"""
from __future__ import annotations

import numpy as np

SOFTMAX_OVER_TOPK, TOPK_OVER_SOFTMAX, TOPK = 0, 1, 2


def _softmax(v):
    m = np.max(v)
    e = np.exp(v - m)
    return e / e.sum()


def router_backward(mode, ids, dscores, E, logits=None, renorm=False):
    ids = np.asarray(ids)
    g = np.asarray(dscores, dtype=np.float64)
    T, K = ids.shape
    out = np.zeros((T, E))
    lg = None if logits is None else np.asarray(logits, dtype=np.float64)
    for t in range(T):
        ok = [k for k in range(K) if 0 <= ids[t, k] < E]
        idx = ids[t, ok]
        gt = g[t, ok]
        if mode == TOPK:
            np.add.at(out[t], idx, gt)
        elif mode == SOFTMAX_OVER_TOPK:
            s = _softmax(lg[t, idx])
            J = np.diag(s) - np.outer(s, s)            # J[k, j] = ds_k / dl[idx_j]
            np.add.at(out[t], idx, J.T @ gt)
        elif mode == TOPK_OVER_SOFTMAX:
            p = _softmax(lg[t])
            Jp = np.diag(p) - np.outer(p, p)           # Jp[i, j] = dp_i / dl_j
            r = p[idx]
            if renorm:
                S = r.sum()
                s = r / S
                Jr = (np.eye(len(idx)) - np.outer(s, np.ones(len(idx)))) / S   # Jr[k, j] = ds_k / dr_j
                dr = Jr.T @ gt
            else:
                dr = gt
            dp = np.zeros(E)
            np.add.at(dp, idx, dr)
            out[t] = Jp.T @ dp
        else:
            raise ValueError(mode)
    return out


def router_forward(mode, logits, ids, renorm=False):
    """Scores [T, K] of the forward (used by the pins)."""
    lg = np.asarray(logits, dtype=np.float64)
    ids = np.asarray(ids)
    T, K = ids.shape
    s = np.zeros((T, K))
    for t in range(T):
        if mode == TOPK:
            s[t] = lg[t, ids[t]]
        elif mode == SOFTMAX_OVER_TOPK:
            s[t] = _softmax(lg[t, ids[t]])
        else:
            r = _softmax(lg[t])[ids[t]]
            s[t] = r / r.sum() if renorm else r
    return s
