"""Oracle: restriction of a large problem to a sample (test infrastructure only).

Full-size workloads are checked on samples the float64 oracle can afford:
  * experts mode -- every row routed to the chosen experts (all their tokens), so their dW1, dW2,
    db1, db2 are exactly those of the full problem (the stable row order inside each expert, and so
    its MXFP8 token groups, is unchanged);
  * tokens mode  -- the chosen tokens with all their K rows, so their dx and ds are exactly those of
    the full problem (every dx/ds term is computed row by row);
  * features     -- with experts mode, a range [i0, i0 + n) of the intermediate features only (gate
    and up columns of W1, rows of W2, checkpoint features; concatenated gate/up layout).  Every
    intermediate feature enters dW1 and dW2 on its own -- dA_raw of feature i contracts the full
    hidden row of dout with row i of W2, and the token-direction MX groups run down one column --
    so dW1's columns and dW2's rows of those features (and db1's columns, and db2) are exactly those
    of the full problem, over every row of the expert.  ds, dx_expanded and dx sum over all
    features and are not (a multiple of 32 features keeps the row-wise groups of dh whole).
Experts are renumbered 0..len-1; rows of unselected experts get id -1 (no row).  This is indexing
only: no arithmetic of the method happens here.
"""
from __future__ import annotations

import numpy as np

from .route_meta import route_meta


def _ckpt_rows(ckpt, meta, K, flats):
    """Gate/up pre-activations [len(flats), 2I] of flat rows f = t*K + k from the block checkpoint
    (I = the checkpoint's feature count)."""
    import torch
    N, _, I, B = ckpt.shape
    r = meta["s_reverse_scatter_idx"][flats]
    eo, bo = meta["expert_offsets"], meta["block_offsets"]
    e = np.searchsorted(eo, r, side="right") - 1
    slot = bo[e] * B + (r - eo[e])
    blk = torch.from_numpy(slot // B)
    b = torch.from_numpy(slot % B)
    gate = ckpt[blk, 0, :, b]       # [n, I]
    up = ckpt[blk, 1, :, b]
    return torch.cat([gate, up], dim=1).to(torch.float64).numpy()


def subproblem(x, dout, W1, W2, s, ids, ckpt, block_size, experts=None, tokens=None, b2=None, features=None):
    """x, dout, W1, W2, ckpt, b2: CPU torch tensors (any float dtype); s, ids: CPU tensors or arrays.
    Exactly one of `experts` / `tokens` is given; `features` = (i0, n) further restricts an experts
    sample to the intermediate features [i0, i0 + n).  Returns dict(x, dout, W1, W2, s, ids, h, b2,
    tokens, experts, columns) with h [T', K, 2I'] float64, experts the original ids of the renumbered
    ones and columns the original W1 columns of the kept ones (gate features, then up features)."""
    import torch
    ids_np = np.asarray(ids)
    T, K = ids_np.shape
    E = W1.shape[0]
    I = W1.shape[2] // 2
    if features is not None:
        assert experts is not None, "a feature range restricts an experts sample"
        i0, n = int(features[0]), int(features[1])
        assert 0 <= i0 and n > 0 and i0 + n <= I
        feat = np.arange(i0, i0 + n)
        columns = np.concatenate([feat, I + feat])
        W1 = W1[:, :, torch.from_numpy(columns)]
        W2 = W2[:, i0:i0 + n, :]
        ckpt = ckpt[:, :, i0:i0 + n, :]
    else:
        columns = np.arange(2 * I)
    meta = route_meta(ids_np, E, block_size)
    if experts is not None:
        experts = np.asarray(sorted(set(int(e) for e in experts)), dtype=np.int64)
        in_sel = np.isin(ids_np, experts)
        toks = np.nonzero(in_sel.any(axis=1))[0]
        keep = in_sel[toks]
    else:
        toks = np.asarray(sorted(set(int(t) for t in tokens)), dtype=np.int64)
        valid = (ids_np[toks] >= 0) & (ids_np[toks] < E)
        experts = np.unique(ids_np[toks][valid])
        keep = valid
    remap = -np.ones(E, dtype=np.int64)
    remap[experts] = np.arange(len(experts))
    ids2 = np.where(keep, remap[np.clip(ids_np[toks], 0, E - 1)], -1)
    flats = (toks[:, None] * K + np.arange(K)[None, :])[keep]
    I2 = W1.shape[2]
    h = np.zeros((len(toks), K, I2))
    if flats.size:
        h[keep] = _ckpt_rows(ckpt, meta, K, flats)
    tt = torch.from_numpy(toks)
    ee = torch.from_numpy(experts)
    s_np = np.asarray(s.numpy() if hasattr(s, "numpy") else s, dtype=np.float64)
    return dict(x=x[tt], dout=dout[tt], W1=W1[ee], W2=W2[ee], s=s_np[toks], ids=ids2, h=h,
                b2=None if b2 is None else b2[ee], tokens=toks, experts=experts, columns=columns)
