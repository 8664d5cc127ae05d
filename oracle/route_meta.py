"""Oracle: routing metadata (test infrastructure only).

Follows the blockwise MoE backward page (parameters token_position_to_id [N*B], block_to_expert
[N,1], block_size, "Dimensions": N = (T*TopK - (E-1)) / B + E - 1) and the grouped-row indices of
sonic-moe backward.py (expert_frequency_offset [E+1], x_gather_idx, s_scatter_idx,
s_reverse_scatter_idx).

Readings where the pages are silent:
  * grouped order inside an expert is stable: rows sorted by (expert, t, k), i.e. by flat index
    f = t*K + k among the rows of that expert;
  * padding slots of token_position_to_id hold -1; unused blocks of block_to_expert hold -1;
  * the "/" of the block-count formula is a ceiling division (the tight worst case);
  * ids outside [0, E) are counted as errors and get no row.
"""
from __future__ import annotations

import numpy as np


def num_blocks_bound(T: int, K: int, E: int, B: int) -> int:
    """N = ceil((T*K - (E-1)) / B) + E - 1, or T*K when fewer rows than E-1 exist."""
    TK = T * K
    if TK <= 0:
        return 0
    num = TK - (E - 1)
    if num <= 0:
        return TK
    return -(-num // B) + E - 1


def route_meta(ids: np.ndarray, E: int, B: int, tile: int = 128) -> dict:
    """Plain per-expert grouping of the flat (t, k) rows.

    Returns int64 arrays:
      expert_offsets [E+1]            exclusive prefix of the per-expert row counts
      x_gather_idx [TK_valid]         grouped row -> token t
      s_scatter_idx [TK_valid]        grouped row -> flat f = t*K + k
      s_reverse_scatter_idx [T*K]     flat f -> grouped row (-1 for an invalid id)
      block_offsets [E+1]             exclusive prefix of ceil(n_e / B)
      num_blocks                      block_offsets[E]
      token_position_to_id [Nb*B]     slot -> token, -1 for padding (Nb = bound)
      block_to_expert [Nb]            block -> expert, -1 for unused blocks
      tile_offsets [E+1]              exclusive prefix of ceil(n_e / tile) * tile (tile-padded rows)
      n_bad                           number of (t,k) with an id outside [0, E)
    """
    ids = np.asarray(ids)
    T, K = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    TK = T * K
    counts = np.zeros(E, dtype=np.int64)
    rows_of = []
    for e in range(E):
        rows = np.nonzero(flat == e)[0]          # ascending flat index = stable (t, k) order
        rows_of.append(rows)
        counts[e] = rows.size
    n_bad = int(np.count_nonzero((flat < 0) | (flat >= E)))
    expert_offsets = np.zeros(E + 1, dtype=np.int64)
    expert_offsets[1:] = np.cumsum(counts)
    s_scatter_idx = np.concatenate(rows_of) if E > 0 else np.zeros(0, np.int64)
    x_gather_idx = s_scatter_idx // K
    rev = np.full(TK, -1, dtype=np.int64)
    rev[s_scatter_idx] = np.arange(s_scatter_idx.size)

    nblk = -(-counts // B)
    block_offsets = np.zeros(E + 1, dtype=np.int64)
    block_offsets[1:] = np.cumsum(nblk)
    Nb = num_blocks_bound(T, K, E, B)
    tpid = np.full(Nb * B, -1, dtype=np.int64)
    b2e = np.full(Nb, -1, dtype=np.int64)
    for e in range(E):
        b2e[block_offsets[e]:block_offsets[e + 1]] = e
        base = block_offsets[e] * B
        tpid[base: base + counts[e]] = rows_of[e] // K

    ntile = -(-counts // tile) * tile
    tile_offsets = np.zeros(E + 1, dtype=np.int64)
    tile_offsets[1:] = np.cumsum(ntile)
    return dict(expert_offsets=expert_offsets, x_gather_idx=x_gather_idx,
                s_scatter_idx=s_scatter_idx, s_reverse_scatter_idx=rev,
                block_offsets=block_offsets, num_blocks=int(block_offsets[E]),
                token_position_to_id=tpid, block_to_expert=b2e, tile_offsets=tile_offsets,
                counts=counts, n_bad=n_bad)


def checkpoint_rows(ckpt: np.ndarray, meta: dict, T: int, K: int) -> np.ndarray:
    """Gate/up pre-activation of every (t, k) from the block checkpoint [N, 2, I, B].

    The blockwise page stores gate_pre = checkpoint[block, 0] and up = checkpoint[block, 1], each
    [I, B] (feature-major, token-minor).  Grouped row r of expert e sits in slot
    block_offsets[e]*B + (r - expert_offsets[e]).  Returns h [T, K, 2I] with gate in [..., :I] and
    up in [..., I:] (rows with an invalid id are zero).
    """
    N, two, I, B = ckpt.shape
    h = np.zeros((T * K, 2 * I), dtype=np.float64)
    eo, bo = meta["expert_offsets"], meta["block_offsets"]
    E = len(eo) - 1
    expert_of_row = np.repeat(np.arange(E), np.diff(eo))      # expert of each grouped row
    r = np.arange(int(eo[E]))
    slot = bo[expert_of_row] * B + (r - eo[expert_of_row])
    blk, b = slot // B, slot % B
    f = meta["s_scatter_idx"]
    h[f, :I] = np.asarray(ckpt[blk, 0, :, b], dtype=np.float64)   # [rows, I]
    h[f, I:] = np.asarray(ckpt[blk, 1, :, b], dtype=np.float64)
    return h.reshape(T, K, 2 * I)
