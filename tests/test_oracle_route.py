"""Pins for oracle.route_meta: brute force over tiny routings and the block-count bound."""
import itertools

import numpy as np
import pytest

from oracle import route_meta as rm


def _brute_grouping(ids, E):
    """Grouped order by sorting (expert, flat index) tuples -- a different construction."""
    T, K = ids.shape
    pairs = sorted((int(ids[t, k]), t * K + k) for t in range(T) for k in range(K)
                   if 0 <= ids[t, k] < E)
    return [f for _, f in pairs], [e for e, _ in pairs]


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (2, 1, 3), (3, 2, 3), (2, 2, 2), (4, 1, 2)])
def test_route_meta_brute_force(T, K, E):
    B = 2
    for flat in itertools.product(range(E), repeat=T * K):
        ids = np.array(flat).reshape(T, K)
        m = rm.route_meta(ids, E, B, tile=4)
        order, experts = _brute_grouping(ids, E)
        assert list(m["s_scatter_idx"]) == order
        assert list(m["x_gather_idx"]) == [f // K for f in order]
        for r, f in enumerate(order):
            assert m["s_reverse_scatter_idx"][f] == r
        counts = np.bincount(np.array(experts, dtype=np.int64), minlength=E)
        assert list(np.diff(m["expert_offsets"])) == list(counts)
        assert m["num_blocks"] == sum(-(-c // B) for c in counts)
        assert m["num_blocks"] <= rm.num_blocks_bound(T, K, E, B)
        # every routed row sits in a block of its own expert, padding slots are -1
        tp = m["token_position_to_id"]
        b2e = m["block_to_expert"]
        used = np.zeros(tp.size, bool)
        for e in range(E):
            for j in range(counts[e]):
                slot = m["block_offsets"][e] * B + j
                assert tp[slot] == order[m["expert_offsets"][e] + j] // K
                assert b2e[slot // B] == e
                used[slot] = True
        assert np.all(tp[~used] == -1)
        assert np.all(b2e[m["num_blocks"]:] == -1)
        assert m["n_bad"] == 0


def test_invalid_ids_are_counted_and_dropped():
    ids = np.array([[0, 5], [-1, 1]])
    m = rm.route_meta(ids, 2, 4)
    assert m["n_bad"] == 2
    assert list(m["s_scatter_idx"]) == [0, 3]
    assert m["s_reverse_scatter_idx"][1] == -1 and m["s_reverse_scatter_idx"][2] == -1


def _max_blocks_over_histograms(TK, E, B):
    best = 0
    for hist in itertools.product(range(TK + 1), repeat=E):
        if sum(hist) == TK:
            best = max(best, sum(-(-n // B) for n in hist))
    return best


@pytest.mark.parametrize("TK,E,B", [(10, 2, 4), (7, 3, 2), (9, 3, 4), (5, 4, 4), (12, 3, 5),
                                    (2, 4, 4), (8, 1, 3), (6, 3, 1)])
def test_block_bound_is_tight_ceiling(TK, E, B):
    """N = ceil((TK-(E-1))/B) + E - 1 is exactly the worst case over all expert histograms."""
    assert rm.num_blocks_bound(TK, 1, E, B) == _max_blocks_over_histograms(TK, E, B)


def test_floor_reading_underallocates():
    # TK=10, E=2, B=4: one expert with 1 row and one with 9 rows needs 1 + 3 = 4 blocks
    assert _max_blocks_over_histograms(10, 2, 4) == 4
    assert (10 - 1) // 4 + 1 == 3
    assert rm.num_blocks_bound(10, 1, 2, 4) == 4


def test_checkpoint_rows_follow_token_position_to_id():
    rng = np.random.default_rng(0)
    T, K, E, B, I = 9, 2, 3, 4, 5
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    m = rm.route_meta(ids, E, B)
    N = rm.num_blocks_bound(T, K, E, B)
    ckpt = rng.standard_normal((N, 2, I, B))
    h = rm.checkpoint_rows(ckpt, m, T, K)
    tp = m["token_position_to_id"]
    # every slot holding token t of expert e carries that (t, k)'s gate/up columns
    for slot in np.nonzero(tp >= 0)[0]:
        blk, b = divmod(int(slot), B)
        e = m["block_to_expert"][blk]
        t = tp[slot]
        k = int(np.nonzero(ids[t] == e)[0][0])
        assert np.array_equal(h[t, k, :I], ckpt[blk, 0, :, b])
        assert np.array_equal(h[t, k, I:], ckpt[blk, 1, :, b])
