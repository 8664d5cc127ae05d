"""moe_route_meta_noalloc, the routing-metadata entry point for callers that cannot allocate device
memory (its scratch is a fixed library-owned device array instead of a workspace): through the C ABI
it must give exactly what moe_route_meta gives, on two calls in a row sharing that array, and refuse
sizes above its fixed scratch without launching anything.  Kept in a file collected last."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ids(T, K, E, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.stack([rng.choice(E, size=K, replace=False) for _ in range(T)]).astype(np.int32))


def _noalloc(mb, ids, E, B):
    T, K = ids.shape
    N = mb.num_blocks_bound(T, K, E, B)
    i32 = dict(dtype=torch.int32, device="cuda")
    out = dict(expert_offsets=torch.empty(E + 1, **i32), x_gather_idx=torch.full((T * K,), -1, **i32),
               s_scatter_idx=torch.full((T * K,), -1, **i32), s_reverse_scatter_idx=torch.empty(T * K, **i32),
               token_position_to_id=torch.empty(N * B, **i32), block_to_expert=torch.empty(N, **i32),
               block_offsets=torch.empty(E + 1, **i32), num_blocks=torch.empty(1, **i32), status=torch.empty(1, **i32))
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = mb.lib().moe_route_meta_noalloc(p(ids), T, K, E, B, *[p(out[k]) for k in (
        "expert_offsets", "x_gather_idx", "s_scatter_idx", "s_reverse_scatter_idx", "token_position_to_id",
        "block_to_expert", "block_offsets", "num_blocks", "status")],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out


def test_noalloc_route_meta_matches_workspace_entry_point_twice():
    import moe_expert_layer_routing_gb300 as mb
    for T, K, E, B, seed in ((16384, 8, 64, 128, 1), (1000, 3, 8, 256, 2)):   # two calls in a row
        ids = _ids(T, K, E, seed).cuda()
        rc, got = _noalloc(mb, ids, E, B)
        assert rc == 0, mb.lib().moe_last_error()
        ref = mb.route_meta(ids, E, B)
        torch.cuda.synchronize()
        for k in ("expert_offsets", "x_gather_idx", "s_scatter_idx", "s_reverse_scatter_idx",
                  "token_position_to_id", "block_to_expert", "block_offsets", "num_blocks", "status"):
            assert torch.equal(got[k].cpu(), ref[k].cpu()), k


def test_noalloc_rejects_sizes_above_its_scratch():
    import moe_expert_layer_routing_gb300 as mb
    ids = torch.zeros(40000, 8, dtype=torch.int32, device="cuda")
    launches = mb.kernel_launches()
    rc, _ = _noalloc(mb, ids, 128, 512)
    assert rc == -2
    assert b"scratch" in mb.lib().moe_last_error()
    assert mb.kernel_launches() == launches


@pytest.mark.parametrize("B,E,K,code,text", [(0, 8, 2, -2, b"block_size"), (100, 8, 2, -2, b"block_size"),
                                             (128, 2048, 2, -2, b"E above"), (128, 8, 9, -1, b"bad sizes")])
def test_noalloc_bad_arguments_return_codes_without_launching(B, E, K, code, text):
    """Bad sizes are refused before the scratch size is computed: a code, moe_route_meta's message and
    no kernel launched (block_size 0 once reached a division by zero on the host)."""
    import moe_expert_layer_routing_gb300 as mb
    ids = torch.zeros(64, K, dtype=torch.int32, device="cuda")
    launches = mb.kernel_launches()
    rc = mb.lib().moe_route_meta_noalloc(ctypes.c_void_p(ids.data_ptr()), 64, K, E, B, *([None] * 9),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == code
    assert text in mb.lib().moe_last_error()
    assert mb.kernel_launches() == launches
