"""CPU checks of the C-ABI library: it builds, loads, and exports every declared entry point; host
functions without device work behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moebwd.h")


@pytest.fixture(scope="module")
def lib():
    from moe_expert_layer_routing_gb300 import _build
    _build.build()
    import moe_expert_layer_routing_gb300 as mb
    return mb.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in moebwd.h but not exported"
    import moe_expert_layer_routing_gb300 as mb
    assert sorted(mb.EXPORTED) == names


def test_block_bound_matches_oracle(lib):
    from oracle.route_meta import num_blocks_bound
    for T, K, E, B in [(256, 2, 4, 128), (16384, 8, 64, 128), (32768, 8, 128, 256), (65536, 8, 128, 512),
                       (3, 1, 8, 128), (0, 2, 4, 128), (10, 1, 2, 128)]:
        assert lib.moe_num_blocks_bound(T, K, E, B) == num_blocks_bound(T, K, E, B)
    assert lib.moe_num_blocks_bound(16384, 8, 64, 128) == 1087
    assert lib.moe_num_blocks_bound(65536, 8, 128, 512) == 1151


def test_workspace_queries(lib):
    import moe_expert_layer_routing_gb300 as mb
    a = mb.MoeBwdArgs(T=256, H=128, I=256, E=4, K=2, block_size=128)
    assert lib.moe_bwd_workspace_size(ctypes.byref(a)) > 0
    bad = mb.MoeBwdArgs(T=256, H=100, I=256, E=4, K=2, block_size=128)
    assert lib.moe_bwd_workspace_size(ctypes.byref(bad)) == 0
    assert b"multiples of 128" in lib.moe_last_error()
    bad2 = mb.MoeBwdArgs(T=256, H=128, I=256, E=4, K=2, block_size=96)
    assert lib.moe_bwd_workspace_size(ctypes.byref(bad2)) == 0
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.moe_bwd_workspace_region(ctypes.byref(a), mb.WS_REGIONS.index("DH"), ctypes.byref(off),
                                        ctypes.byref(nb)) == 0
    P = lib.moe_tile_rows_capacity(256, 2, 4)
    assert P % 128 == 0 and P >= 512
    assert nb.value == P * 2 * 256 * 2 and off.value % 256 == 0
    assert lib.moe_route_meta_workspace_size(256, 2, 4, 128) > 0
    assert lib.linear_bwd_workspace_size(4096, 4096, 4096, 1) > 0


def test_host_argument_errors(lib):
    import moe_expert_layer_routing_gb300 as mb
    a = mb.MoeBwdArgs(T=256, H=128, I=256, E=4, K=2, block_size=128)
    assert lib.moe_bwd(ctypes.byref(a), None) == -1          # null pointers, caught on the host
    assert b"null" in lib.moe_last_error()
    assert lib.mxfp8_quantize(None, 1, 1, 32, 32, None, 0, 0, None, None, 1, None) == -1
    assert lib.linear_bwd(None, None, None, 128, 128, 128, 1, 1, None, None, None, 0, None) == -1
    assert lib.moe_route_meta(None, 4, 2, 4, 100, *([None] * 10), 0, None) == -2


def test_product_path_refuses_cpu_tensors():
    import torch
    import moe_expert_layer_routing_gb300 as mb
    with pytest.raises(mb.MoeError):
        mb.mxfp8_quantize(torch.zeros(32, 32, dtype=torch.bfloat16))


@pytest.mark.parametrize("T,K,E,B,code,text", [
    (1000, 2, 8, 0, -2, b"block_size"),      # used to divide by zero in the scratch-size query
    (1000, 2, 8, 100, -2, b"block_size"),
    (1000, 2, 2048, 128, -2, b"E above"),
    (1000, 9, 8, 128, -1, b"bad sizes"),     # K > E
    (-1, 2, 8, 128, -1, b"bad sizes"),
])
def test_route_meta_entry_points_reject_bad_sizes_alike(lib, T, K, E, B, code, text):
    """moe_route_meta and moe_route_meta_noalloc check their size arguments in the same order with the
    same codes, before anything else (no CUDA call, no launch): this runs without a GPU."""
    import moe_expert_layer_routing_gb300 as mb
    before = mb.kernel_launches()
    assert lib.moe_route_meta(None, T, K, E, B, *([None] * 10), 0, None) == code
    assert text in lib.moe_last_error()
    assert lib.moe_route_meta_noalloc(None, T, K, E, B, *([None] * 10)) == code
    msg = lib.moe_last_error()
    assert text in msg and msg.startswith(b"moe_route_meta_noalloc")
    assert mb.kernel_launches() == before


def test_route_meta_workspace_size_is_zero_for_rejected_sizes(lib):
    for B in (0, -128, 100):
        assert lib.moe_route_meta_workspace_size(1000, 2, 8, B) == 0
    assert lib.moe_route_meta_workspace_size(1000, 2, 2048, 128) == 0


def test_options_defaults_and_validation(lib):
    import moe_expert_layer_routing_gb300 as mb
    assert mb.get_option("WAIT_LIMIT_NS") == 2_000_000_000
    assert mb.get_option("PAIR_GEMMS") == 1 and mb.get_option("PAIR_TILE_N") == 256
    assert mb.get_option("G1_TILE_N") == 0 and mb.get_option("PREP_TILE_ORDER") == 1
    assert mb.get_option("G1_GATHER") == 0 and mb.get_option("PDL") == 1
    assert mb.get_option("LINEAR_CONCURRENT") == 1
    # the binding names every option the library has: the last is valid, the one past it is not
    assert lib.moe_get_option(len(mb.OPTIONS) - 1) >= 0 and lib.moe_get_option(len(mb.OPTIONS)) == -1
    assert lib.moe_set_option(99, 1) == -1 and b"unknown option" in lib.moe_last_error()
    assert lib.moe_get_option(99) == -1
    for name, bad in (("WAIT_LIMIT_NS", 0), ("PAIR_GEMMS", 3), ("PAIR_TILE_N", 192), ("G1_TILE_N", 64),
                      ("G2_TILE_N", 192), ("PREP_TILE_ORDER", 2), ("LINEAR_CONCURRENT", 2)):
        assert lib.moe_set_option(mb.OPTIONS.index(name), bad) == -1
        assert b"not allowed" in lib.moe_last_error()
    mb.set_option("G1_WARPS", 8)
    with mb.option("G1_TILE_N", 192):
        assert mb.get_option("G1_TILE_N") == 192
        a = mb.MoeBwdArgs(T=256, H=256, I=384, E=4, K=2, block_size=128, precision=1)
        n192 = lib.moe_bwd_workspace_size(ctypes.byref(a))
    assert mb.get_option("G1_TILE_N") == 0
    mb.set_option("G1_TILE_N", 128)
    n128 = lib.moe_bwd_workspace_size(ctypes.byref(a))
    mb.set_option("G1_TILE_N", None)
    mb.set_option("G1_WARPS", None)
    assert mb.get_option("G1_TILE_N") == 0 and mb.get_option("G1_WARPS") == 0
    assert n192 > 0 and n128 > 0 and n192 != n128   # the tile width moves the ds partials' region


def test_mn_operands_option_moves_the_bf16_layout(lib):
    """MOE_OPT_MN_OPERANDS (default 1): BF16's dW1 GEMM reads dh itself, so the DH_T region is empty;
    with 0 it holds dh^T [2I,P] bf16.  MXFP8 keeps dh^T either way.  Host-only (workspace sizes)."""
    import moe_expert_layer_routing_gb300 as mb
    assert mb.get_option("MN_OPERANDS") == 1
    assert lib.moe_set_option(mb.OPTIONS.index("MN_OPERANDS"), 2) == -1

    def dh_t_bytes(precision):
        a = mb.MoeBwdArgs(T=256, H=256, I=384, E=4, K=2, block_size=128, precision=precision)
        off, nb = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.moe_bwd_workspace_region(ctypes.byref(a), mb.WS_REGIONS.index("DH_T"), ctypes.byref(off),
                                            ctypes.byref(nb)) == 0
        return nb.value, lib.moe_bwd_workspace_size(ctypes.byref(a))

    P = mb.tile_rows_capacity(256, 2, 4)
    nb_mn, total_mn = dh_t_bytes(0)
    assert nb_mn == 0 and dh_t_bytes(1)[0] == 2 * 384 * P
    with mb.option("MN_OPERANDS", 0):
        nb, total = dh_t_bytes(0)
        assert nb == 2 * 384 * P * 2 and total >= total_mn + nb   # bf16 dh^T back in the workspace
        assert dh_t_bytes(1)[0] == 2 * 384 * P
    assert mb.get_option("MN_OPERANDS") == 1


def test_mxfp8_bias_with_saved_scaled_dout_is_refused(lib):
    import moe_expert_layer_routing_gb300 as mb
    a = mb.MoeBwdArgs(T=256, H=128, I=256, E=4, K=2, block_size=128, precision=1, has_bias=1, affinity=0)
    assert lib.moe_bwd_workspace_size(ctypes.byref(a)) > 0          # MXFP8 with biases is supported
    a.down_proj_act_ckpt = 4096                                     # (pointer value only checked for presence)
    assert lib.moe_bwd_workspace_size(ctypes.byref(a)) == 0
    assert b"down_proj_act_ckpt" in lib.moe_last_error()


def test_moe_bwd_size_limits_refused_on_the_host(lib):
    """The documented limits (1 <= K <= E <= 1024, K <= 64, H and I multiples of 128, the four block
    sizes) are checked before any work: the workspace query returns 0 with a message, at the limits
    it returns a size."""
    import moe_expert_layer_routing_gb300 as mb

    def size(**kw):
        a = mb.MoeBwdArgs(**dict(dict(T=256, H=128, I=128, E=128, K=8, block_size=128, precision=0), **kw))
        return lib.moe_bwd_workspace_size(ctypes.byref(a))

    assert size(E=1024, K=64) > 0 and size(block_size=1024) > 0
    for kw, text in ((dict(E=128, K=65), b"K <= 64"), (dict(E=4, K=5), b"K <= E"), (dict(E=1025), b"E above"),
                     (dict(H=192), b"multiples of 128"), (dict(block_size=2048), b"block_size")):
        assert size(**kw) == 0, kw
        assert text in lib.moe_last_error(), (kw, lib.moe_last_error())


def test_empty_calls_return_without_work(lib):
    """Empty problems are valid and do nothing (their pointers may be null): a quantisation of zero rows
    or columns, a router backward of zero tokens, a linear backward whose outputs are all empty (K = 0);
    no kernel is launched (host-only: no device is touched)."""
    import moe_expert_layer_routing_gb300 as mb
    before = mb.kernel_launches()
    assert lib.mxfp8_quantize(None, 0, 0, 32, 32, None, 0, 0, None, None, 0, None) == 0
    assert lib.mxfp8_quantize(None, 0, 64, 0, 0, None, 1, 1, None, None, 1, None) == 0
    assert lib.moe_router_bwd(1, 1, None, None, None, None, 0, 2, 8, None, None) == 0
    assert lib.linear_bwd(None, None, None, 128, 128, 0, 1, 1, None, None, None, 0, None) == 0
    assert lib.linear_bwd(None, None, None, 128, 128, 0, 7, 1, None, None, None, 0, None) == -1   # precision
    assert lib.linear_bwd(None, None, None, 100, 128, 0, 1, 1, None, None, None, 0, None) == -2   # not x128
    assert mb.kernel_launches() == before
