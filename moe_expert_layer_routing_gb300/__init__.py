"""Python binding of libmoebwd: MoE expert-layer backward (BF16 / MXFP8) on one GB300 GPU.

Argument marshalling only: every step of the computation runs in the CUDA kernels of the shared
library (include/moebwd.h).  PyTorch provides device memory and streams.  The library is loaded on
first use; if it has not been built, or no CUDA device is present, calls raise -- there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .inputs import (AFFINITY_ON_H, AFFINITY_ON_I, FP8_E4M3, FP8_E5M2, PREC_BF16,  # noqa: F401
                     PREC_MXFP8)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoebwd.so")

QUANT_ROWWISE, QUANT_COLWISE = 0, 1
SF_PLAIN, SF_TILED = 0, 1
STATUS_BAD_EXPERT_ID, STATUS_TIMEOUT, STATUS_BAD_ROUTE_META = 1, 2, 4
ACT_CHECKPOINT, ACT_RECOMPUTE = 0, 1
GLU_SWIGLU, GLU_GEGLU = 0, 1
GATE_UP_CONCAT, GATE_UP_INTERLEAVED = 0, 1

WS_REGIONS = ["EXPERT_OFFSETS", "TILE_OFFSETS", "BLOCK_OFFSETS", "TILE_ROW_FLAT", "FLAT_TILE_ROW",
              "DOUT_G", "DOUT_G_SF", "DOUT_GT", "DOUT_GT_SF", "X_GT", "X_GT_SF", "DH", "DH_SF",
              "DH_T", "DH_T_SF", "AP_T", "AP_T_SF", "DX_EXP", "X_G", "X_G_SF", "GATE_UP_CKPT", "DOUT_Q"]

EXPORTED = ["moe_last_error", "moe_version", "moe_num_blocks_bound", "moe_route_meta_workspace_size",
            "moe_route_meta", "mxfp8_quantize", "moe_bwd_workspace_size", "moe_bwd",
            "moe_bwd_workspace_region", "moe_tile_rows_capacity", "linear_bwd_workspace_size",
            "linear_bwd", "moe_profile_enable", "moe_profile_read", "moe_kernel_launches",
            "moe_route_meta_noalloc", "moe_router_bwd", "moe_set_option", "moe_get_option"]

# library options (moe_set_option)
OPTIONS = ["WAIT_LIMIT_NS", "PAIR_GEMMS", "PAIR_TILE_N", "G1_TILE_N", "G2_TILE_N", "G3_TILE_N", "G4_TILE_N",
           "PREP_TILE_ORDER", "G1_GATHER", "G1_WARPS", "PDL", "MN_OPERANDS", "LINEAR_CONCURRENT"]

STAGES = ["route", "prep", "G1_dA_dswiglu", "G3_dW2", "G2_dx_expanded", "G4_dW1", "reduce", "G0_recompute_h"]


class MoeError(RuntimeError):
    pass


class MoeBwdArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("T", "H", "I", "E", "K", "block_size", "precision", "affinity", "fp8_act", "fp8_w",
                 "has_bias")] + \
               [(n, ctypes.c_void_p) for n in
                ("x", "dout", "W1", "W2", "W1_q", "W1_sf", "W2_q", "W2_sf", "b2", "s", "ids",
                 "gate_up_ckpt", "dx", "dW1", "dW2", "ds", "db1", "db2", "status_dev", "workspace")] + \
               [("workspace_bytes", ctypes.c_size_t), ("accumulate", ctypes.c_int), ("act_src", ctypes.c_int)] + \
               [(n, ctypes.c_void_p) for n in ("W1t", "W1t_q", "W1t_sf", "b1", "ds_masked", "num_valid_tokens")] + \
               [(n, ctypes.c_int) for n in ("glu", "gate_up_layout")] + \
               [(n, ctypes.c_void_p) for n in ("intermediate_ckpt", "scaled_intermediate_ckpt", "down_proj_act_ckpt",
                                               "gate_act_ckpt")] + \
               [(n, ctypes.c_void_p) for n in ("expert_offsets", "s_scatter_idx", "block_offsets",
                                               "token_position_to_id", "block_to_expert")]

ROUTE_META_FIELDS = ("expert_offsets", "s_scatter_idx", "block_offsets", "token_position_to_id", "block_to_expert")


_lib = None


def lib():
    """The loaded shared library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise MoeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "moe_last_error": ([], ctypes.c_char_p),
        "moe_version": ([], ctypes.c_char_p),
        "moe_num_blocks_bound": ([i64, i32, i32, i32], i64),
        "moe_route_meta_workspace_size": ([i32, i32, i32, i32], sz),
        "moe_route_meta": ([vp, i32, i32, i32, i32] + [vp] * 10 + [sz, vp], i32),
        "mxfp8_quantize": ([vp, i64, i64, i64, i64, vp, i32, i32, vp, vp, i32, vp], i32),
        "moe_bwd_workspace_size": ([ctypes.POINTER(MoeBwdArgs)], sz),
        "moe_bwd": ([ctypes.POINTER(MoeBwdArgs), vp], i32),
        "moe_bwd_workspace_region": ([ctypes.POINTER(MoeBwdArgs), i32, ctypes.POINTER(sz),
                                      ctypes.POINTER(sz)], i32),
        "moe_tile_rows_capacity": ([i32, i32, i32], i64),
        "linear_bwd_workspace_size": ([i64, i64, i64, i32], sz),
        "linear_bwd": ([vp, vp, vp, i64, i64, i64, i32, i32, vp, vp, vp, sz, vp], i32),
        "moe_profile_enable": ([i32], i32),
        "moe_profile_read": ([ctypes.POINTER(ctypes.c_double), i32, ctypes.POINTER(i32)], i32),
        "moe_kernel_launches": ([], ctypes.c_uint64),
        "moe_route_meta_noalloc": ([vp, i32, i32, i32, i32] + [vp] * 9 + [vp], i32),
        "moe_router_bwd": ([i32, i32, vp, vp, vp, vp, i32, i32, i32, vp, vp], i32),
        "moe_set_option": ([i32, i64], i32),
        "moe_get_option": ([i32], i64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(rc: int, what: str):
    if rc != 0:
        raise MoeError(f"{what} failed ({rc}): {lib().moe_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise MoeError("tensors must be CUDA tensors (there is no CPU path)")
        if t is not None and not t.is_contiguous():
            raise MoeError("tensors must be contiguous")


def profile_enable(enable: bool = True):
    """Start (or stop) recording per-stage CUDA events inside moe_bwd; discards earlier records."""
    _check(lib().moe_profile_enable(int(enable)), "moe_profile_enable")


def profile_read() -> tuple[dict, int]:
    """Total milliseconds per stage over the profiled moe_bwd calls, and the number of calls."""
    arr = (ctypes.c_double * len(STAGES))()
    calls = ctypes.c_int()
    _check(lib().moe_profile_read(arr, len(STAGES), ctypes.byref(calls)), "moe_profile_read")
    return {n: arr[i] for i, n in enumerate(STAGES)}, calls.value


def set_option(name: str, value: int | None):
    """Set a library option by its name in OPTIONS (None restores the default)."""
    _check(lib().moe_set_option(OPTIONS.index(name), -1 if value is None else int(value)), "moe_set_option")


def get_option(name: str) -> int:
    return int(lib().moe_get_option(OPTIONS.index(name)))


class option:
    """Context manager: set a library option for the duration of a block, then restore its old value."""

    def __init__(self, name: str, value: int):
        self.name, self.value = name, value

    def __enter__(self):
        self.old = get_option(self.name)
        set_option(self.name, self.value)
        return self

    def __exit__(self, *exc):
        set_option(self.name, self.old)
        return False


def kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().moe_kernel_launches())


def num_blocks_bound(T: int, K: int, E: int, block_size: int) -> int:
    return int(lib().moe_num_blocks_bound(T, K, E, block_size))


def tile_rows_capacity(T: int, K: int, E: int) -> int:
    return int(lib().moe_tile_rows_capacity(T, K, E))


def _ws(nbytes: int, device):
    # 256-byte aligned by the CUDA caching allocator
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def route_meta(ids: torch.Tensor, E: int, block_size: int, stream=None) -> dict:
    """moe_route_meta on int32 ids [T,K]; returns the metadata tensors and the status word."""
    _need_cuda(ids)
    assert ids.dtype == torch.int32 and ids.dim() == 2
    T, K = ids.shape
    dev = ids.device
    N = num_blocks_bound(T, K, E, block_size)
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(expert_offsets=torch.empty(E + 1, **i32), x_gather_idx=torch.full((T * K,), -1, **i32),
               s_scatter_idx=torch.full((T * K,), -1, **i32), s_reverse_scatter_idx=torch.empty(T * K, **i32),
               token_position_to_id=torch.empty(max(N * block_size, 1), **i32),
               block_to_expert=torch.empty(max(N, 1), **i32), block_offsets=torch.empty(E + 1, **i32),
               num_blocks=torch.empty(1, **i32), status=torch.empty(1, **i32))
    wsz = lib().moe_route_meta_workspace_size(T, K, E, block_size)
    ws = _ws(wsz, dev)
    rc = lib().moe_route_meta(_ptr(ids), T, K, E, block_size, *[_ptr(out[k]) for k in (
        "expert_offsets", "x_gather_idx", "s_scatter_idx", "s_reverse_scatter_idx", "token_position_to_id",
        "block_to_expert", "block_offsets", "num_blocks", "status")], _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "moe_route_meta")
    out["token_position_to_id"] = out["token_position_to_id"][: N * block_size]
    out["block_to_expert"] = out["block_to_expert"][:N]
    out["_workspace"] = ws
    return out


def sf_bytes(rows: int, cols: int, scale_layout: int) -> int:
    """Scale bytes of an [rows, cols] matrix quantised along cols."""
    if scale_layout == SF_TILED:
        return ((rows + 127) // 128) * ((cols + 127) // 128) * 512
    return rows * (cols // 32)


def mxfp8_quantize(x: torch.Tensor, axis: int = QUANT_ROWWISE, fmt: int = FP8_E5M2,
                   row_index: torch.Tensor | None = None, scale_layout: int = SF_TILED, stream=None):
    """mxfp8_quantize on a bf16 [src_rows, cols] tensor.  Returns (codes uint8, scales uint8).
    ROWWISE: codes [rows, cols]; COLWISE: codes of the transposed matrix [cols, rows]."""
    _need_cuda(x, row_index)
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    src_rows, cols = x.shape
    rows = row_index.numel() if row_index is not None else src_rows
    if axis == QUANT_ROWWISE:
        q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
        sf = torch.zeros(sf_bytes(rows, cols, scale_layout), dtype=torch.uint8, device=x.device)
    else:
        q = torch.empty(cols, rows, dtype=torch.uint8, device=x.device)
        sf = torch.zeros(sf_bytes(cols, rows, scale_layout), dtype=torch.uint8, device=x.device)
    rc = lib().mxfp8_quantize(_ptr(x), src_rows, rows, cols, cols, _ptr(row_index), axis, fmt, _ptr(q),
                              _ptr(sf), scale_layout, _stream(stream))
    _check(rc, "mxfp8_quantize")
    return q, sf


def quantize_weights(W: torch.Tensor, fmt: int = FP8_E4M3, stream=None):
    """Pre-quantise expert weights [E, R, C] along C (the contraction of their GEMM) as the [E*R, C]
    matrix with tiled scales, the layout moe_bwd expects for W1_q/W1_sf, W2_q/W2_sf and (given the
    per-expert transpose of W1) W1t_q/W1t_sf."""
    E, R, C = W.shape
    return mxfp8_quantize(W.reshape(E * R, C), QUANT_ROWWISE, fmt, None, SF_TILED, stream)


class MoeBwd:
    """One MoE backward problem bound to device buffers: outputs and workspace are allocated once,
    run() enqueues moe_bwd on the stream (no host synchronisation)."""

    def __init__(self, *, T, H, I, E, K, block_size, precision=PREC_BF16, affinity=AFFINITY_ON_H,
                 fp8_act=FP8_E5M2, fp8_w=FP8_E4M3, has_bias=False, accumulate=False, act_src=ACT_CHECKPOINT,
                 ds_masked=False, glu=GLU_SWIGLU, gate_up_layout=GATE_UP_CONCAT, device="cuda"):
        self.a = MoeBwdArgs()
        self.a.glu = int(glu)
        self.a.gate_up_layout = int(gate_up_layout)
        self.a.accumulate = int(bool(accumulate))
        self.a.act_src = int(act_src)
        for k, v in dict(T=T, H=H, I=I, E=E, K=K, block_size=block_size, precision=precision,
                         affinity=affinity, fp8_act=fp8_act, fp8_w=fp8_w, has_bias=int(bool(has_bias))).items():
            setattr(self.a, k, int(v))
        self.device = torch.device(device)
        size = lib().moe_bwd_workspace_size(ctypes.byref(self.a))
        if size == 0:
            raise MoeError(f"unsupported moe_bwd configuration: {lib().moe_last_error().decode()}")
        self.workspace = _ws(size, self.device)
        dev = self.device
        self.dx = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.dW1 = torch.empty(E, H, 2 * I, dtype=torch.bfloat16, device=dev)
        self.dW2 = torch.empty(E, I, H, dtype=torch.bfloat16, device=dev)
        self.ds = torch.empty(T, K, dtype=torch.float32, device=dev)
        self.db1 = torch.empty(E, 2 * I, dtype=torch.float32, device=dev) if has_bias else None
        self.db2 = torch.empty(E, H, dtype=torch.float32, device=dev) if has_bias else None
        self.ds_masked = torch.empty(T * E, dtype=torch.float32, device=dev) if ds_masked else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self._keep = []

    def bind(self, *, x, dout, s, ids, ckpt=None, W1=None, W2=None, W1_q=None, W1_sf=None, W2_q=None, W2_sf=None,
             b2=None, W1t=None, W1t_q=None, W1t_sf=None, b1=None, num_valid_tokens=None, intermediate_ckpt=None,
             scaled_intermediate_ckpt=None, down_proj_act_ckpt=None, gate_act_ckpt=None, route_meta=None):
        """ckpt: the [N,2,I,B] checkpoint (act_src ACT_CHECKPOINT).  W1t (bf16 [E,2I,H]) or W1t_q/W1t_sf
        and optionally b1 [E,2I]: the operands of the recomputation (act_src ACT_RECOMPUTE).
        intermediate_ckpt / scaled_intermediate_ckpt / gate_act_ckpt [N,I,B] and down_proj_act_ckpt
        [N,B,H] (bf16, block layout): saved forward values, see the MoeBwdArgs fields.
        route_meta: routing metadata from the caller (a dict with int32 CUDA tensors expert_offsets,
        s_scatter_idx, block_offsets and optionally token_position_to_id, block_to_expert -- e.g.
        route_meta()'s result); None: moe_bwd computes it from ids."""
        _need_cuda(x, dout, s, ids, ckpt, W1, W2, W1_q, W1_sf, W2_q, W2_sf, b2, W1t, W1t_q, W1t_sf, b1, num_valid_tokens,
                   intermediate_ckpt, scaled_intermediate_ckpt, down_proj_act_ckpt, gate_act_ckpt)
        if num_valid_tokens is not None:
            assert num_valid_tokens.dtype == torch.int32 and num_valid_tokens.numel() == 1
        a = self.a
        Nb = num_blocks_bound(a.T, a.K, a.E, a.block_size)
        for t in (intermediate_ckpt, scaled_intermediate_ckpt, gate_act_ckpt):
            assert t is None or (t.dtype == torch.bfloat16 and tuple(t.shape) == (Nb, a.I, a.block_size))
        assert down_proj_act_ckpt is None or (down_proj_act_ckpt.dtype == torch.bfloat16 and
                                              tuple(down_proj_act_ckpt.shape) == (Nb, a.block_size, a.H))
        assert x.dtype == torch.bfloat16 and dout.dtype == torch.bfloat16
        assert s.dtype == torch.float32 and ids.dtype == torch.int32
        assert tuple(x.shape) == (a.T, a.H) and tuple(dout.shape) == (a.T, a.H)
        assert tuple(s.shape) == (a.T, a.K) and tuple(ids.shape) == (a.T, a.K)
        if ckpt is not None:
            N = num_blocks_bound(a.T, a.K, a.E, a.block_size)
            assert ckpt.dtype == torch.bfloat16
            assert tuple(ckpt.shape) == (N, 2, a.I, a.block_size), (tuple(ckpt.shape), N)
        if W1t is not None:
            assert W1t.dtype == torch.bfloat16 and tuple(W1t.shape) == (a.E, 2 * a.I, a.H)
        if b1 is not None:
            assert b1.dtype == torch.bfloat16 and tuple(b1.shape) == (a.E, 2 * a.I)
        for name, t in dict(x=x, dout=dout, s=s, ids=ids, gate_up_ckpt=ckpt, W1=W1, W2=W2, W1_q=W1_q,
                            W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf, b2=b2, W1t=W1t, W1t_q=W1t_q, W1t_sf=W1t_sf,
                            b1=b1, num_valid_tokens=num_valid_tokens, intermediate_ckpt=intermediate_ckpt,
                            scaled_intermediate_ckpt=scaled_intermediate_ckpt,
                            down_proj_act_ckpt=down_proj_act_ckpt, gate_act_ckpt=gate_act_ckpt).items():
            setattr(a, name, None if t is None else t.data_ptr())
        for name in ("dx", "dW1", "dW2", "ds", "db1", "db2", "ds_masked", "status"):
            t = getattr(self, name)
            setattr(a, "status_dev" if name == "status" else name, None if t is None else t.data_ptr())
        rm = {k: (route_meta or {}).get(k) for k in ROUTE_META_FIELDS}
        for k, t in rm.items():
            _need_cuda(t)
            assert t is None or t.dtype == torch.int32, k
            setattr(a, k, None if t is None else t.data_ptr())
        a.workspace = self.workspace.data_ptr()
        a.workspace_bytes = self.workspace.numel()
        self._keep = [x, dout, s, ids, ckpt, W1, W2, W1_q, W1_sf, W2_q, W2_sf, b2, W1t, W1t_q, W1t_sf, b1,
                      num_valid_tokens, intermediate_ckpt, scaled_intermediate_ckpt, down_proj_act_ckpt, gate_act_ckpt,
                      *rm.values()]
        return self

    def run(self, stream=None):
        _check(lib().moe_bwd(ctypes.byref(self.a), _stream(stream)), "moe_bwd")
        return self

    def outputs(self) -> dict:
        return dict(dx=self.dx, dW1=self.dW1, dW2=self.dW2, ds=self.ds, db1=self.db1, db2=self.db2,
                    ds_masked=self.ds_masked, status=self.status)

    def region(self, name: str) -> torch.Tensor:
        """Bytes of one workspace region (see MOE_WS_* in include/moebwd.h)."""
        off, nb = ctypes.c_size_t(), ctypes.c_size_t()
        rc = lib().moe_bwd_workspace_region(ctypes.byref(self.a), WS_REGIONS.index(name), ctypes.byref(off),
                                            ctypes.byref(nb))
        _check(rc, "moe_bwd_workspace_region")
        return self.workspace[off.value: off.value + nb.value]

    @property
    def tile_rows(self) -> int:
        return tile_rows_capacity(self.a.T, self.a.K, self.a.E)


def moe_bwd(*, x, dout, s, ids, E, I, block_size, ckpt=None, W1=None, W2=None, W1_q=None, W1_sf=None, W2_q=None,
            W2_sf=None, b2=None, W1t=None, W1t_q=None, W1t_sf=None, b1=None, precision=PREC_BF16,
            affinity=AFFINITY_ON_H, fp8_act=FP8_E5M2, fp8_w=FP8_E4M3, accumulate=False, stream=None) -> dict:
    """One-shot MoE backward (allocates outputs and workspace).  Returns dx, dW1, dW2, ds, db1, db2
    and the device status word (nonzero: invalid expert ids or a pipeline timeout).  Without ckpt the
    gate/up pre-activations are recomputed from x and W1t (or W1t_q/W1t_sf) plus b1."""
    T, H = x.shape
    K = ids.shape[1]
    op = MoeBwd(T=T, H=H, I=I, E=E, K=K, block_size=block_size, precision=precision, affinity=affinity,
                fp8_act=fp8_act, fp8_w=fp8_w, has_bias=b2 is not None, accumulate=accumulate,
                act_src=ACT_CHECKPOINT if ckpt is not None else ACT_RECOMPUTE, device=x.device)
    op.bind(x=x, dout=dout, s=s, ids=ids, ckpt=ckpt, W1=W1, W2=W2, W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q,
            W2_sf=W2_sf, b2=b2, W1t=W1t, W1t_q=W1t_q, W1t_sf=W1t_sf, b1=b1).run(stream)
    out = op.outputs()
    out["_op"] = op
    return out


ROUTER_SOFTMAX_OVER_TOPK, ROUTER_TOPK_OVER_SOFTMAX, ROUTER_TOPK = 0, 1, 2


def router_bwd(mode: int, ids: torch.Tensor, dscores: torch.Tensor, E: int, logits=None, scores=None,
               renorm: bool = False, stream=None) -> torch.Tensor:
    """moe_router_bwd: gradient of the router logits [T, E] from the scores' gradient [T, K]."""
    _need_cuda(ids, dscores, logits, scores)
    T, K = ids.shape
    out = torch.empty(T, E, dtype=torch.float32, device=ids.device)
    rc = lib().moe_router_bwd(mode, int(renorm), _ptr(logits), _ptr(scores), _ptr(dscores), _ptr(ids), T, K, E,
                              _ptr(out), _stream(stream))
    _check(rc, "moe_router_bwd")
    return out


class LinearBwd:
    """Dense linear backward dX = dY @ W, dW = dY^T @ X with buffers allocated once."""

    def __init__(self, M, N, K, precision=PREC_MXFP8, fp8=FP8_E5M2, device="cuda"):
        self.M, self.N, self.K, self.precision, self.fp8 = M, N, K, precision, fp8
        dev = torch.device(device)
        self.workspace = _ws(lib().linear_bwd_workspace_size(M, N, K, precision), dev)
        self.dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(N, K, dtype=torch.bfloat16, device=dev)

    def run(self, dY, W, X, stream=None):
        _need_cuda(dY, W, X)
        rc = lib().linear_bwd(_ptr(dY), _ptr(W), _ptr(X), self.M, self.N, self.K, self.precision, self.fp8,
                              _ptr(self.dX), _ptr(self.dW), _ptr(self.workspace), self.workspace.numel(),
                              _stream(stream))
        _check(rc, "linear_bwd")
        return self


def linear_bwd(dY, W, X, precision=PREC_MXFP8, fp8=FP8_E5M2, stream=None):
    M, N = dY.shape
    K = X.shape[1]
    op = LinearBwd(M, N, K, precision, fp8, dY.device).run(dY, W, X, stream)
    return dict(dX=op.dX, dW=op.dW)
