"""Seeded synthetic inputs for the MoE expert-layer backward and the dense MXFP8 linear backward.

This module is shared by the tests, the benchmark and the smoke check.  It only draws random
numbers and builds the forward router's top-K selection (softmax over logits, top-K, renormalise),
which is how the routing inputs of the backward are produced; it holds none of the backward's
arithmetic.  Every tensor is created from an explicit seed.

Workloads (shapes follow the problem statement of the blockwise MoE backward page, "Dimensions"
list, and the dense matmul backward page, "Forward pass convention"):

  tiny_bf16          T=256   H=128  I=256  E=4   K=2  B=128  BF16  affinity on H, no bias
  dense_mxfp8_4096   M=N=K=4096 dense linear backward, MXFP8 e5m2 on every operand
  finegrained_bf16   T=16384 H=2048 I=1024 E=64  K=8  B=128  BF16  affinity on H, biases
  manyexpert_mxfp8   T=32768 H=2048 I=768  E=128 K=8  B=256  MXFP8 affinity on I
  imbalanced_mxfp8   T=65536 H=4096 I=1536 E=128 K=8  B=512  MXFP8 affinity on I, Zipf routing
plus reduced shapes (profile_*) used only to size ncu captures.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

AFFINITY_ON_H = 0
AFFINITY_ON_I = 1
PREC_BF16 = 0
PREC_MXFP8 = 1
FP8_E4M3 = 0
FP8_E5M2 = 1


@dataclass(frozen=True)
class MoeConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    block_size: int
    precision: int = PREC_BF16
    affinity: int = AFFINITY_ON_H
    bias: bool = False
    zipf_alpha: float = 0.0          # 0 = plain N(0,1) logits
    fp8_act: int = FP8_E5M2
    fp8_w: int = FP8_E4M3
    seed: int = 1000

    @property
    def TK(self) -> int:
        return self.T * self.K

    def useful_flops(self) -> int:
        """12*T*K*H*I: three GEMMs of 2*TK*H*I (G1, G3 over I) and two of 4*TK*H*I (G2, G4 over 2I)."""
        return 12 * self.T * self.K * self.H * self.I


@dataclass(frozen=True)
class LinearConfig:
    name: str
    M: int
    N: int
    K: int
    fp8: int = FP8_E5M2
    w_scale: float = 0.02
    seed: int = 1001

    def useful_flops(self) -> int:
        return 4 * self.M * self.N * self.K


CONFIGS = {
    "tiny_bf16": MoeConfig("tiny_bf16", T=256, H=128, I=256, E=4, K=2, block_size=128, seed=1000),
    "dense_mxfp8_4096": LinearConfig("dense_mxfp8_4096", M=4096, N=4096, K=4096, seed=1001),
    "finegrained_bf16": MoeConfig("finegrained_bf16", T=16384, H=2048, I=1024, E=64, K=8,
                                  block_size=128, bias=True, seed=1002),
    "manyexpert_mxfp8": MoeConfig("manyexpert_mxfp8", T=32768, H=2048, I=768, E=128, K=8,
                                  block_size=256, precision=PREC_MXFP8, affinity=AFFINITY_ON_I,
                                  seed=1003),
    "imbalanced_mxfp8": MoeConfig("imbalanced_mxfp8", T=65536, H=4096, I=1536, E=128, K=8,
                                  block_size=512, precision=PREC_MXFP8, affinity=AFFINITY_ON_I,
                                  zipf_alpha=1.2, seed=1004),
    # reduced shapes of the two MoE paths for kernel profiling (inputs > L2, a few GB in total)
    "profile_mxfp8_small": MoeConfig("profile_mxfp8_small", T=8192, H=2048, I=768, E=32, K=8,
                                     block_size=256, precision=PREC_MXFP8, affinity=AFFINITY_ON_I,
                                     seed=1005),
    "profile_mxfp8_medium": MoeConfig("profile_mxfp8_medium", T=16384, H=4096, I=768, E=32, K=8,
                                      block_size=256, precision=PREC_MXFP8, affinity=AFFINITY_ON_I,
                                      seed=1007),
    "profile_bf16_small": MoeConfig("profile_bf16_small", T=8192, H=2048, I=1024, E=32, K=8,
                                    block_size=128, bias=True, seed=1006),
}


def num_blocks_bound(T: int, K: int, E: int, B: int) -> int:
    """Block-count bound N = ceil((T*K - (E-1)) / B) + E - 1 (at least 1 when T*K > 0)."""
    TK = T * K
    if TK <= 0:
        return 0
    num = TK - (E - 1)
    if num <= 0:
        return TK  # fewer rows than experts: at most one block per routed row
    return -(-num // B) + E - 1


def _topk_route(logits: torch.Tensor, K: int):
    """Forward router: softmax over all experts, top-K, renormalise the K kept scores."""
    p = torch.softmax(logits.float(), dim=-1)
    s, ids = torch.topk(p, K, dim=-1)
    s = s / s.sum(dim=-1, keepdim=True)
    return s.float().contiguous(), ids.to(torch.int32).contiguous()


def _zipf_bias(E: int, alpha: float, gen: torch.Generator, device) -> torch.Tensor:
    ranks = torch.randperm(E, generator=gen, device=device).to(torch.float32) + 1.0
    return -alpha * torch.log(ranks)


def _route(cfg: MoeConfig, gen: torch.Generator, device):
    logits = torch.randn(cfg.T, cfg.E, generator=gen, device=device)
    if cfg.zipf_alpha <= 0.0:
        return _topk_route(logits, cfg.K) + (None, logits)
    bias = _zipf_bias(cfg.E, cfg.zipf_alpha, gen, device)

    def loads(c):
        _, ids = _topk_route(logits + c * bias, cfg.K)
        return torch.bincount(ids.flatten().long(), minlength=cfg.E)

    # Smallest bias strength (bisection on a fixed seed) at which the hottest expert takes at least
    # 90% of the tokens (the ceiling with distinct top-K ids is 100% = E/K times the mean) and at
    # least one expert receives no token.
    lo, hi = 0.0, 64.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        ld = loads(mid)
        if ld.max().item() >= 0.9 * cfg.T and (ld == 0).any().item():
            hi = mid
        else:
            lo = mid
    s, ids = _topk_route(logits + hi * bias, cfg.K)
    return s, ids, hi, logits + hi * bias


@dataclass
class MoeInputs:
    cfg: MoeConfig
    x: torch.Tensor          # [T,H] bf16
    dout: torch.Tensor       # [T,H] bf16
    W1: torch.Tensor         # [E,H,2I] bf16, columns 0..I-1 gate, I..2I-1 up
    W2: torch.Tensor         # [E,I,H] bf16
    b1: torch.Tensor | None  # [E,2I] bf16
    b2: torch.Tensor | None  # [E,H] bf16
    s: torch.Tensor          # [T,K] fp32 routing scores (renormalised)
    ids: torch.Tensor        # [T,K] int32 expert ids
    ckpt: torch.Tensor       # [N,2,I,B] bf16 gate/up pre-activation checkpoint (block layout)
    zipf_strength: float | None = None
    extra: dict = field(default_factory=dict)


def make_moe_inputs(cfg: MoeConfig, device="cpu") -> MoeInputs:
    """All tensors of one MoE backward problem, drawn from cfg.seed on `device`.

    x, dout ~ N(0,1); W1, W2 ~ N(0, 0.02^2); b1, b2 ~ N(0, 0.01^2); routing from N(0,1) logits
    (plus a Zipf per-expert bias when cfg.zipf_alpha > 0).  The gate/up checkpoint is the forward's
    saved pre-activation in the block layout [N, 2, I, B]; it is drawn as N(0, (0.02*sqrt(H))^2),
    the spread of x @ W1 under the stated initialisation, for every slot (padding slots included:
    they are never read).  The same tensors go to the GPU library and to the oracle.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(cfg.seed)
    T, H, I, E, K, B = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.block_size
    x = torch.randn(T, H, generator=gen, device=device).to(torch.bfloat16)
    dout = torch.randn(T, H, generator=gen, device=device).to(torch.bfloat16)
    W1 = (torch.randn(E, H, 2 * I, generator=gen, device=device) * 0.02).to(torch.bfloat16)
    W2 = (torch.randn(E, I, H, generator=gen, device=device) * 0.02).to(torch.bfloat16)
    b1 = b2 = None
    if cfg.bias:
        b1 = (torch.randn(E, 2 * I, generator=gen, device=device) * 0.01).to(torch.bfloat16)
        b2 = (torch.randn(E, H, generator=gen, device=device) * 0.01).to(torch.bfloat16)
    s, ids, zs, logits = _route(cfg, gen, device)
    N = num_blocks_bound(T, K, E, B)
    ckpt = (torch.randn(N, 2, I, B, generator=gen, device=device) * (0.02 * math.sqrt(H))).to(torch.bfloat16)
    return MoeInputs(cfg, x, dout, W1, W2, b1, b2, s, ids, ckpt, zs, extra=dict(logits=logits.float().contiguous()))


@dataclass
class LinearInputs:
    cfg: LinearConfig
    X: torch.Tensor   # [M,K] bf16
    W: torch.Tensor   # [N,K] bf16
    dY: torch.Tensor  # [M,N] bf16


def make_linear_inputs(cfg: LinearConfig, device="cpu") -> LinearInputs:
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(cfg.seed)
    X = torch.randn(cfg.M, cfg.K, generator=gen, device=device).to(torch.bfloat16)
    W = (torch.randn(cfg.N, cfg.K, generator=gen, device=device) * cfg.w_scale).to(torch.bfloat16)
    dY = torch.randn(cfg.M, cfg.N, generator=gen, device=device).to(torch.bfloat16)
    return LinearInputs(cfg, X, W, dY)


def small_moe(name="small", T=256, H=128, I=256, E=4, K=2, B=128, seed=7, **kw) -> MoeConfig:
    """A custom small MoE configuration (tests use it for ragged and degenerate cases)."""
    return MoeConfig(name, T=T, H=H, I=I, E=E, K=K, block_size=B, seed=seed, **kw)


def with_ids(inp: MoeInputs, ids: torch.Tensor, s: torch.Tensor | None = None) -> MoeInputs:
    """Replace the routing of a problem (tests use it for hand-made expert loads)."""
    cfg = inp.cfg
    N = num_blocks_bound(cfg.T, cfg.K, cfg.E, cfg.block_size)
    ckpt = inp.ckpt
    if ckpt.shape[0] < N:
        gen = torch.Generator(device=ckpt.device).manual_seed(cfg.seed + 17)
        ckpt = (torch.randn(N, 2, cfg.I, cfg.block_size, generator=gen, device=ckpt.device)
                * (0.02 * math.sqrt(cfg.H))).to(torch.bfloat16)
    return replace(inp, ids=ids.to(torch.int32).contiguous(),
                   s=(inp.s if s is None else s.float().contiguous()), ckpt=ckpt)
