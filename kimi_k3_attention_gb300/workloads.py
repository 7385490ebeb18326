"""Seeded synthetic inputs for the fused AttnRes + add2 + RMSNorm epilogue.

This module only draws random tensors; it holds none of the op's arithmetic,
so both the CUDA path and the CPU oracle can be fed from it.  Every tensor is
drawn in float32 from a seeded torch.Generator and rounded to BF16 (or, for
the FP16 workloads, FP16) by torch.

Distributions (the second parameter of N(0, x) is a variance):
  prefix, add, add2, bank ~ N(0, 1);  w ~ N(0, 1/H);  gamma = 1 + 0.1 N(0, 1)
Shapes: prefix/add/add2/new_prefix/out [M, H]; bank [N, M, H]; w, gamma [H].
H = 7168 is the hidden size of the model the epilogue serves (TensorRT-LLM PR
#20546, section "Model"); N = 1..12 bank snapshots and 1..32 decode tokens are
the fused window of the same page.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch

H_MODEL = 7168
EPS = 1e-6


@dataclass
class Inputs:
    prefix: torch.Tensor
    add: torch.Tensor
    add2: Optional[torch.Tensor]
    bank: torch.Tensor
    w: torch.Tensor
    gamma: torch.Tensor
    eps: float = EPS

    @property
    def M(self) -> int:
        return self.prefix.shape[0]

    @property
    def N(self) -> int:
        return self.bank.shape[0]

    @property
    def H(self) -> int:
        return self.prefix.shape[1]

    def to(self, device) -> "Inputs":
        mv = lambda t: None if t is None else t.to(device).contiguous()  # noqa: E731
        return Inputs(mv(self.prefix), mv(self.add), mv(self.add2), mv(self.bank),
                      mv(self.w), mv(self.gamma), self.eps)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device="cpu", dtype=torch.bfloat16):
    return (torch.randn(shape, generator=g, dtype=torch.float32, device=device) * std).to(dtype)


def make_inputs(M, N, H=H_MODEL, seed=0, add2=True, device="cpu", eps=EPS,
                dtype=torch.bfloat16) -> Inputs:
    """Standard N(0,1) workload.  Draw order: prefix, add, add2, bank, w, gamma.
    dtype: torch.bfloat16 (the model's) or torch.float16."""
    g = _gen(seed, device)
    prefix = _normal((M, H), 1.0, g, device, dtype)
    add = _normal((M, H), 1.0, g, device, dtype)
    a2 = _normal((M, H), 1.0, g, device, dtype) if add2 else None
    bank = _normal((N, M, H), 1.0, g, device, dtype)
    w = _normal((H,), 1.0 / math.sqrt(H), g, device, dtype)
    gamma = (1.0 + 0.1 * torch.randn((H,), generator=g, dtype=torch.float32, device=device)).to(dtype)
    return Inputs(prefix, add, a2, bank, w, gamma, eps)


def pr_reference_case() -> Inputs:
    """M=4 tokens, N=3 snapshots, H=7168, add2 present, seed 0."""
    return make_inputs(4, 3, H_MODEL, seed=0, add2=True)


def decode_sweep_cases():
    """M in {1,8,16,32} x N in 1..12 x add2 in {present, absent}: 96 cases,
    seed 1000 + case index.  Yields (case_index, M, N, has_add2)."""
    idx = 0
    for M in (1, 8, 16, 32):
        for N in range(1, 13):
            for has_add2 in (True, False):
                yield idx, M, N, has_add2
                idx += 1


def decode_sweep_inputs(idx, M, N, has_add2, H=H_MODEL, device="cpu") -> Inputs:
    return make_inputs(M, N, H, seed=1000 + idx, add2=has_add2, device=device)


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16).to(torch.int32) & 0xFFFF


def _from_bits(b: torch.Tensor) -> torch.Tensor:
    b = b.to(torch.int32)
    b = torch.where(b >= 32768, b - 65536, b)
    return b.to(torch.int16).view(torch.bfloat16)


def stress_inputs(M=32, N=12, H=H_MODEL, seed=7, special_prefix=False) -> Inputs:
    """Bit-exactness stress.  25% of the (m, j) positions are special: half get
    BF16 subnormal add/add2 (mantissa 1..127, random signs), half get
    near-cancelling pairs add ~ N(0,1), add2 = -add moved by k in {-2..2} ulp.
    The rest: add, add2 ~ N(0, 1e-3).  prefix, bank ~ N(0, 1).
    special_prefix=True also makes prefix +-0 or a random subnormal at the
    special positions, so subnormal sums reach the updated prefix."""
    g = _gen(seed)
    P = M * H
    prefix = _normal((M, H), 1.0, g)
    add = _normal((M, H), math.sqrt(1e-3), g)
    add2 = _normal((M, H), math.sqrt(1e-3), g)
    bank = _normal((N, M, H), 1.0, g)
    w = _normal((H,), 1.0 / math.sqrt(H), g)
    gamma = (1.0 + 0.1 * torch.randn((H,), generator=g, dtype=torch.float32)).to(torch.bfloat16)

    perm = torch.randperm(P, generator=g)
    n_special = P // 4
    sub_pos = perm[: n_special // 2]
    can_pos = perm[n_special // 2: n_special]

    ab = _bits(add).reshape(-1).clone()
    a2b = _bits(add2).reshape(-1).clone()
    pb = _bits(prefix).reshape(-1).clone()

    def rand_sub(n):
        mant = torch.randint(1, 128, (n,), generator=g, dtype=torch.int32)
        sign = torch.randint(0, 2, (n,), generator=g, dtype=torch.int32) << 15
        return mant | sign

    ab[sub_pos] = rand_sub(len(sub_pos))
    a2b[sub_pos] = rand_sub(len(sub_pos))

    base = _bits(_normal((len(can_pos),), 1.0, g))
    k = torch.randint(-2, 3, (len(can_pos),), generator=g, dtype=torch.int32)
    mag = torch.clamp((base & 0x7FFF) + k, min=0)
    ab[can_pos] = base
    a2b[can_pos] = (base & 0x8000) ^ 0x8000 | mag

    if special_prefix:
        sp = torch.cat([sub_pos, can_pos])
        half = len(sp) // 2
        zeros = torch.randint(0, 2, (half,), generator=g, dtype=torch.int32) << 15
        pb[sp[:half]] = zeros
        pb[sp[half:]] = rand_sub(len(sp) - half)

    return Inputs(_from_bits(pb).reshape(M, H), _from_bits(ab).reshape(M, H),
                  _from_bits(a2b).reshape(M, H), bank, w, gamma, EPS)


@dataclass
class ChainLayer:
    w: torch.Tensor
    gamma: torch.Tensor
    routed: torch.Tensor
    shared: torch.Tensor


def chain_inputs(M=8, H=H_MODEL, layers=25, seed=2546):
    """25-layer decoder chain with deferred MoE tails.

    Returns (embedding [M,H], P0 [M,H], [ChainLayer] * layers).  Layer l gets
    its own w_l, gamma_l and the tail (routed, shared) ~ N(0, 0.5) that the
    previous MoE layer deferred (layer 0's tail is drawn too).  The bank
    starts as [embedding]; the schedule of bank appends is the caller's."""
    g = _gen(seed)
    emb = _normal((M, H), 1.0, g)
    p0 = _normal((M, H), 1.0, g)
    out = []
    for _ in range(layers):
        w = _normal((H,), 1.0 / math.sqrt(H), g)
        gamma = (1.0 + 0.1 * torch.randn((H,), generator=g, dtype=torch.float32)).to(torch.bfloat16)
        routed = _normal((M, H), math.sqrt(0.5), g)
        shared = _normal((M, H), math.sqrt(0.5), g)
        out.append(ChainLayer(w, gamma, routed, shared))
    return emb, p0, out


def chain_appends_after(layer: int, last_append: int = 21) -> bool:
    """The bank grows 1 -> 12: a copy of the carried prefix is appended after
    every odd layer up to 21, so layers 22..24 run with N = 12.  A deeper
    chain (61 layers, last_append = 59) grows the bank to 31 snapshots."""
    return layer % 2 == 1 and layer <= last_append


def bandwidth_inputs(device="cuda", seed=4, M=8192, N=12, H=H_MODEL, add2=True,
                     dtype=torch.bfloat16) -> Inputs:
    """M=8192 tokens, N=12, H=7168, add2 present: ~2.0 GB per call.  Drawn on
    `device` (a CUDA generator when device is a GPU) to keep set-up short."""
    return make_inputs(M, N, H, seed=seed, add2=add2, device=device, dtype=dtype)
