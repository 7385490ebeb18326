"""The fold on the GPU against the oracle, pair by pair: every finite 16-bit
value against every exponent and sign of the other operand.

Section "Op" of TensorRT-LLM PR #20546 fixes the bits of each fold addition:
a float32 round-to-nearest addition, rounded to the element format with
subnormals kept.  The kernels add the two 16-bit operands with one paired
16-bit addition, which rounds the exact sum once; these tests check that the
two give the same bits over the operand space (the oracle rounds the exact
float64 sum once).  BF16 and FP16, through the standalone fold kernel and
through the fused kernel's fold."""
import numpy as np
import pytest
import torch

from kimi_k3_attention_gb300 import binding
from kimi_k3_attention_gb300 import workloads as wl
from oracle import bf16_decode, fold, fp16_decode

from gpu_helpers import Guarded, run_gpu, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


FORMATS = {
    # name: (torch dtype, decode, exponent field mask, mantissa bits, max exponent field)
    "bf16": (torch.bfloat16, bf16_decode, 0x7F80, 7, 254),
    "fp16": (torch.float16, fp16_decode, 0x7C00, 10, 30),
}


def _operands(fmt, seed, per_exponent):
    """a: every finite pattern; b: for every exponent field value and both
    signs, `per_exponent` random mantissas (the first exponent, zeros and
    subnormals, also takes mantissa 0 and the largest).  Returns the flat
    (a, b) pairs of their product, padded to a multiple of 8."""
    dt, dec, emask, mbits, emax = FORMATS[fmt]
    allb = np.arange(65536, dtype=np.uint16)
    allb = allb[np.isfinite(dec(allb))]
    rng = np.random.default_rng(seed)
    exps = np.arange(emax + 1, dtype=np.uint16) << mbits
    mant = rng.integers(0, 1 << mbits, (exps.size, per_exponent)).astype(np.uint16)
    picks = np.concatenate([(exps[:, None] | mant).ravel(), [0, (1 << mbits) - 1]]).astype(np.uint16)
    picks = np.concatenate([picks, picks | 0x8000])
    a = np.tile(allb, picks.size)
    b = np.repeat(picks, allb.size)
    pad = (-a.size) % 8
    return np.concatenate([a, np.zeros(pad, np.uint16)]), np.concatenate([b, np.zeros(pad, np.uint16)])


def _tensor(bits, dt, shape):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dt).view(*shape)


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_standalone_fold_every_exponent_pair(fmt):
    """new_prefix = prefix + add (no second addend) through the standalone
    fold kernel: one paired addition per element."""
    dt = FORMATS[fmt][0]
    a, b = _operands(fmt, seed=101, per_exponent=1 if fmt == "bf16" else 2)
    Hs = 8192
    M = -(-a.size // Hs)
    total = M * Hs
    a = np.resize(a, total)
    b = np.resize(b, total)
    ref, _ = fold(a, b, None, fmt)
    P = _tensor(a, dt, (M, Hs)).cuda()
    A = _tensor(b, dt, (M, Hs)).cuda()
    newp = Guarded((M, Hs), dtype=dt)
    binding.attnres_tail_add(P, A, None, newp.t)
    torch.cuda.synchronize()
    assert newp.guards_intact()
    got = u16(newp.t).ravel()
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (fmt, bad.size, hex(a[bad[0]]), hex(b[bad[0]]), hex(got[bad[0]]),
                           hex(ref[bad[0]]))


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_fused_fold_inner_addition_every_exponent_pair(fmt):
    """The fused kernel's inner addition s = add + add2 with prefix +0 (so
    new_prefix = +0 + s; the oracle takes the same two roundings)."""
    dt = FORMATS[fmt][0]
    a, b = _operands(fmt, seed=202, per_exponent=1 if fmt == "bf16" else 2)
    Hs = 7168
    M = -(-a.size // Hs)
    total = M * Hs
    a = np.resize(a, total)
    b = np.resize(b, total)
    p = np.zeros(total, np.uint16)
    ref, _ = fold(p, a, b, fmt)
    inp = wl.make_inputs(M, 1, Hs, seed=7, dtype=dt)
    inp.prefix, inp.add, inp.add2 = _tensor(p, dt, (M, Hs)), _tensor(a, dt, (M, Hs)), _tensor(b, dt, (M, Hs))
    inp.bank.zero_()
    gnp, _ = run_gpu(inp)
    got = gnp.ravel()
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (fmt, bad.size, hex(a[bad[0]]), hex(b[bad[0]]), hex(got[bad[0]]),
                           hex(ref[bad[0]]))


@pytest.mark.parametrize("M,Hs", [(1, 8), (3, 24), (32, 7168), (77, 16384)])
@pytest.mark.parametrize("add2", [True, False])
def test_fp16_tail_add_bit_exact(M, Hs, add2):
    """The standalone fold on FP16 tensors: subnormal and near-cancelling
    addends, +-0 and subnormal prefixes, bit-exact to the oracle's FP16 fold."""
    rng = np.random.default_rng(M * 31 + Hs)
    n = M * Hs
    inp = wl.make_inputs(M, 1, Hs, seed=M + Hs, dtype=torch.float16)
    p, a, a2 = (u16(x).ravel().copy() for x in (inp.prefix, inp.add, inp.add2))
    pos = rng.permutation(n)[: n // 2]
    sub, can = pos[: len(pos) // 2], pos[len(pos) // 2:]
    rs = lambda k: (rng.integers(1, 1024, k) | (rng.integers(0, 2, k) << 15)).astype(np.uint16)  # noqa: E731
    a[sub], a2[sub], p[sub] = rs(len(sub)), rs(len(sub)), rs(len(sub))
    a2[can] = ((a[can].astype(np.int64) ^ 0x8000) + rng.integers(-2, 3, len(can))).clip(0, 0xFFFF)
    p[can] = (rng.integers(0, 2, len(can)) << 15).astype(np.uint16)
    dt = torch.float16
    P, A, A2 = (_tensor(x, dt, (M, Hs)).cuda() for x in (p, a, a2))
    newp = Guarded((M, Hs), dtype=dt)
    binding.attnres_tail_add(P, A, A2 if add2 else None, newp.t)
    torch.cuda.synchronize()
    assert newp.guards_intact()
    ref, _ = fold(p, a, a2 if add2 else None, "fp16")
    assert (u16(newp.t).ravel() == ref).all()
    # in place: new_prefix is prefix
    Q = P.clone()
    binding.attnres_tail_add(Q, A, A2 if add2 else None, Q)
    torch.cuda.synchronize()
    assert (u16(Q).ravel() == ref).all()
