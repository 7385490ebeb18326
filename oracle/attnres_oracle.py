"""CPU oracle for the fused AttnRes + add2 + RMSNorm decode epilogue.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain reference that the
CUDA library is checked against.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the library itself never does, and
this module imports nothing from the library.

What it computes, per token m (all tensors BF16 bit patterns, H columns):

  (a2) fold     s  = bf16(add + add2)          (s = add when add2 is absent)
                np = bf16(prefix + s)
       Source: TensorRT-LLM PR #20546 ("Kimi K3: fold the MoE-tail additions
       into the next attention-residual"), section "Op": the updated prefix sum
       is bf16(layer_residual + bf16(layer_residual_add + layer_residual_add2)),
       bit for bit the two BF16 tensor additions, subnormals kept.
  (a3) stats    over the N+1 sources v_0..v_{N-1} = bank[0..N-1, m, :] and
                v_N = np[m, :]:  ss_i = sum_j v_ij^2,  d_i = sum_j w_j v_ij
  (a4) logits   l_i = w . RMSNorm(v_i) = d_i / sqrt(ss_i / H + eps);
                alpha = softmax(l)
  (a5) mixture  h_j = sum_i alpha_i v_ij
  (a6) output   out_j = h_j / sqrt(mean(h^2) + eps) * gamma_j
       Steps (a3)-(a6): the attention-residual depth mixture over the snapshot
       bank plus the updated prefix, followed by RMSNorm, as specified for this
       op; the PR pages name the attention-residual + RMSNorm consumer (section
       "Description" and "Op") but do not write its math out.

Arithmetic of the oracle:
  * BF16 is decoded to float64 and encoded back with integer arithmetic only,
    so the host's FTZ/DAZ floating-point state can never touch a subnormal
    (the smallest BF16 subnormal, 2^-133, is a normal float64).
  * The fold adds in float64 and rounds once to BF16 (round to nearest even).
    The exact sum of two BF16 values rounded to float64 (53 bits) and then to
    BF16 (8 bits) equals the correctly rounded BF16 sum, because 53 >= 2*8+2
    (double rounding is innocuous for addition at that width); the same holds
    for the float32 route (24 >= 18) that the PR describes.  Hence both routes
    give the correctly rounded sum, which is what this oracle returns.
  * The mixture and the output norm are evaluated in float64 and NOT rounded:
    the float64 `out` is compared against the GPU's BF16 output within a
    tolerance (see oracle/tolerance.py).
  * FP16 tensors (fmt="fp16", IEEE binary16) take the same steps with the
    FP16 codec: the PR's fused window is BF16 (section "Model"), and the same
    op on a model kept in FP16 is read as every tensor and both fold
    roundings in FP16.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "Format",
    "BF16",
    "FP16",
    "decode",
    "encode_rne",
    "bf16_decode",
    "bf16_encode_rne",
    "fp16_decode",
    "fp16_encode_rne",
    "fold",
    "mixture",
    "attnres_add_rmsnorm",
    "attnres_rmsnorm",
    "algorithmic_bytes",
]

class Format:
    """A binary 16-bit floating-point format: 1 sign bit, `ebits` exponent bits
    (bias 2^(ebits-1) - 1), `mbits` mantissa bits, IEEE-style subnormals,
    infinities and NaNs.  BF16 is (8, 7); FP16 (IEEE binary16) is (5, 10)."""

    def __init__(self, name, ebits, mbits):
        self.name, self.ebits, self.mbits = name, ebits, mbits
        self.bias = (1 << (ebits - 1)) - 1
        self.emax = (1 << ebits) - 2 - self.bias              # largest normal exponent
        self.min_normal = 2.0 ** (1 - self.bias)
        self.sub_exp = 1 - self.bias - mbits                  # subnormal quantum 2^sub_exp
        self.max_finite = (2.0 - 2.0 ** -mbits) * 2.0 ** self.emax
        # Values at or above this magnitude round (to nearest even) to
        # infinity: the midpoint between the largest finite value and
        # 2^(emax+1); the largest finite value's last mantissa bit is odd, so
        # the tie goes up.
        self.overflow = (2.0 - 2.0 ** -(mbits + 1)) * 2.0 ** self.emax
        self.exp_mask = (1 << ebits) - 1
        self.inf_bits = self.exp_mask << mbits
        self.qnan_bits = self.inf_bits | (1 << (mbits - 1))


BF16 = Format("bf16", 8, 7)
FP16 = Format("fp16", 5, 10)
FORMATS = {"bf16": BF16, "fp16": FP16}


def _fmt(fmt) -> Format:
    return fmt if isinstance(fmt, Format) else FORMATS[fmt]


def decode(bits, fmt="bf16") -> np.ndarray:
    """16-bit bit patterns (uint16) of format `fmt` -> exact float64 values.

    Exponent field 0 encodes zero and subnormals (mantissa * 2^sub_exp); the
    all-ones exponent encodes infinities (mantissa 0) and NaN (mantissa != 0);
    otherwise the value is 1.mantissa * 2^(exponent - bias).
    """
    f = _fmt(fmt)
    u = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = (u >> 15) & 1
    e = (u >> f.mbits) & f.exp_mask
    m = u & ((1 << f.mbits) - 1)
    normal_sig = (m + (1 << f.mbits)).astype(np.float64)   # 1.m as an integer * 2^mbits
    sub_sig = m.astype(np.float64)
    mag = np.where(
        e == 0,
        np.ldexp(sub_sig, f.sub_exp),
        np.ldexp(normal_sig, (e - f.bias - f.mbits).astype(np.int64)),
    )
    mag = np.where(e == f.exp_mask, np.where(m == 0, np.inf, np.nan), mag)
    return np.where(sign == 1, -mag, mag)


def encode_rne(x, fmt="bf16") -> np.ndarray:
    """float64 values -> bit patterns of format `fmt`, one rounding to nearest
    even.

    The rounding is done on an integer significand: |x| is scaled by an exact
    power of two so that one quantum of the format becomes 1, rounded with
    np.rint (ties to even), and the bit pattern is assembled from the result.
    Magnitudes at or above the overflow threshold give infinity; NaN encodes as
    the format's quiet NaN with the input's sign dropped.
    """
    f = _fmt(fmt)
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    a_safe = np.where(nan | np.isinf(a), 0.0, a)

    # Unbiased exponent E with |x| = 1.f * 2^E (frexp gives mantissa in [0.5, 1)).
    _, fe = np.frexp(a_safe)
    E = fe.astype(np.int64) - 1
    # Quantum at this magnitude: 2^(E - mbits) for normals, 2^sub_exp below
    # the smallest normal.
    qexp = np.where(a_safe < f.min_normal, f.sub_exp, E - f.mbits)
    n = np.ldexp(a_safe, -qexp)                           # exact scaling
    r = np.rint(n)                                         # ties to even
    y = np.ldexp(r, qexp)                                  # rounded magnitude, exact

    # Assemble the bits of y (exactly a value of the format, or >= 2^(emax+1)).
    _, ye = np.frexp(y)
    yE = ye.astype(np.int64) - 1
    is_sub = y < f.min_normal
    sub_bits = np.where(is_sub, np.ldexp(y, -f.sub_exp), 0.0).astype(np.int64)
    mant = np.where(is_sub, 0, np.ldexp(y, -(yE - f.mbits)).astype(np.int64) - (1 << f.mbits))
    norm_bits = ((yE + f.bias) << f.mbits) | np.clip(mant, 0, (1 << f.mbits) - 1)
    bits = np.where(is_sub, sub_bits, norm_bits)
    bits = np.where((y >= 2.0 ** (f.emax + 1)) | (a >= f.overflow), f.inf_bits, bits)
    bits = np.where(neg, bits | 0x8000, bits)
    bits = np.where(nan, f.qnan_bits, bits)
    return bits.astype(np.uint16)


def bf16_decode(bits) -> np.ndarray:
    """BF16 (1 sign, 8 exponent bits with bias 127, 7 mantissa bits;
    subnormals mantissa * 2^-133) -> exact float64."""
    return decode(bits, BF16)


def bf16_encode_rne(x) -> np.ndarray:
    """float64 -> BF16 bits, one rounding to nearest even (NaN -> 0x7FC0)."""
    return encode_rne(x, BF16)


def fp16_decode(bits) -> np.ndarray:
    """FP16 (IEEE binary16: 1 sign, 5 exponent bits with bias 15, 10 mantissa
    bits; subnormals mantissa * 2^-24) -> exact float64."""
    return decode(bits, FP16)


def fp16_encode_rne(x) -> np.ndarray:
    """float64 -> FP16 bits, one rounding to nearest even (|x| >= 65520 gives
    infinity; NaN -> 0x7E00)."""
    return encode_rne(x, FP16)


def fold(prefix, add, add2=None, fmt="bf16"):
    """Step (a2): the MoE-tail fold into the prefix sum.

    Returns (new_prefix_bits, s_bits) with s = bf16(add + add2) (or add when
    add2 is None) and new_prefix = bf16(prefix + s), each a correctly rounded
    BF16 addition.  TensorRT-LLM PR #20546, section "Op".  With fmt="fp16"
    every tensor and both roundings are FP16 instead (the exact sum of two
    FP16 values rounded to float64 and then to FP16 is the correctly rounded
    FP16 sum, 53 >= 2*11+2; the float32 route qualifies too, 24 >= 24).
    """
    if add2 is None:
        s = np.asarray(add, dtype=np.uint16)
    else:
        s = encode_rne(decode(add, fmt) + decode(add2, fmt), fmt)
    np_bits = encode_rne(decode(prefix, fmt) + decode(s, fmt), fmt)
    return np_bits, s


def mixture(V, w, gamma, eps):
    """Steps (a3)-(a6) in float64 for a batch of tokens.

    V:     (T, S, H) float64, the S = N+1 sources of each token, bank snapshots
           first and the updated prefix last.
    w:     (H,) float64 pseudo-query.   gamma: (H,) float64 RMSNorm weight.
    eps:   the epsilon of both RMSNorms (inside the square root).

    Returns a dict with
      out    (T, H)  h / sqrt(mean(h^2) + eps) * gamma, unrounded
      bound  (T, H)  r_h * |gamma_j| * sum_i alpha_i |v_ij|: the scale of the
                     terms that meet in out_j, used by the tolerance check
      alpha  (T, S)  the softmax weights;  logits (T, S);  h (T, H)
    """
    V = np.asarray(V, dtype=np.float64)
    T, S, H = V.shape
    w = np.asarray(w, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)

    # (a3) per-source sum of squares and dot product with the pseudo-query.
    ss = np.sum(V * V, axis=2)                        # (T, S)
    d = np.sum(V * w[None, None, :], axis=2)          # (T, S)
    # (a4) l_i = w . (v_i / rms(v_i)) = d_i / sqrt(ss_i / H + eps); softmax.
    logits = d / np.sqrt(ss / H + eps)
    z = logits - np.max(logits, axis=1, keepdims=True)
    e = np.exp(z)
    alpha = e / np.sum(e, axis=1, keepdims=True)
    # (a5) mixture h = sum_i alpha_i v_i.
    h = np.sum(alpha[:, :, None] * V, axis=1)         # (T, H)
    # (a6) RMSNorm(h) * gamma.
    r_h = 1.0 / np.sqrt(np.sum(h * h, axis=1, keepdims=True) / H + eps)
    out = h * r_h * gamma[None, :]
    bound = r_h * np.abs(gamma)[None, :] * np.sum(alpha[:, :, None] * np.abs(V), axis=1)
    return {"out": out, "bound": bound, "alpha": alpha, "logits": logits, "h": h}


def attnres_add_rmsnorm(prefix, add, add2, bank, w, gamma, eps, tokens=None, chunk=64,
                        with_h=False, fmt="bf16"):
    """The whole op on BF16 bit patterns (FP16 with fmt="fp16").

    prefix, add, add2: (M, H) uint16 (add2 may be None);  bank: (N, M, H)
    uint16;  w, gamma: (H,) uint16;  eps: the float32 epsilon the GPU sees
    (it is rounded to float32 here so both sides use the same value).
    tokens: optional index array; when given, only those tokens are computed
    (the fold included), which lets a full-size call be checked on a sample.

    Returns (new_prefix_bits (T, H) uint16, out (T, H) float64, bound (T, H)),
    and with with_h=True also (h (T, H) float64, h_bound (T, H)): the pre-norm
    mixture and the scale sum_i alpha_i |v_ij| of the terms that meet in it.
    """
    prefix = np.asarray(prefix, dtype=np.uint16)
    add = None if add is None else np.asarray(add, dtype=np.uint16)
    bank = np.asarray(bank, dtype=np.uint16)
    if bank.ndim != 3:
        raise ValueError("bank must be (N, M, H)")
    N, M, H = bank.shape
    if tokens is None:
        tokens = np.arange(M)
    tokens = np.asarray(tokens, dtype=np.int64)
    eps64 = float(np.float32(eps))
    w64 = decode(w, fmt)
    g64 = decode(gamma, fmt)

    np_all = np.empty((len(tokens), H), dtype=np.uint16)
    out_all = np.empty((len(tokens), H), dtype=np.float64)
    bound_all = np.empty((len(tokens), H), dtype=np.float64)
    h_all = np.empty((len(tokens), H), dtype=np.float64) if with_h else None
    hb_all = np.empty((len(tokens), H), dtype=np.float64) if with_h else None
    for c0 in range(0, len(tokens), chunk):
        t = tokens[c0:c0 + chunk]
        if add is None:
            np_bits = prefix[t]          # no fold: the prefix itself is the source
        else:
            np_bits, _ = fold(prefix[t], add[t],
                              None if add2 is None else np.asarray(add2, dtype=np.uint16)[t], fmt)
        V = np.empty((len(t), N + 1, H), dtype=np.float64)
        V[:, :N, :] = decode(bank[:, t, :], fmt).transpose(1, 0, 2)
        V[:, N, :] = decode(np_bits, fmt)
        r = mixture(V, w64, g64, eps64)
        np_all[c0:c0 + len(t)] = np_bits
        out_all[c0:c0 + len(t)] = r["out"]
        bound_all[c0:c0 + len(t)] = r["bound"]
        if with_h:
            h_all[c0:c0 + len(t)] = r["h"]
            hb_all[c0:c0 + len(t)] = np.sum(r["alpha"][:, :, None] * np.abs(V), axis=1)
    if with_h:
        return np_all, out_all, bound_all, h_all, hb_all
    return np_all, out_all, bound_all


def attnres_rmsnorm(prefix, bank, w, gamma, eps, tokens=None, chunk=64, with_h=False,
                    fmt="bf16"):
    """The attention-residual + RMSNorm alone (no fold): the sources are
    bank[0..N-1, m] and prefix[m] itself.  TensorRT-LLM PR #20546, section
    "Performance", measures the fused epilogue against this op.

    Returns (out (T, H) float64, bound (T, H)) [, h, h_bound with with_h]."""
    r = attnres_add_rmsnorm(prefix, None, None, bank, w, gamma, eps, tokens=tokens, chunk=chunk,
                            with_h=with_h, fmt=fmt)
    return r[1:]


def algorithmic_bytes(M, N, H, has_add2):
    """Bytes one call must move: every input read once, both outputs written
    once, plus w and gamma: (N+3 or N+2) reads + 2 writes of M*H BF16, + 4H."""
    R = M * H * 2
    return (N + (3 if has_add2 else 2)) * R + 2 * R + 4 * H
