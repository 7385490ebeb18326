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
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_decode",
    "bf16_encode_rne",
    "fold",
    "mixture",
    "attnres_add_rmsnorm",
    "attnres_rmsnorm",
    "algorithmic_bytes",
]

_BF16_MAX_FINITE = (2.0 - 2.0 ** -7) * 2.0 ** 127
# Values at or above this magnitude round (to nearest even) to infinity: the
# midpoint between the largest finite BF16 and 2^128, and the largest finite
# value's last mantissa bit is odd, so the tie goes up.
_BF16_OVERFLOW = (2.0 - 2.0 ** -8) * 2.0 ** 127
_BF16_MIN_NORMAL = 2.0 ** -126
_BF16_SUBNORMAL_QUANTUM = 2.0 ** -133
_BF16_QNAN = np.uint16(0x7FC0)


def bf16_decode(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact float64 values.

    Layout: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits.
    Exponent 0 encodes zero and subnormals (mantissa * 2^-133); exponent 255
    encodes infinities (mantissa 0) and NaN (mantissa != 0).
    """
    u = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = (u >> 15) & 1
    e = (u >> 7) & 0xFF
    m = u & 0x7F
    normal_sig = (m + 128).astype(np.float64)          # 1.m as an integer * 2^7
    sub_sig = m.astype(np.float64)
    mag = np.where(
        e == 0,
        np.ldexp(sub_sig, -133),
        np.ldexp(normal_sig, (e - 127 - 7).astype(np.int64)),
    )
    mag = np.where(e == 255, np.where(m == 0, np.inf, np.nan), mag)
    return np.where(sign == 1, -mag, mag)


def bf16_encode_rne(x) -> np.ndarray:
    """float64 values -> BF16 bit patterns, one rounding to nearest even.

    The rounding is done on an integer significand: |x| is scaled by an exact
    power of two so that one BF16 quantum becomes 1, rounded with np.rint
    (ties to even), and the bit pattern is assembled from the result.
    NaN encodes as 0x7FC0 with the input's sign dropped.
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    a_safe = np.where(nan | np.isinf(a), 0.0, a)

    # Unbiased exponent E with |x| = 1.f * 2^E (frexp gives mantissa in [0.5, 1)).
    _, fe = np.frexp(a_safe)
    E = fe.astype(np.int64) - 1
    # BF16 quantum at this magnitude: 2^(E-7) for normals, 2^-133 below 2^-126.
    qexp = np.where(a_safe < _BF16_MIN_NORMAL, -133, E - 7)
    n = np.ldexp(a_safe, -qexp)                           # exact scaling
    r = np.rint(n)                                         # ties to even
    y = np.ldexp(r, qexp)                                  # rounded magnitude, exact

    # Assemble the bits of y (which is exactly a BF16 value or >= 2^128).
    _, ye = np.frexp(y)
    yE = ye.astype(np.int64) - 1
    is_sub = y < _BF16_MIN_NORMAL
    sub_bits = np.where(is_sub, np.ldexp(y, 133), 0.0).astype(np.int64)
    mant = np.where(is_sub, 0, np.ldexp(y, -(yE - 7)).astype(np.int64) - 128)
    norm_bits = ((yE + 127) << 7) | np.clip(mant, 0, 127)
    bits = np.where(is_sub, sub_bits, norm_bits)
    bits = np.where((y >= 2.0 ** 128) | (a >= _BF16_OVERFLOW), 0x7F80, bits)
    bits = np.where(neg, bits | 0x8000, bits)
    bits = np.where(nan, int(_BF16_QNAN), bits)
    return bits.astype(np.uint16)


def fold(prefix, add, add2=None):
    """Step (a2): the MoE-tail fold into the BF16 prefix sum.

    Returns (new_prefix_bits, s_bits) with s = bf16(add + add2) (or add when
    add2 is None) and new_prefix = bf16(prefix + s), each a correctly rounded
    BF16 addition.  TensorRT-LLM PR #20546, section "Op".
    """
    if add2 is None:
        s = np.asarray(add, dtype=np.uint16)
    else:
        s = bf16_encode_rne(bf16_decode(add) + bf16_decode(add2))
    np_bits = bf16_encode_rne(bf16_decode(prefix) + bf16_decode(s))
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
                        with_h=False):
    """The whole op on BF16 bit patterns.

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
    w64 = bf16_decode(w)
    g64 = bf16_decode(gamma)

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
            np_bits, _ = fold(prefix[t], add[t], None if add2 is None else np.asarray(add2, dtype=np.uint16)[t])
        V = np.empty((len(t), N + 1, H), dtype=np.float64)
        V[:, :N, :] = bf16_decode(bank[:, t, :]).transpose(1, 0, 2)
        V[:, N, :] = bf16_decode(np_bits)
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


def attnres_rmsnorm(prefix, bank, w, gamma, eps, tokens=None, chunk=64, with_h=False):
    """The attention-residual + RMSNorm alone (no fold): the sources are
    bank[0..N-1, m] and prefix[m] itself.  TensorRT-LLM PR #20546, section
    "Performance", measures the fused epilogue against this op.

    Returns (out (T, H) float64, bound (T, H)) [, h, h_bound with with_h]."""
    r = attnres_add_rmsnorm(prefix, None, None, bank, w, gamma, eps, tokens=tokens, chunk=chunk,
                            with_h=with_h)
    return r[1:]


def algorithmic_bytes(M, N, H, has_add2):
    """Bytes one call must move: every input read once, both outputs written
    once, plus w and gamma: (N+3 or N+2) reads + 2 writes of M*H BF16, + 4H."""
    R = M * H * 2
    return (N + (3 if has_add2 else 2)) * R + 2 * R + 4 * H
