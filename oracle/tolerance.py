"""Parity criteria between a BF16 (or FP16) GPU result and the float64 oracle.

TEST INFRASTRUCTURE ONLY (see oracle/attnres_oracle.py).

new_prefix: bit-exact.  The fold is a pair of correctly rounded BF16 additions
(TensorRT-LLM PR #20546, section "Op"), so there is exactly one right answer.

out: the GPU evaluates the mixture and the norm in float32 and rounds once to
BF16; the oracle keeps float64 and does not round.  An element passes when

    |delta| <= max(2 * ulp_bf16(ref), 2^-16)                                (1)
    and (|ref| > 4 or |delta| <= 1.5e-2)                                    (2)

with ulp_bf16(x) = 2^(floor(log2|x|) - 7) for normal magnitudes (2^-133 below
2^-126).  (1) is "within 2 BF16 ulp per element" with an absolute floor: the
float32 accumulation of O(1) terms carries an absolute error near
(N+1) * 2^-24 * bound, so an output that cancels to |ref| < ~1e-4 cannot hold a
2-ulp relative bound.  2^-16 is ~100x that float32 error at bound ~ 1.  (2) is
the absolute cap for |out| <= 4.  Every element that passes only through the
floor must still satisfy |delta| <= 64 * 2^-24 * bound_j + 2^-133 (a float32
error model of the mixture), and the number of such elements is reported.

FP16 outputs (fmt="fp16") take the same criterion with the FP16 unit in the
last place, ulp_fp16(x) = 2^(floor(log2|x|) - 10) (2^-24 below 2^-14), and the
smallest FP16 subnormal 2^-24 in place of 2^-133: 2 FP16 ulp is 8x tighter
than 2 BF16 ulp, the floor and the float32 error model are those of the same
float32 arithmetic.
"""
from __future__ import annotations

import numpy as np

from .attnres_oracle import BF16, _fmt, decode

ULP_FACTOR = 2.0
ABS_FLOOR = 2.0 ** -16
CAP_ABS = 1.5e-2
CAP_RANGE = 4.0
F32_BOUND_FACTOR = 64 * 2.0 ** -24


def ulp(x, fmt="bf16") -> np.ndarray:
    """Unit in the last place of the format at the magnitude of x."""
    f = _fmt(fmt)
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(a == 0, 1.0, a))
    u = np.ldexp(1.0, (e.astype(np.int64) - 1) - f.mbits)
    return np.where(a < f.min_normal, 2.0 ** f.sub_exp, u)


def ulp_bf16(x) -> np.ndarray:
    return ulp(x, BF16)


def check_out(gpu_bits, ref, bound, fmt="bf16"):
    """Returns a dict: ok, n, n_fail, n_floor (elements passing only through
    the absolute floor), max_abs, max_ulp, first failing index if any."""
    f = _fmt(fmt)
    got = decode(gpu_bits, f)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    finite = np.isfinite(ref)
    delta = np.abs(got - ref)
    delta = np.where(finite, delta, 0.0)
    u = ulp(ref, f)
    strict = delta <= ULP_FACTOR * u
    tol = np.maximum(ULP_FACTOR * u, ABS_FLOOR)
    ok1 = delta <= tol
    ok2 = (np.abs(ref) > CAP_RANGE) | (delta <= CAP_ABS)
    floor_only = ok1 & ~strict
    ok3 = ~floor_only | (delta <= F32_BOUND_FACTOR * bound + 2.0 ** f.sub_exp)
    okv = (ok1 & ok2 & ok3) | ~finite
    fails = np.flatnonzero(~okv.ravel())
    return {
        "ok": bool(fails.size == 0),
        "n": int(okv.size),
        "n_fail": int(fails.size),
        "n_floor": int(np.count_nonzero(floor_only)),
        "max_abs": float(delta.max()) if delta.size else 0.0,
        "max_ulp": float((delta / u).max()) if delta.size else 0.0,
        "first_fail": None if fails.size == 0 else np.unravel_index(fails[0], okv.shape),
    }
