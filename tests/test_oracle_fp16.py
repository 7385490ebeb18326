"""Pins of the oracle's FP16 path (no GPU): the integer FP16 codec against
numpy's half-precision conversions and the definition of round-to-nearest-
even, the fold against hand-derived cases and against numpy's FP16 additions,
the mixture on FP16 tensors against closed forms and a 50-digit evaluation,
and the FP16 tolerance."""
import math
import os

import mpmath
import numpy as np
import pytest
import torch

from oracle import (FP16, attnres_add_rmsnorm, check_out, fold, fp16_decode, fp16_encode_rne,
                    ulp)


def _np_half_to_f64(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _np_f64_to_half_bits(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


# ---- codec

def test_decode_all_patterns_match_numpy():
    allb = np.arange(65536, dtype=np.uint16)
    ours = fp16_decode(allb)
    ref = _np_half_to_f64(allb)
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0x0000])


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0xC000, -2.0), (0x1000, 2.0 ** -11), (0x0001, 2.0 ** -24),
    (0x03FF, 1023 * 2.0 ** -24), (0x0400, 2.0 ** -14), (0x7BFF, 65504.0), (0x3E00, 1.5),
    (0x4248, 3.140625), (0x4BFF, 16 - 2.0 ** -7),
])
def test_decode_known_values(bits, value):
    assert fp16_decode(np.array([bits], np.uint16))[0] == value


def test_encode_roundtrip_all_finite():
    allb = np.arange(65536, dtype=np.uint16)
    v = fp16_decode(allb)
    fin = np.isfinite(v)
    assert (fp16_encode_rne(v[fin]) == allb[fin]).all()


def test_encode_matches_numpy_rounding():
    """numpy converts float64 to float16 with one rounding to nearest even;
    random magnitudes over the whole range, every midpoint between
    neighbouring FP16 values and the values either side of each midpoint."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal(400_000) * np.exp2(rng.integers(-30, 18, 400_000))
    allb = np.arange(0, 0x7C00, dtype=np.uint16)
    v = fp16_decode(allb)
    mids = (v[:-1] + v[1:]) / 2
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
                        [65504.0, 65519.999, 65520.0, 65536.0, 1e6, 2.0 ** -25, 2.0 ** -26]])
    assert (fp16_encode_rne(x) == _np_f64_to_half_bits(x)).all()


def test_encode_is_nearest_and_ties_even():
    rng = np.random.default_rng(22)
    x = rng.standard_normal(200_000) * np.exp2(rng.integers(-28, 15, 200_000))
    b = fp16_encode_rne(x).astype(np.int64)
    mag = b & 0x7FFF
    y = fp16_decode(b.astype(np.uint16))
    lo = fp16_decode(((mag - 1).clip(0) | (b & 0x8000)).astype(np.uint16))
    hi = fp16_decode(((mag + 1).clip(max=0x7BFF) | (b & 0x8000)).astype(np.uint16))
    err = np.abs(y - x)
    assert (err <= np.abs(lo - x)).all() and (err <= np.abs(hi - x)).all()
    tie = ((err == np.abs(lo - x)) & (mag > 0) | (err == np.abs(hi - x)) & (mag < 0x7BFF)) & (err > 0)
    assert (mag[tie] % 2 == 0).all()


def test_encode_specials():
    v = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 65504.0, 65519.99, 65520.0, -65520.0,
                  2.0 ** -25, 2.0 ** -25 * 1.0001, 3 * 2.0 ** -25])
    assert list(fp16_encode_rne(v)) == [0x0000, 0x8000, 0x7C00, 0xFC00, 0x7E00, 0x7BFF, 0x7BFF,
                                        0x7C00, 0xFC00, 0x0000, 0x0001, 0x0002]


def test_format_constants():
    assert FP16.bias == 15 and FP16.max_finite == 65504.0 and FP16.overflow == 65520.0
    assert FP16.min_normal == 2.0 ** -14 and FP16.sub_exp == -24
    assert FP16.inf_bits == 0x7C00 and FP16.qnan_bits == 0x7E00


# ---- fold

def _load_cases(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "fold_cases_fp16.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(tuple(int(x, 16) for x in line.split()[:4]))
    return rows


def test_golden_fold_cases(golden_dir):
    cases = _load_cases(golden_dir)
    assert len(cases) >= 16
    p, a, a2, e = (np.array(c, np.uint16) for c in zip(*cases))
    got, _ = fold(p, a, a2, "fp16")
    assert (got == e).all(), [hex(x) for x in got]
    s = fp16_encode_rne(fp16_decode(a) + fp16_decode(a2))
    assert (fold(p, s, None, "fp16")[0] == e).all()


def test_golden_cases_match_numpy_half(golden_dir):
    p, a, a2, e = (np.array(c, np.uint16) for c in zip(*_load_cases(golden_dir)))
    h = lambda b: b.view(np.float16)  # noqa: E731
    with np.errstate(over="ignore"):
        ref = (h(p) + (h(a) + h(a2))).view(np.uint16)
    assert (ref == e).all()


def _random_patterns(rng, n):
    kind = rng.integers(0, 4, n)
    normal = fp16_encode_rne(rng.standard_normal(n) * np.exp2(rng.integers(-26, 15, n)))
    sub = (rng.integers(0, 1024, n) | (rng.integers(0, 2, n) << 15)).astype(np.uint16)
    zero = (rng.integers(0, 2, n) << 15).astype(np.uint16)
    small = fp16_encode_rne(rng.standard_normal(n))
    return np.select([kind == 0, kind == 1, kind == 2], [normal, sub, zero], small).astype(np.uint16)


def test_fold_matches_numpy_half_additions():
    """prefix + (add + add2) in numpy float16: each addition is a correctly
    rounded FP16 sum."""
    rng = np.random.default_rng(23)
    n = 400_000
    p, a, a2 = (_random_patterns(rng, n) for _ in range(3))
    idx = rng.choice(n, n // 4, replace=False)
    a2[idx] = ((a[idx].astype(np.int64) ^ 0x8000) + rng.integers(-2, 3, len(idx))).clip(0, 0xFFFF)
    ok = np.isfinite(fp16_decode(a2)) & np.isfinite(fp16_decode(a))
    p, a, a2 = p[ok], a[ok], a2[ok]
    got, _ = fold(p, a, a2, "fp16")
    h = lambda b: b.view(np.float16)  # noqa: E731
    with np.errstate(over="ignore"):
        ref = (h(p) + (h(a) + h(a2))).view(np.uint16)
    assert (got == ref).all()


def test_inner_add_brute_force_against_float32():
    """Every finite FP16 a against 512 b patterns (every exponent, both signs,
    subnormals): the oracle's float64 route equals the float32 route (add in
    float32, round to FP16), the kernel's arithmetic."""
    a = np.arange(65536, dtype=np.uint16)
    a = a[np.isfinite(fp16_decode(a))]
    rng = np.random.default_rng(24)
    b = np.concatenate([np.arange(0, 0x7C00, 128, dtype=np.uint16),
                        np.arange(0, 1024, 16, dtype=np.uint16),
                        rng.integers(0, 0x7C00, 136).astype(np.uint16)])
    b = np.concatenate([b, b | 0x8000])[:512]
    af = fp16_decode(a).astype(np.float32)
    for bb in b:
        bf = np.float32(fp16_decode(np.array([bb], np.uint16))[0])
        with np.errstate(over="ignore"):
            r = (af + bf).astype(np.float16).view(np.uint16)
        got = fp16_encode_rne(fp16_decode(a) + fp16_decode(np.full_like(a, bb)))
        assert (got == r).all(), hex(int(bb))


def test_two_addends_equal_one_presummed_addend():
    rng = np.random.default_rng(25)
    n = 200_000
    p, a, a2 = (_random_patterns(rng, n) for _ in range(3))
    s = fp16_encode_rne(fp16_decode(a) + fp16_decode(a2))
    assert (fold(p, a, a2, "fp16")[0] == fold(p, s, None, "fp16")[0]).all()


# ---- mixture on FP16 tensors

def _h(x):
    return fp16_encode_rne(np.asarray(x, np.float64))


def test_all_sources_equal_reduce_to_rms_norm():
    rng = np.random.default_rng(26)
    H, N, M = 64, 5, 3
    v = _h(rng.standard_normal((M, H)))
    gamma = _h(1 + 0.1 * rng.standard_normal(H))
    w = _h(0.3 * rng.standard_normal(H))
    bank = np.broadcast_to(v, (N, M, H))
    zero = np.zeros((M, H), np.uint16)
    new_p, out, _ = attnres_add_rmsnorm(v, zero, None, bank, w, gamma, 1e-6, fmt="fp16")
    assert (new_p == v).all()
    ref = torch.nn.functional.rms_norm(torch.from_numpy(_np_half_to_f64(v)), (H,),
                                       torch.from_numpy(_np_half_to_f64(gamma)),
                                       float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)


def test_brute_force_high_precision():
    mpmath.mp.dps = 50
    rng = np.random.default_rng(27)
    H, N = 16, 3
    bank = _h(rng.standard_normal((N, 1, H)))
    prefix, add, add2 = (_h(rng.standard_normal((1, H))) for _ in range(3))
    w = _h(rng.standard_normal(H) / math.sqrt(H))
    gamma = _h(1 + 0.1 * rng.standard_normal(H))
    new_p, out, _ = attnres_add_rmsnorm(prefix, add, add2, bank, w, gamma, 1e-6, fmt="fp16")
    # the updated prefix from numpy's FP16 additions, the mixture from the definition
    h = lambda b: b.view(np.float16)  # noqa: E731
    assert (new_p == (h(prefix) + (h(add) + h(add2))).view(np.uint16)).all()
    src = np.concatenate([_np_half_to_f64(bank[:, 0]), _np_half_to_f64(new_p)], axis=0)
    eps = mpmath.mpf(float(np.float32(1e-6)))
    v = [[mpmath.mpf(float(x)) for x in row] for row in src]
    wm = [mpmath.mpf(float(x)) for x in _np_half_to_f64(w)]
    gm = [mpmath.mpf(float(x)) for x in _np_half_to_f64(gamma)]
    logits = [mpmath.fsum(a * b for a, b in zip(wm, r)) / mpmath.sqrt(mpmath.fsum(x * x for x in r) / H + eps)
              for r in v]
    mx = max(logits)
    ex = [mpmath.exp(lv - mx) for lv in logits]
    z = mpmath.fsum(ex)
    hh = [mpmath.fsum(ex[i] / z * v[i][j] for i in range(N + 1)) for j in range(H)]
    rh = 1 / mpmath.sqrt(mpmath.fsum(x * x for x in hh) / H + eps)
    ref = np.array([float(hh[j] * rh * gm[j]) for j in range(H)])
    np.testing.assert_allclose(out[0], ref, rtol=1e-13, atol=1e-15)


# ---- tolerance

def test_fp16_ulp():
    assert ulp(np.array([1.0]), "fp16")[0] == 2.0 ** -10
    assert ulp(np.array([1.5]), "fp16")[0] == 2.0 ** -10
    assert ulp(np.array([2.0 ** -20]), "fp16")[0] == 2.0 ** -24
    assert ulp(np.array([65504.0]), "fp16")[0] == 32.0


def test_fp16_tolerance_is_two_fp16_ulp():
    ref = np.array([1.25, -3.0, 0.75])
    bound = np.abs(ref)
    exact = fp16_encode_rne(ref)
    assert check_out(exact, ref, bound, "fp16")["ok"]
    two = fp16_encode_rne(ref + 2 * 2.0 ** -10 * np.array([1, -2, 0.5]) * 0.999)
    assert check_out(two, ref, bound, "fp16")["ok"]
    # 3 FP16 ulp off: well inside 2 BF16 ulp, still a failure for FP16
    three = (exact.astype(np.int64) + 3).astype(np.uint16)
    r = check_out(three, ref, bound, "fp16")
    assert not r["ok"] and r["n_fail"] == 3
