"""Pins of the oracle's fold (no GPU): the hand-derived golden cases, the
two-addends-equal-one-pre-summed-addend invariant, PyTorch's own BF16
additions, and a brute-force sweep of the inner addition against float32."""
import os

import numpy as np
import pytest
import torch

from oracle import bf16_decode, bf16_encode_rne, fold


def _load_cases(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "fold_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            p, a, a2, e = (int(x, 16) for x in line.split()[:4])
            rows.append((p, a, a2, e))
    return rows


def _u16(*xs):
    return np.array(xs, dtype=np.uint16)


def _t(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16).copy()).view(torch.bfloat16)


def _tbits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_golden_fold_cases(golden_dir):
    cases = _load_cases(golden_dir)
    assert len(cases) >= 13
    p, a, a2, e = (np.array(c, np.uint16) for c in zip(*cases))
    got, _ = fold(p, a, a2)
    assert (got == e).all(), [hex(x) for x in got]
    # the same cases with add2 absent and add holding bf16(add + add2)
    s = bf16_encode_rne(bf16_decode(a) + bf16_decode(a2))
    got1, _ = fold(p, s, None)
    assert (got1 == e).all()


def test_golden_cases_match_torch_bf16(golden_dir):
    torch.set_flush_denormal(False)
    p, a, a2, e = (np.array(c, np.uint16) for c in zip(*_load_cases(golden_dir)))
    assert (_tbits(_t(p) + (_t(a) + _t(a2))) == e).all()


def _random_patterns(rng, n):
    """Mixed BF16 patterns: normals of all scales, subnormals, zeros and
    near-cancelling pairs."""
    kind = rng.integers(0, 4, n)
    normal = bf16_encode_rne(rng.standard_normal(n) * np.exp2(rng.integers(-135, 20, n)))
    sub = (rng.integers(0, 128, n) | (rng.integers(0, 2, n) << 15)).astype(np.uint16)
    zero = (rng.integers(0, 2, n) << 15).astype(np.uint16)
    small = bf16_encode_rne(rng.standard_normal(n))
    return np.select([kind == 0, kind == 1, kind == 2], [normal, sub, zero], small).astype(np.uint16)


def test_fold_matches_torch_two_additions():
    """prefix + (routed + shared) in PyTorch BF16 (section "Test Coverage":
    the same prefix sum as prefix + (routed + shared) in PyTorch)."""
    torch.set_flush_denormal(False)
    rng = np.random.default_rng(3)
    n = 400_000
    p = _random_patterns(rng, n)
    a = _random_patterns(rng, n)
    a2 = _random_patterns(rng, n)
    # near-cancelling pairs: a2 = -a moved by up to 2 ulp
    idx = rng.choice(n, n // 4, replace=False)
    a2[idx] = ((a[idx].astype(np.int64) ^ 0x8000) + rng.integers(-2, 3, len(idx))).clip(0, 0xFFFF)
    ok = np.isfinite(bf16_decode(a2))
    p, a, a2 = p[ok], a[ok], a2[ok]
    got, _ = fold(p, a, a2)
    ref = _tbits(_t(p) + (_t(a) + _t(a2)))
    assert (got == ref).all()


def test_two_addends_equal_one_presummed_addend():
    rng = np.random.default_rng(4)
    n = 200_000
    p, a, a2 = (_random_patterns(rng, n) for _ in range(3))
    s = bf16_encode_rne(bf16_decode(a) + bf16_decode(a2))
    assert (fold(p, a, a2)[0] == fold(p, s, None)[0]).all()


def test_fold_without_add2_is_one_addition():
    rng = np.random.default_rng(5)
    p, a = _random_patterns(rng, 100_000), _random_patterns(rng, 100_000)
    torch.set_flush_denormal(False)
    assert (fold(p, a, None)[0] == _tbits(_t(p) + _t(a))).all()


def _f32_ok():
    tiny = np.array([1e-45], dtype=np.float32)
    return (tiny + tiny)[0] != 0


def test_inner_add_brute_force_against_float32():
    """Every BF16 pattern a against 1024 patterns b that cover every exponent,
    both signs and the subnormals: the oracle's float64 route must equal the
    float32 route the PR describes (add in float32, round to BF16)."""
    if not _f32_ok():
        pytest.skip("host float32 flushes subnormals")
    a = np.arange(65536, dtype=np.uint16)
    a = a[np.isfinite(bf16_decode(a))]
    rng = np.random.default_rng(6)
    b = np.concatenate([
        np.arange(0, 0x8000, 64, dtype=np.uint16),          # one per exponent step
        np.arange(0, 128, 1, dtype=np.uint16)[::2],          # subnormals
        rng.integers(0, 0x7F80, 448).astype(np.uint16),
    ])
    b = np.concatenate([b, b | 0x8000])[:1024]
    af32 = (a.astype(np.uint32) << 16).view(np.float32)
    for bb in b:
        bf32 = np.array([np.uint32(bb) << 16], np.uint32).view(np.float32)[0]
        s32 = af32 + bf32
        # round float32 -> BF16 to nearest even with integer arithmetic
        u = s32.view(np.uint32).astype(np.uint64)
        r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
        r = np.where(np.isnan(s32), 0x7FC0, r)
        got = bf16_encode_rne(bf16_decode(a) + bf16_decode(np.full_like(a, bb)))
        assert (got == r).all(), hex(int(bb))
