"""Pins of the oracle's mixture and output norm (no GPU): hand-derived closed
forms, cases that reduce to torch's rms_norm, invariants of the definition,
and a 50-digit evaluation on tiny inputs."""
import math

import mpmath
import numpy as np
import pytest
import torch

from oracle import attnres_add_rmsnorm, bf16_decode, bf16_encode_rne, mixture


def _b(vals):
    return bf16_encode_rne(np.asarray(vals, dtype=np.float64))


def _op(prefix, add, add2, bank, w, gamma, eps):
    return attnres_add_rmsnorm(_b(prefix), _b(add), None if add2 is None else _b(add2),
                               _b(bank), _b(w), _b(gamma), eps)


@pytest.mark.parametrize("b", [0.5, -0.75, 2.0, 0.0])
def test_closed_form_two_sources(b):
    """N=1, H=2.  Bank snapshot v0 = (1, 1); the fold gives the updated prefix
    v1 = (0.5, -0.5) + (0.5, -0.5) + 0 = (1, -1); w = (0, b).
    Both sources have mean square 1, so r = 1/sqrt(1 + eps) and the logits are
    (b r, -b r): alpha0 - alpha1 = tanh(b r), h = (1, tanh(b r)), and
    out = (1, t) gamma / sqrt((1 + t^2)/2 + eps)."""
    eps = 1e-6
    e32 = float(np.float32(eps))
    gamma = [1.5, 0.75]
    _, out, _ = _op([[0.5, -0.5]], [[0.5, -0.5]], [[0.0, 0.0]], [[[1.0, 1.0]]], [0.0, b], gamma, eps)
    t = math.tanh(b / math.sqrt(1.0 + e32))
    s = 1.0 / math.sqrt((1.0 + t * t) / 2.0 + e32)
    expect = np.array([1.0 * s * 1.5, t * s * 0.75])
    np.testing.assert_allclose(out[0], expect, rtol=1e-14, atol=0)


@pytest.mark.parametrize("b", [0.5, 3.0])
def test_closed_form_eps_matters(b):
    """Same geometry scaled by 2^-10 with eps = 2^-20: mean squares equal eps,
    so r = 2^10/sqrt(2), logits (b/sqrt2, -b/sqrt2), h = 2^-10 (1, t) with
    t = tanh(b/sqrt2), and out = (1, t) gamma / sqrt((1 + t^2)/2 + 1).
    A missing eps, eps outside the root, or unnormalised weights all move it."""
    eps = 2.0 ** -20
    s10 = 2.0 ** -10
    gamma = [1.0, -2.0]
    _, out, _ = _op([[s10, -s10]], [[0.0, 0.0]], None, [[[s10, s10]]], [0.0, b], gamma, eps)
    t = math.tanh(b / math.sqrt(2.0))
    s = 1.0 / math.sqrt((1.0 + t * t) / 2.0 + 1.0)
    np.testing.assert_allclose(out[0], [s, -2.0 * t * s], rtol=1e-14)


def _bf(x):
    """Round to the nearest BF16 value (kept as float64)."""
    return bf16_decode(bf16_encode_rne(x))


def _rand_bf16(rng, shape, std=1.0):
    return _bf(rng.standard_normal(shape) * std)


def test_all_sources_equal_reduce_to_rms_norm():
    """With every source equal to v, alpha is uniform, h = v and out must be
    torch.nn.functional.rms_norm(v, (H,), gamma, eps)."""
    rng = np.random.default_rng(10)
    H, N, M = 64, 5, 3
    v = _rand_bf16(rng, (M, H))
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    w = _rand_bf16(rng, (H,), 0.3)
    bank = np.broadcast_to(v, (N, M, H))
    eps = 1e-6
    new_p, out, _ = _op(v, np.zeros((M, H)), None, bank, w, gamma, eps)
    assert (new_p == _b(v)).all()
    ref = torch.nn.functional.rms_norm(torch.from_numpy(v), (H,), torch.from_numpy(gamma),
                                       float(np.float32(eps))).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)


def test_zero_query_gives_mean_of_sources():
    """w = 0: all logits are 0, alpha = 1/(N+1) and h is the mean of the N bank
    snapshots and the UPDATED prefix; out = rms_norm(mean) * gamma."""
    rng = np.random.default_rng(11)
    H, N, M = 32, 4, 2
    bank = _rand_bf16(rng, (N, M, H))
    prefix = _rand_bf16(rng, (M, H))
    add = _rand_bf16(rng, (M, H))
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    new_p, out, _ = _op(prefix, add, None, bank, np.zeros(H), gamma, 1e-6)
    src = np.concatenate([bank, bf16_decode(new_p)[None]], axis=0)
    mean = src.sum(axis=0) / (N + 1)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(mean), (H,), torch.from_numpy(gamma),
                                       float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("k,N", [(0, 5), (2, 5), (5, 5), (17, 31), (31, 31)])
def test_dominant_source_selected(k, N):
    """w = 1 * v_k: l_k ~ H * rms(v_k) while the other logits are O(sqrt H), so
    alpha -> e_k and out -> rms_norm(v_k) * gamma.  Source N is the updated
    prefix.  A flipped logit sign would select the opposite end."""
    rng = np.random.default_rng(12 + k + N)
    H = 256
    bank = _rand_bf16(rng, (N, 1, H))
    prefix = _rand_bf16(rng, (1, H))
    add = _rand_bf16(rng, (1, H))
    new_p = bf16_decode(_op(prefix, add, None, bank, np.zeros(H), np.ones(H), 1e-6)[0])
    src = np.concatenate([bank[:, 0], new_p], axis=0)
    w = src[k]
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    _, out, _ = _op(prefix, add, None, bank, w, gamma, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(src[k][None]), (H,), torch.from_numpy(gamma),
                                       float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


def test_logits_are_scale_invariant():
    """Doubling a snapshot (exact in BF16) leaves its logit w . RMSNorm(v) and
    hence alpha unchanged (up to eps), while h sees the doubled row."""
    rng = np.random.default_rng(13)
    H, N = 128, 3
    V = _rand_bf16(rng, (1, N + 1, H))
    w = _rand_bf16(rng, (H,), 1 / math.sqrt(H))
    g = np.ones(H)
    r1 = mixture(V, w, g, 1e-6)
    V2 = V.copy()
    V2[0, 1] *= 2
    r2 = mixture(V2, w, g, 1e-6)
    np.testing.assert_allclose(r1["logits"], r2["logits"], rtol=1e-5)
    np.testing.assert_allclose(r1["alpha"], r2["alpha"], rtol=1e-5)
    assert not np.allclose(r1["h"], r2["h"])


def test_bank_permutation_invariance():
    rng = np.random.default_rng(14)
    H, N, M = 64, 6, 2
    bank = _rand_bf16(rng, (N, M, H))
    prefix, add, add2 = (_rand_bf16(rng, (M, H)) for _ in range(3))
    w = _rand_bf16(rng, (H,), 0.2)
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    perm = rng.permutation(N)
    _, o1, _ = _op(prefix, add, add2, bank, w, gamma, 1e-6)
    _, o2, _ = _op(prefix, add, add2, bank[perm], w, gamma, 1e-6)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)


def test_tokens_are_independent_and_subsettable():
    rng = np.random.default_rng(15)
    H, N, M = 32, 3, 5
    bank = _rand_bf16(rng, (N, M, H))
    prefix, add, add2 = (_rand_bf16(rng, (M, H)) for _ in range(3))
    w = _rand_bf16(rng, (H,), 0.2)
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    args = [_b(x) for x in (prefix, add, add2, bank, w, gamma)]
    p_all, o_all, _ = attnres_add_rmsnorm(*args, 1e-6)
    p_sub, o_sub, _ = attnres_add_rmsnorm(*args, 1e-6, tokens=np.array([4, 1]))
    assert (p_sub == p_all[[4, 1]]).all()
    np.testing.assert_array_equal(o_sub, o_all[[4, 1]])


def _mp_reference(src, w, gamma, eps):
    """50-digit evaluation of one token from the definition."""
    mpmath.mp.dps = 50
    S, H = src.shape
    eps = mpmath.mpf(float(np.float32(eps)))
    v = [[mpmath.mpf(float(x)) for x in row] for row in src]
    wm = [mpmath.mpf(float(x)) for x in w]
    logits = []
    for i in range(S):
        ms = mpmath.fsum(x * x for x in v[i]) / H
        dot = mpmath.fsum(a * b for a, b in zip(wm, v[i]))
        logits.append(dot / mpmath.sqrt(ms + eps))
    mx = max(logits)
    ex = [mpmath.exp(li - mx) for li in logits]
    z = mpmath.fsum(ex)
    alpha = [e / z for e in ex]
    h = [mpmath.fsum(alpha[i] * v[i][j] for i in range(S)) for j in range(H)]
    rh = 1 / mpmath.sqrt(mpmath.fsum(x * x for x in h) / H + eps)
    return np.array([float(h[j] * rh * mpmath.mpf(float(gamma[j]))) for j in range(H)])


@pytest.mark.parametrize("H,N,M", [(8, 1, 2), (16, 2, 3), (8, 12, 1), (8, 20, 1), (16, 31, 1)])
def test_brute_force_high_precision(H, N, M):
    rng = np.random.default_rng(100 + H + N)
    bank = _rand_bf16(rng, (N, M, H))
    prefix, add, add2 = (_rand_bf16(rng, (M, H)) for _ in range(3))
    w = _rand_bf16(rng, (H,), 1 / math.sqrt(H))
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    new_p, out, _ = _op(prefix, add, add2, bank, w, gamma, 1e-6)
    for m in range(M):
        src = np.concatenate([bank[:, m], bf16_decode(new_p[m])[None]], axis=0)
        ref = _mp_reference(src, w, gamma, 1e-6)
        np.testing.assert_allclose(out[m], ref, rtol=1e-13, atol=1e-15)


def test_alone_equals_fold_with_zero_addend():
    """The attention-residual alone is the fused op with a +0 addend (the
    fold then leaves every value of the prefix unchanged)."""
    from oracle import attnres_rmsnorm
    rng = np.random.default_rng(16)
    H, N, M = 64, 4, 3
    bank = _rand_bf16(rng, (N, M, H))
    prefix = _rand_bf16(rng, (M, H))
    w = _rand_bf16(rng, (H,), 0.2)
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    out_a, _ = attnres_rmsnorm(_b(prefix), _b(bank), _b(w), _b(gamma), 1e-6)
    _, out_f, _ = _op(prefix, np.zeros((M, H)), None, bank, w, gamma, 1e-6)
    np.testing.assert_array_equal(out_a, out_f)


@pytest.mark.parametrize("b", [0.5, -1.25])
def test_closed_form_alone_and_tap(b):
    """No fold: the prefix (1, -1) is the second source directly; the tap is
    the pre-norm mixture h = (1, tanh(b r)) of the two-source closed form."""
    from oracle import attnres_rmsnorm
    e32 = float(np.float32(1e-6))
    gamma = [1.5, 0.75]
    out, _, h, _ = attnres_rmsnorm(_b([[1.0, -1.0]]), _b([[[1.0, 1.0]]]), _b([0.0, b]), _b(gamma),
                                   1e-6, with_h=True)
    t = math.tanh(b / math.sqrt(1.0 + e32))
    s = 1.0 / math.sqrt((1.0 + t * t) / 2.0 + e32)
    np.testing.assert_allclose(h[0], [1.0, t], rtol=1e-14)
    np.testing.assert_allclose(out[0], [1.5 * s, 0.75 * t * s], rtol=1e-14)


def test_no_snapshots_is_rmsnorm_of_the_new_prefix():
    """N = 0: the updated prefix is the only source, alpha = 1, and out is
    torch's rms_norm of it."""
    rng = np.random.default_rng(17)
    H, M = 96, 4
    prefix, add, add2 = (_rand_bf16(rng, (M, H)) for _ in range(3))
    gamma = _bf(1 + 0.1 * _rand_bf16(rng, (H,)))
    w = _rand_bf16(rng, (H,), 0.3)
    new_p, out, _ = _op(prefix, add, add2, np.zeros((0, M, H)), w, gamma, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(bf16_decode(new_p)), (H,),
                                       torch.from_numpy(gamma), float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)
