"""The parity criterion itself (no GPU)."""
import numpy as np

from oracle import bf16_encode_rne, check_out, ulp_bf16


def test_ulp_values():
    assert ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7
    assert ulp_bf16(np.array([3.0]))[0] == 2.0 ** -6
    assert ulp_bf16(np.array([-0.75]))[0] == 2.0 ** -8
    assert ulp_bf16(np.array([2.0 ** -130]))[0] == 2.0 ** -133


def test_correct_rounding_passes_and_three_ulp_fails():
    ref = np.array([1.0 + 2.0 ** -9, 0.3, -1.7])
    ok = check_out(bf16_encode_rne(ref), ref, np.abs(ref))
    assert ok["ok"] and ok["max_ulp"] <= 0.5
    bad = check_out(bf16_encode_rne(ref + 3 * ulp_bf16(ref)), ref, np.abs(ref))
    assert not bad["ok"]


def test_cap_at_large_magnitude():
    # |ref| in [2, 4): one ulp is 2^-6 = 0.0156 > 1.5e-2, so a 1-ulp miss fails the cap
    ref = np.array([3.0])
    assert not check_out(bf16_encode_rne(np.array([3.0 + 2.0 ** -6])), ref, ref)["ok"]
    ref = np.array([5.0])   # above 4 only the 2-ulp rule applies
    assert check_out(bf16_encode_rne(np.array([5.0 + 2.0 ** -5])), ref, ref)["ok"]


def test_floor_for_cancelled_outputs():
    ref = np.array([1e-7])
    got = bf16_encode_rne(np.array([1e-7 + 3e-8]))
    r = check_out(got, ref, np.array([1.0]))
    assert r["ok"] and r["n_floor"] == 1
    # the floor needs the float32 error model to hold as well
    assert not check_out(got, ref, np.array([1e-3]))["ok"]


# ---- the error scale the criterion uses: bound_j = r_h |gamma_j| sum_i alpha_i |v_ij|
# (out) and h_bound_j = sum_i alpha_i |v_ij| (the mixture tap), pinned on two
# hand-computed two-source cases (H = 2, N = 1: v_0 = bank[0] = (1, -1), and
# the updated prefix v_1 = prefix + 0 = (3, 1); gamma = (1, -2); eps = 2^-20).

def _two_source_case(w):
    from oracle import attnres_add_rmsnorm
    enc = lambda *x: bf16_encode_rne(np.array(x, dtype=np.float64))  # noqa: E731
    bank = enc(1.0, -1.0).reshape(1, 1, 2)
    prefix = enc(3.0, 1.0).reshape(1, 2)
    add = enc(0.0, 0.0).reshape(1, 2)
    eps = 2.0 ** -20
    return attnres_add_rmsnorm(prefix, add, None, bank, enc(*w), enc(1.0, -2.0), eps, with_h=True)


def test_error_scale_uniform_weights():
    """w = 0: both logits 0, alpha = (1/2, 1/2); h = (2, 0), mean(h^2) = 2,
    r_h = 1/sqrt(2 + 2^-20).  By hand: out = (2 r_h, 0); bound = r_h * (1 *
    (1 + 3)/2, 2 * (1 + 1)/2) = (2 r_h, 2 r_h); h_bound = (2, 1)."""
    np_bits, out, bound, h, hb = _two_source_case((0.0, 0.0))
    r_h = 1.0 / np.sqrt(2.0 + 2.0 ** -20)
    assert np.allclose(h[0], [2.0, 0.0], rtol=0, atol=1e-15)
    assert np.allclose(out[0], [2.0 * r_h, 0.0], rtol=1e-14, atol=1e-15)
    assert np.allclose(bound[0], [2.0 * r_h, 2.0 * r_h], rtol=1e-14, atol=0)
    assert np.allclose(hb[0], [2.0, 1.0], rtol=1e-14, atol=0)


def test_error_scale_one_dominant_source():
    """w = (0, 1024): d = (-1024, 1024), logits about -1024 and +458, so
    alpha_0 = exp(-1482) is 0 in float64 and alpha = (0, 1): h = v_1 = (3, 1),
    r_h = 1/sqrt(5 + 2^-20).  By hand: out = (3 r_h, -2 r_h); bound =
    (3 r_h, 2 r_h); h_bound = (3, 1).  (A swapped source order would give
    h_bound = (1, 1).)"""
    np_bits, out, bound, h, hb = _two_source_case((0.0, 1024.0))
    r_h = 1.0 / np.sqrt(5.0 + 2.0 ** -20)
    assert np.array_equal(h[0], [3.0, 1.0])
    assert np.allclose(out[0], [3.0 * r_h, -2.0 * r_h], rtol=1e-14, atol=0)
    assert np.allclose(bound[0], [3.0 * r_h, 2.0 * r_h], rtol=1e-14, atol=0)
    assert np.array_equal(hb[0], [3.0, 1.0])
