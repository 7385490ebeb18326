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
