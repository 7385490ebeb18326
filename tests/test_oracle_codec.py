"""Pins of the oracle's integer BF16 codec against torch's conversions and
against the definition of round-to-nearest-even (no GPU)."""
import numpy as np
import pytest
import torch

from oracle import bf16_decode, bf16_encode_rne


def _torch_bits_to_f64(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def test_decode_all_patterns_match_torch():
    allb = np.arange(65536, dtype=np.uint16)
    ours = bf16_decode(allb)
    ref = _torch_bits_to_f64(allb)
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    # the sign of zero survives
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0x0000])


@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x3B80, 2.0 ** -8), (0x0001, 2.0 ** -133),
    (0x007F, 127 * 2.0 ** -133), (0x0080, 2.0 ** -126), (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127),
    (0x3FC0, 1.5), (0x4049, 3.140625),
])
def test_decode_known_values(bits, value):
    assert bf16_decode(np.array([bits], np.uint16))[0] == value


def test_encode_roundtrip_all_finite():
    allb = np.arange(65536, dtype=np.uint16)
    v = bf16_decode(allb)
    fin = ~np.isnan(v)
    assert (bf16_encode_rne(v[fin]) == allb[fin]).all()


def test_encode_matches_torch_float32_rounding():
    """torch rounds float32 -> bfloat16 to nearest even; every float32 is exact
    in float64, so a single rounding from float64 must agree bit for bit."""
    torch.set_flush_denormal(False)
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # plus every float32 whose low 16 bits sit at the rounding boundary
    hi = rng.integers(0, 2 ** 16, size=200_000, dtype=np.uint64).astype(np.uint32) << 16
    u = np.concatenate([u, hi | 0x8000, hi | 0x7FFF, hi | 0x8001, hi])
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (bf16_encode_rne(f.astype(np.float64)) == ref).all()


def test_encode_is_nearest_and_ties_even():
    """Property check from the definition: the result is a nearest BF16 value
    and, at an exact midpoint, the one with an even mantissa."""
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(200_000) * np.exp2(rng.integers(-140, 120, 200_000)),
        # exact midpoints between neighbouring BF16 values
        (bf16_decode(np.arange(1, 0x7F7F, 7, dtype=np.uint16)) +
         bf16_decode(np.arange(2, 0x7F80, 7, dtype=np.uint16))) / 2,
    ])
    b = bf16_encode_rne(x).astype(np.int64)
    mag_bits = b & 0x7FFF
    y = bf16_decode(b.astype(np.uint16))
    lo = bf16_decode(((mag_bits - 1).clip(0) | (b & 0x8000)).astype(np.uint16))
    hi = bf16_decode(((mag_bits + 1).clip(max=0x7F7F) | (b & 0x8000)).astype(np.uint16))
    err = np.abs(y - x)
    assert (err <= np.abs(lo - x)).all() and (err <= np.abs(hi - x)).all()
    tie = (err == np.abs(lo - x)) & (mag_bits > 0) | (err == np.abs(hi - x)) & (mag_bits < 0x7F7F)
    tie &= err > 0
    assert (mag_bits[tie] % 2 == 0).all()


def test_encode_specials():
    v = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e39, -1e39, 2.0 ** -134, 2.0 ** -134 * 1.0001])
    b = bf16_encode_rne(v)
    assert list(b) == [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x7F80, 0xFF80, 0x0000, 0x0001]
