"""Pins for the oracle's 16-bit formats: NumPy's float16 conversion, torch's bfloat16
conversion of float32 values, and hand-made ties (round half to even)."""
import numpy as np
import pytest
import torch

from oracle import formats


def test_fp16_matches_numpy_float64_conversion():
    # NumPy converts float64 -> float16 directly with round-to-nearest-even.
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000) * 4,
        rng.standard_normal(2000) * 1e-6,          # subnormal range of fp16
        rng.standard_normal(2000) * 7e4,           # overflow range
        np.array([65504.0, 65519.999, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25, 0.0, -0.0]),
    ])
    got = formats.encode_bits(x, "fp16")
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_bf16_matches_torch_on_float32_values():
    # For float32 inputs torch's bfloat16 conversion is a single correct RNE rounding.
    rng = np.random.default_rng(2)
    x32 = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 3,
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormal range
        np.array([3.39e38, -3.39e38, 1.0, -0.0], dtype=np.float32),
    ])
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = formats.encode_bits(x32.astype(np.float64), "bf16")
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("dtype,mant", [("fp16", 10), ("bf16", 7)])
def test_ties_go_to_even(dtype, mant):
    ulp = 2.0 ** -mant
    # halfway between 1 and 1+ulp -> 1 (even); halfway between 1+ulp and 1+2ulp -> 1+2ulp
    assert formats.round_rne(1.0 + ulp / 2, dtype) == 1.0
    assert formats.round_rne(1.0 + 1.5 * ulp, dtype) == 1.0 + 2 * ulp
    assert formats.round_rne(-(1.0 + 1.5 * ulp), dtype) == -(1.0 + 2 * ulp)
    # just above a tie rounds up; float64 keeps the tiny excess that float32 would lose
    assert formats.round_rne(1.0 + ulp / 2 + 2.0 ** -40, dtype) == 1.0 + ulp


def test_no_double_rounding_from_float64():
    # x lies just above the bf16 tie 1 + 2^-8, but a float32 step would land exactly on
    # the tie (2^-25 is a quarter of float32's spacing at 1) and then round down to 1.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -25
    assert np.float32(x) == np.float32(1.0 + 2.0 ** -8)
    assert formats.round_rne(x, "bf16") == 1.0 + 2.0 ** -7


def test_decode_encode_roundtrip_all_patterns():
    for dtype in ("fp16", "bf16"):
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        vals = formats.decode_bits(bits, dtype)
        back = formats.encode_bits(vals, dtype)
        finite = np.isfinite(vals)
        np.testing.assert_array_equal(back[finite], bits[finite])
        assert np.all(back[np.isnan(vals)] == formats.FORMATS[dtype]["qnan"])


def test_planted_round_half_up_is_caught():
    """A plausible mistake (round half away from zero) fails the tie pin."""
    def round_half_up(x, dtype):
        f = formats.FORMATS[dtype]
        x = np.asarray(x, dtype=np.float64)
        _, e2 = np.frexp(x)
        q = np.ldexp(1.0, np.maximum(e2 - 1, f["emin"]) - f["mant"])
        return np.floor(x / q + 0.5) * q
    ulp = 2.0 ** -7
    assert round_half_up(1.0 + ulp / 2, "bf16") != 1.0
