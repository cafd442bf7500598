"""Pins of the FP8 (E4M3) Stage-2 weight oracle against sources other than itself: the format's
closed-form value set, torch's float8_e4m3fn cast, saturation, and the per-row scale rule.
(Technical summary, "Experimental Results", Compatibility: Prox is orthogonal to FP8 weight
quantization.)"""
import numpy as np
import torch

import oracle.fp8_weights as F8


def _closed_form_values():
    """Every finite non-negative E4M3 value from the format's definition: exponent field
    e in 1..15 (bias 7) with mantissa m in 0..7, except e = 15, m = 7 (NaN); subnormals
    m / 8 * 2^-6."""
    vals = {m / 8 * 2.0 ** -6 for m in range(8)}
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.add((1 + m / 8) * 2.0 ** (e - 7))
    return np.array(sorted(vals))


def test_value_set_is_the_format():
    v = _closed_form_values()
    assert len(v) == 127 and v.max() == 448.0 and v[1] == 2.0 ** -9
    # every format value is a fixed point, and the codes are the format's bit patterns
    np.testing.assert_array_equal(F8.e4m3_round(v.astype(np.float32)), v)
    np.testing.assert_array_equal(F8.e4m3_round(-v.astype(np.float32)), -v)
    codes = F8.e4m3_bits(v)
    from_bits = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(from_bits.astype(np.float64), v)


def test_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(400_000) * rng.choice([1e-4, 1e-2, 1.0, 30.0, 200.0], 400_000))
    x = np.clip(x, -448, 448).astype(np.float32)
    # the midpoints between neighbouring values (ties go to the even mantissa)
    v = _closed_form_values()
    mids = ((v[1:] + v[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(F8.e4m3_round(x), want)


def test_saturation_and_zero():
    got = F8.e4m3_round(np.array([448.0, 449.0, 470.0, 1e6, -1e9, 0.0, -0.0], np.float32))
    np.testing.assert_array_equal(got, [448, 448, 448, 448, -448, 0, 0])
    # values that round to zero keep their sign, as torch's cast does
    tiny = np.array([1e-4, -1e-4, 2.0 ** -11, -(2.0 ** -11), 0.0, -0.0], np.float32)
    want = torch.from_numpy(tiny).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F8.e4m3_bits(F8.e4m3_round(tiny)), want)
    assert list(want) == [0, 0x80, 0, 0x80, 0, 0x80]


def test_row_scale_rule():
    rng = np.random.default_rng(1)
    w = torch.from_numpy(rng.standard_normal((64, 256)).astype(np.float32) * 0.02)
    w = w.to(torch.bfloat16).float().numpy()
    w[3] = 0.0                                            # an all-zero row: scale 0, codes 0
    q, s = F8.quantize_rows_e4m3(w)
    amax = np.abs(w).max(axis=1)
    np.testing.assert_array_equal(s, (amax / np.float32(448)).astype(np.float32))
    assert s[3] == 0 and not q[3].any()
    # the largest entry of each row maps to about +-448; relative error within half a step
    for r in (0, 10, 63):
        j = np.argmax(np.abs(w[r]))
        assert abs(abs(q[r, j]) - 448) <= 16
    nz = np.abs(w) > 2.0 ** -6 * s[:, None]               # normal range of the row
    rel = np.abs(q * s[:, None] - w)[nz] / np.abs(w)[nz]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)
