"""Pins of the fp8 (E4M3) quantization oracle against the format's definition."""
import numpy as np

from oracle import k2_fp8 as Q8

F32 = np.float32


def test_e4m3_table_landmarks():
    v = Q8.E4M3_VALUES
    assert v[0x00] == 0.0 and v[0x38] == 1.0 and v[0x40] == 2.0 and v[0x30] == 0.5
    assert v[0x7E] == 448.0 and np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0xB8] == -1.0 and v[0xFE] == -448.0
    finite = v[~np.isnan(v)]
    assert finite.size == 254 and np.max(finite) == 448.0


def test_encode_is_round_to_nearest_even_and_saturates():
    vals = Q8.E4M3_VALUES
    for c in range(0x7E):  # every pair of neighbours: the midpoint goes to the even code
        a, b = vals[c], vals[c + 1]
        mid = (a + b) / 2
        assert Q8.e4m3_encode([mid])[0] == (c if c % 2 == 0 else c + 1)
        assert Q8.e4m3_encode([np.nextafter(mid, -1)])[0] == c
        assert Q8.e4m3_encode([np.nextafter(mid, 2e3)])[0] == c + 1
        assert Q8.e4m3_encode([a])[0] == c
    assert Q8.e4m3_encode([1e9, -1e9, 449.0, 480.0]).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]
    # rounding keeps the sign: negative values that round to zero are negative zero
    assert Q8.e4m3_encode([-0.0, 0.0, 1e-12, -1e-12]).tolist() == [0x80, 0, 0, 0x80]
    assert Q8.E4M3_VALUES[0x80] == 0.0
    assert Q8.e4m3_encode([-1.0, -0.5]).tolist() == [0xB8, 0xB0]


def test_row_quantization_error_and_scale():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 300)) * 0.02).astype(F32)
    w[5] = 0.0
    codes, s = Q8.quantize_rows(w)
    assert s[5] == 0 and not codes[5].any()
    d = Q8.dequantize_rows(codes, s)
    for r in range(64):
        if r == 5:
            continue
        # each element within half a step of its binade: relative error <= 2^-4 (3 mantissa bits)
        big = np.abs(w[r]) >= s[r] * 2.0 ** -6  # normal codes
        rel = np.abs(d[r][big] - w[r][big]) / np.abs(w[r][big])
        assert np.max(rel) <= 2.0 ** -4 + 1e-6
        # the row's largest magnitude is the largest code, +-448
        assert codes[r][np.argmax(np.abs(w[r]))] & 0x7F == 0x7E
