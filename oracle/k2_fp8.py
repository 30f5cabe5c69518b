"""Oracle of fp8 (E4M3) weight-only quantization.

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` alone; no code shared with
the library.

k2-burn README, "Post-training quantization": a quantize step produces fp8
(E4M3) checkpoints that the engine runs directly.  The page names the format
only; the reading taken: one fp32 scale per weight row
(output feature), s = max|w| / 448 (448 = the largest finite E4M3 value),
code = E4M3(w / s) rounded to nearest, ties to even, saturating at +-448; a
row of zeros gets s = 0 and codes 0.  The weight the model computes with is
E4M3(code) * s.

E4M3 (the OCP 8-bit floating point format): 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; no
infinities; the all-ones exponent with mantissa 7 is NaN, so the largest
finite magnitude is 1.75 * 2^8 = 448.  The division w / s is one float32
operation, as on the device.
"""
import numpy as np

F32 = np.float32


def e4m3_value(code: int) -> float:
    """The real number an E4M3 code stands for (NaN for the two NaN codes)."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_VALUES = np.array([e4m3_value(c) for c in range(256)])
_POS_CODES = np.arange(0, 0x7F)        # 0 .. 0x7E: the non-negative finite codes, increasing
_POS_VALUES = E4M3_VALUES[_POS_CODES]
assert np.all(np.diff(_POS_VALUES) > 0)


def e4m3_encode(x) -> np.ndarray:
    """uint8 codes of float32 values: nearest, ties to the even code, saturating;
    the sign is kept (negative values rounding to zero give 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), _POS_VALUES[-1])
    hi = np.clip(np.searchsorted(_POS_VALUES, a), 1, _POS_VALUES.size - 1)
    lo = hi - 1
    dlo, dhi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(_POS_CODES[lo] % 2 == 0, lo, hi)))
    pick = np.where(a <= 0.0, 0, pick)
    codes = _POS_CODES[pick].astype(np.uint8)
    # sign-magnitude: rounding keeps the sign, so a negative value that rounds
    # to zero is negative zero (0x80), as in IEEE 754 rounding
    return np.where(np.signbit(x), codes | 0x80, codes).astype(np.uint8)


def quantize_rows(w):
    """(codes [rows, cols] uint8, scales [rows] float32) of float32 rows."""
    w = np.asarray(w, dtype=F32)
    amax = np.max(np.abs(w), axis=1).astype(F32)
    scale = (amax / F32(448.0)).astype(F32)
    safe = np.where(scale > 0, scale, F32(1.0)).astype(F32)
    codes = e4m3_encode((w / safe[:, None]).astype(F32))
    codes[scale == 0] = 0
    return codes, scale


def dequantize_rows(codes, scales):
    """The weights the fp8 model computes with (float64)."""
    return E4M3_VALUES[codes] * np.asarray(scales, dtype=np.float64)[:, None]


PROJECTIONS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def fp8_weights(get):
    """A weight getter (name, layer) -> values, with every projection matrix and
    the lm_head replaced by its fp8 quantization (embedding and gains kept)."""
    cache = {}

    def getq(name, layer):
        w = get(name, layer)
        if name not in PROJECTIONS and name != "lm_head":
            return w
        key = (name, layer)
        if key not in cache:
            cache[key] = dequantize_rows(*quantize_rows(np.asarray(w, dtype=F32)))
        return cache[key]

    return getq
