"""Pins of the int4 block quantization oracle (oracle/k2_q4.py) against the
definition of symmetric block quantization, without a GPU.

  * a hand-worked block whose scale is a power of two, so every quotient is
    exact and the ties (x.5) show the rounding rule;
  * each code is the integer of [-7, 7] nearest to the float32 quotient, ties
    to the even one (brute force over the 15 candidates);
  * blocks run along the row: 64 consecutive weights, a ragged last block,
    and changing one weight touches only its own block;
  * |w - c s| <= s / 2, and the largest magnitude of a block takes code +-7;
  * the block-wise product (integer dot product times scale) equals a plain
    loop over the dequantized weights.
"""
import numpy as np

from oracle import k2_q4 as Q4

F32 = np.float32


def test_hand_worked_block():
    # amax 0.875 -> s = 0.125 exactly: quotients 7, -3.5, 0.5, 1.5, 2.5, -0.5, 6.5, -7, 0.25, -6.75
    vals = [0.875, -0.4375, 0.0625, 0.1875, 0.3125, -0.0625, 0.8125, -0.875, 0.03125, -0.84375]
    w = np.zeros((1, 64), F32)
    w[0, :len(vals)] = vals
    codes, s = Q4.quantize_rows(w)
    assert s.shape == (1, 1) and s[0, 0] == F32(0.125)
    assert codes[0, :len(vals)].tolist() == [7, -4, 0, 2, 2, 0, 6, -7, 0, -7]
    assert not codes[0, len(vals):].any()


def brute_code(q):
    cands = np.arange(-7, 8, dtype=np.float64)
    d = np.abs(cands - float(q))
    best = cands[d == d.min()]
    return int(best[0]) if best.size == 1 else int(best[np.mod(best, 2) == 0][0])


def test_codes_are_the_nearest_integer_ties_to_even():
    rng = np.random.default_rng(8)
    w = (rng.standard_normal((6, 192)) * 0.03).astype(F32)
    # quotients landing on exact halves: a block with scale 1/8 (amax 7/8)
    w[0, :64] = (rng.integers(-14, 15, 64) / 16.0).astype(F32)
    w[0, 0] = F32(0.875)
    codes, s = Q4.quantize_rows(w)
    for r in range(w.shape[0]):
        for c in range(w.shape[1]):
            sb = s[r, c // 64]
            q = (w[r, c] / sb).astype(F32)
            assert codes[r, c] == brute_code(q), (r, c)
    q = w[0, :64].astype(np.float64) / float(s[0, 0])
    assert np.any(q - np.floor(q) == 0.5)  # the block holds ties


def test_blocks_run_along_the_row_with_a_ragged_tail():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((3, 150)) * 0.1).astype(F32)
    codes, s = Q4.quantize_rows(w)
    assert s.shape == (3, 3)
    for r in range(3):
        for b, (lo, hi) in enumerate([(0, 64), (64, 128), (128, 150)]):
            assert s[r, b] == F32(np.max(np.abs(w[r, lo:hi])) / F32(7))
    w2 = w.copy()
    w2[1, 70] = F32(5.0)  # only block (1, 1) changes
    c2, s2 = Q4.quantize_rows(w2)
    changed = s2 != s
    assert changed.sum() == 1 and changed[1, 1]
    diff = np.nonzero((c2 != codes).any(axis=0))[0]
    assert diff.min() >= 64 and diff.max() < 128 and np.array_equal(np.nonzero((c2 != codes).any(axis=1))[0], [1])


def test_error_bound_extremes_and_zero_blocks():
    rng = np.random.default_rng(10)
    w = (rng.standard_normal((16, 256)) * 0.02).astype(F32)
    w[4, 64:128] = 0.0
    codes, s = Q4.quantize_rows(w)
    assert s[4, 1] == 0 and not codes[4, 64:128].any()
    assert codes.min() >= -7 and codes.max() <= 7
    d = Q4.dequantize_rows(codes, s)
    per_col = np.repeat(s.astype(np.float64), 64, axis=1)
    assert np.all(np.abs(d - w) <= per_col / 2 * (1 + 1e-6))
    for r in range(16):
        for b in range(4):
            blk = w[r, 64 * b:64 * (b + 1)]
            if s[r, b] > 0:
                assert abs(int(codes[r, 64 * b + int(np.argmax(np.abs(blk)))])) == 7


def test_blockwise_product_equals_a_plain_loop():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((5, 130)) * 0.05).astype(F32)
    x = rng.standard_normal(130)
    codes, s = Q4.quantize_rows(w)
    y = Q4.matvec(codes, s, x)
    for r in range(5):
        want = sum(float(codes[r, k]) * float(s[r, k // 64]) * x[k] for k in range(130))
        assert abs(y[r] - want) <= 1e-12 * max(1.0, abs(want))
