"""Oracle of int4 block-scaled weight-only quantization ("Q4S", block 64).

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` alone; no code shared with
the library.

k2-burn README, "Post-training quantization" / "Quantization": the quantize
step produces int4 "Q4S" checkpoints with block size 64, and only the Linear
weights (the projections and the lm_head) are quantized.  The page names the
scheme, the bit width and the block size only; the reading taken:

  * a block is 64 consecutive weights of one row (one output feature) along
    the input dimension; a row whose length is not a multiple of 64 ends in a
    shorter block;
  * "S", symmetric: signed codes in [-7, 7] (the range symmetric about zero),
    no zero point;
  * each block's scale s = max|w| / 7, one float32 division;
  * code = w / s (one float32 division) rounded to the nearest integer, ties
    to even, clamped to [-7, 7]; a block of zeros gets s = 0 and codes 0;
  * the weight the model computes with is code * s.
"""
import numpy as np

F32 = np.float32
BLOCK = 64
QMAX = 7


def quantize_rows(w, block=BLOCK):
    """(codes [rows, cols] int8 in [-7, 7], scales [rows, ceil(cols / block)]
    float32) of float32 rows."""
    w = np.asarray(w, dtype=F32)
    rows, cols = w.shape
    nb = (cols + block - 1) // block
    codes = np.zeros((rows, cols), dtype=np.int8)
    scales = np.zeros((rows, nb), dtype=F32)
    for b in range(nb):
        blk = w[:, b * block:(b + 1) * block]
        amax = np.max(np.abs(blk), axis=1).astype(F32)
        s = (amax / F32(QMAX)).astype(F32)
        safe = np.where(s > 0, s, F32(1.0)).astype(F32)
        q = np.rint((blk / safe[:, None]).astype(F32)).astype(np.float64)  # nearest, ties to even
        q = np.clip(q, -QMAX, QMAX)
        q[s == 0] = 0
        codes[:, b * block:(b + 1) * block] = q.astype(np.int8)
        scales[:, b] = s
    return codes, scales


def dequantize_rows(codes, scales, block=BLOCK):
    """The weights the int4 model computes with (float64): code * its block's scale."""
    codes = np.asarray(codes, dtype=np.float64)
    per_col = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=1)[:, :codes.shape[1]]
    return codes * per_col


def matvec(codes, scales, x, block=BLOCK):
    """y = W x computed the way the format is defined: each block's integer
    dot product times the block's scale, summed over blocks (float64)."""
    codes = np.asarray(codes, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    y = np.zeros(codes.shape[0])
    for b in range(scales.shape[1]):
        sl = slice(b * block, (b + 1) * block)
        y += np.asarray(scales[:, b], dtype=np.float64) * (codes[:, sl] @ x[sl])
    return y


PROJECTIONS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def q4_weights(get):
    """A weight getter (name, layer) -> values, with every projection matrix and
    the lm_head replaced by its int4 quantization (embedding and gains kept)."""
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
