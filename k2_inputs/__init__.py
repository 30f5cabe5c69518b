"""Seeded synthetic inputs for the K2-Horizon dense GQA decoder.

This module is shared by the CPU oracle tests and by the CUDA path, and it holds
none of the decoder's arithmetic: only model shapes, seeded random tensors
(weights, prompt ids, pre-filled KV rows) and the storage rounding of those
inputs to the dtype they are stored in (bf16 weights, fp16 KV rows).

The pages run a trained checkpoint that is not available, so every input is
random-init data of the published shape (k2-burn README, "Model shape"), in the
spirit of the synthetic weight constructors of cpu_weights.rs
(`synthetic_tiny`, `synthetic_prod_width_dummy`).

Recipe (all deterministic, independent of thread count):
  * weights: N(0, 1) * 0.02 drawn as float32 by numpy's PCG64 generator, one
    stream per (seed, tensor id, 4 Mi-element chunk); rounded to bf16 with
    round-to-nearest-even when the model stores bf16 weights;
  * norm gains: 1 (``gain_scale`` > 0 draws 1 + N(0,1)*gain_scale instead, used
    by tests that must see the gain applied);
  * prompt ids: uniform integers in [0, vocab) from PCG64(seed);
  * pre-filled KV rows: N(0, 1) float32 rounded to fp16.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

# ----------------------------------------------------------------------------
# shapes
# ----------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Shape of a dense GQA decoder (field names follow the model's config)."""

    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    norm_groups: int
    vocab: int
    eps: float = 1e-6
    rope_theta: float = 10000.0
    weight_dtype: str = "bf16"  # "f32" | "bf16"

    def replace(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)


# tiny fp32 model: 16 prompt ids then 16 greedy steps, fp32 KV
TINY = ModelShape(hidden=64, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=16,
                  intermediate=256, norm_groups=2, vocab=512, weight_dtype="f32")
# the 3.7B shape (k2-burn README, "Model shape")
K2_3P7B = ModelShape(hidden=2560, n_layers=36, n_heads=32, n_kv_heads=8, head_dim=128,
                     intermediate=10240, norm_groups=2, vocab=250624, weight_dtype="bf16")
# one decoder layer of the 3.7B shape (the embedding/lm_head are small, unused
# by the layer-only step)
K2_LAYER = K2_3P7B.replace(n_layers=1, vocab=512)
# a medium bf16 model: several GEMV tiles per CTA, a ragged vocab tail, 3 layers
MEDIUM = ModelShape(hidden=512, n_layers=3, n_heads=8, n_kv_heads=2, head_dim=64,
                    intermediate=1536, norm_groups=2, vocab=1000, weight_dtype="bf16")

SHAPES = {"tiny": TINY, "k2_3p7b": K2_3P7B, "k2_layer": K2_LAYER, "medium": MEDIUM}

LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


def tensor_shape(s: ModelShape, name: str) -> tuple:
    """nn.Linear convention: a projection weight is [out_features, in_features]."""
    H, d = s.hidden, s.head_dim
    return {
        "embed": (s.vocab, H),
        "lm_head": (s.vocab, H),
        "final_norm": (H,),
        "attn_norm": (H,),
        "mlp_norm": (H,),
        "wq": (s.n_heads * d, H),
        "wk": (s.n_kv_heads * d, H),
        "wv": (s.n_kv_heads * d, H),
        "wo": (H, s.n_heads * d),
        "w_gate": (s.intermediate, H),
        "w_up": (s.intermediate, H),
        "w_down": (H, s.intermediate),
    }[name]


def tensor_id(s: ModelShape, name: str, layer: int = -1) -> int:
    """Fixed draw order: embed, per layer the nine layer tensors, final_norm, lm_head."""
    if name == "embed":
        return 0
    if name == "final_norm":
        return 1 + 9 * s.n_layers
    if name == "lm_head":
        return 2 + 9 * s.n_layers
    assert 0 <= layer < s.n_layers
    return 1 + 9 * layer + LAYER_TENSORS.index(name)


# ----------------------------------------------------------------------------
# seeded draws
# ----------------------------------------------------------------------------

_CHUNK = 1 << 22
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = _cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1))
    return _POOL


def normal_f32(seed: int, tid: int, n: int) -> np.ndarray:
    """n standard normals (float32), chunked streams so threads may fill them."""
    out = np.empty(n, dtype=np.float32)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, c])))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        list(_pool().map(fill, range(nchunks)))
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Tensor:
    """A generated weight: `stored` is what a device copy holds (float32 values or
    bf16 bit patterns), `values` the same numbers widened to float32."""

    stored: np.ndarray
    values: np.ndarray


def _chunked(n: int, fn):
    """Runs fn(lo, hi, chunk_index) over 4 Mi-element chunks, in threads."""
    nchunks = (n + _CHUNK - 1) // _CHUNK
    jobs = [(c * _CHUNK, min(n, (c + 1) * _CHUNK), c) for c in range(nchunks)]
    if nchunks <= 1:
        for j in jobs:
            fn(*j)
    else:
        list(_pool().map(lambda j: fn(*j), jobs))


def weight(s: ModelShape, name: str, layer: int = -1, seed: int = 0,
           scale: float = 0.02, gain_scale: float = 0.0) -> Tensor:
    shape = tensor_shape(s, name)
    n = int(np.prod(shape))
    tid = tensor_id(s, name, layer)
    is_norm = name.endswith("norm")
    bf16 = s.weight_dtype == "bf16"
    assert bf16 or s.weight_dtype == "f32"
    values = np.empty(n, dtype=np.float32)
    stored = np.empty(n, dtype=np.uint16) if bf16 else values

    def fill(lo, hi, c):
        if is_norm and gain_scale <= 0:
            v = np.ones(hi - lo, dtype=np.float32)
        else:
            g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, c])))
            v = g.standard_normal(hi - lo, dtype=np.float32)
            if is_norm:
                v = np.float32(1.0) + v * np.float32(gain_scale)
            else:
                v *= np.float32(scale)
        if bf16:
            b = bf16_bits(v)
            stored[lo:hi] = b
            values[lo:hi] = bf16_to_f32(b)
        else:
            values[lo:hi] = v

    _chunked(n, fill)
    return Tensor(stored=stored.reshape(shape), values=values.reshape(shape))


def logit_rows(rows: int, vocab: int, seed: int, scale: float = 3.0, ties: int = 0, neg_inf: int = 0,
               nan: int = 0) -> np.ndarray:
    """Synthetic fp32 logit rows [rows, vocab], N(0, scale^2) per entry; in each
    row `ties` more entries copy the row's largest value and `neg_inf` / `nan`
    entries are set to -inf / NaN (their positions drawn from the same seed)."""
    out = normal_f32(seed, 9, rows * vocab).reshape(rows, vocab) * np.float32(scale)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 10])))
    for r in range(rows):
        pick = g.permutation(vocab)[:ties + neg_inf + nan]
        out[r, pick[:ties]] = out[r].max()
        out[r, pick[ties:ties + neg_inf]] = -np.inf
        out[r, pick[ties + neg_inf:]] = np.nan
    return out.astype(np.float32)


def prompt_ids(vocab: int, n: int, seed: int = 1) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    return g.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def kv_fill_f16(shape: tuple, seed: int = 2) -> np.ndarray:
    """Pre-filled KV rows: N(0,1) rounded to fp16."""
    n = int(np.prod(shape))
    return normal_f32(seed, 0, n).astype(np.float16).reshape(shape)


def hidden_f32(n: int, seed: int = 3) -> np.ndarray:
    """An N(0,1) hidden-state vector for the layer-only workload."""
    return normal_f32(seed, 0, n)
