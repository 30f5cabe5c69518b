"""CPU oracle for the K2-Horizon dense GQA decoder forward step.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline / reference legs of
``bench.py``; nothing on the product path imports, links or runs it, and it
imports nothing from the CUDA package.  It shares no code with the kernels:
only the seeded input generator module (``k2_inputs``) serves both sides.

What it computes is written from the pages' statement of the model:
  * k2-burn README, "Status: v0": GroupedRMSNorm, split-half RoPE, GQA
    attention, SwiGLU MLP; a preallocated per-layer KV cache, prefill then
    single-token decode; temperature 0 = greedy argmax.
  * k2-burn README, "Model shape": hidden 2560, 36 layers, 32 q heads over
    8 KV heads (4x repeat), head_dim 128, intermediate 10240, 2 norm groups,
    vocab 250624, eps 1e-6, untied lm_head.
  * k2-burn README, "Limitations": plain SDPA (matmul + softmax); the page
    upcasts the softmax to fp32 -- here every step is float64.
  * k2-burn README, "KV cache storage": KV stored as the activation dtype,
    f16, or symmetric int8 with per-block scales.
  * k2-burn README, "Project layout": layer.rs is "norm+attn residual,
    norm+mlp residual"; model.rs is "embed -> layers -> norm -> lm_head".
  * kimi-k3-in-c, k3_run.c, ``argmax_``: the first index of the maximum wins.
  * kimi-k3-in-c, k3_run.c, header "DECODE STRATEGY": incremental decode must
    give the same tokens as full-prefix recompute (its GATE 3).

Precision: float64 arithmetic throughout.  The only roundings are the storage
roundings the method itself defines -- weights stored as bf16 (given as
inputs) and K/V rows stored as fp32, fp16 or int8+fp16 scale (``store_kv``).
The int8 quantiser takes its rounding decisions in float32, the precision the
CUDA kernels use for the same decision.

Readings where the pages are silent:
  * GroupedRMSNorm: the hidden vector is split into ``groups`` contiguous
    equal groups; each group is divided by sqrt(mean(x_g^2) + eps); the result
    is multiplied by one full-length gain.  No mean subtraction, no bias.  All
    three norms (input, post-attention, final) are grouped.
  * RoPE: split-half ("rotate_half") pairs element i with i + d/2;
    theta_i = theta^(-2i/d); absolute 0-based positions; K is cached after
    RoPE, V is not rotated.
  * GQA: query head h reads KV head floor(h / (n_heads / n_kv_heads)).
  * Attention: scale 1/sqrt(head_dim), causal, no soft-cap, no bias.
  * int8 KV: one fp16 scale per (token, KV head, K or V) over head_dim values:
    s = fp16(amax / 127) (clamped to the largest finite fp16), code =
    clamp(rne(u / s), -127, 127); s == 0 gives code 0.
  * No biases anywhere.

Pins: tests/test_oracle_pins.py checks every function here against closed
forms, library routines it reduces to, brute force, and invariants.
"""
from __future__ import annotations

import math
from typing import Callable, Dict, Optional

import numpy as np

F64 = np.float64

MUTANTS = (
    None,
    "skip_last_layer",      # a decoder layer is skipped
    "head_map_modulo",      # q head h reads KV head h % n_kv instead of h // rep
    "rope_interleaved",     # RoPE pairs (2i, 2i+1) instead of (i, i+d/2)
    "one_norm_group",       # plain RMSNorm instead of grouped
    "no_attn_scale",        # the 1/sqrt(d) is dropped
    "attend_excludes_self", # the newly appended KV row is not attended to
    "k_pos_shift",          # K rotated one position ahead of Q
    "swiglu_swapped",       # silu applied to the up branch instead of the gate
    "no_silu",              # the gate branch enters the product without silu
)


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------

def grouped_rms_norm(x, gain, groups: int, eps: float):
    """GroupedRMSNorm (k2-burn README, "Status: v0" and "Model shape":
    layernorm_num_groups, rms_norm_eps).

    x: [..., H]; gain: [H].  y_g = x_g / sqrt(mean(x_g^2) + eps), then y * gain.
    """
    x = np.asarray(x, dtype=F64)
    H = x.shape[-1]
    assert H % groups == 0
    xg = x.reshape(x.shape[:-1] + (groups, H // groups))
    ms = np.mean(xg * xg, axis=-1, keepdims=True)
    y = (xg / np.sqrt(ms + eps)).reshape(x.shape)
    return y * np.asarray(gain, dtype=F64)


def rope_inv_freq(head_dim: int, theta: float):
    """theta_i = theta^(-2i/d), i in [0, d/2)  (RoPE "default" type, k2-burn
    README, "Status: v0", RoPE scaling)."""
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(theta), -2.0 * i / head_dim)


def rope_split_half(u, positions, theta: float, interleaved: bool = False):
    """Split-half rotary embedding (k2-burn README, "Status: v0").

    u: [T, n_heads, d]; positions: [T] absolute positions.  For i < d/2 with
    a = u[i], b = u[i + d/2], phi = pos * theta_i:
        u[i] <- a cos(phi) - b sin(phi),   u[i + d/2] <- b cos(phi) + a sin(phi).
    ``interleaved`` is the planted mutant pairing (2i, 2i+1).
    """
    u = np.asarray(u, dtype=F64)
    d = u.shape[-1]
    half = d // 2
    ang = np.asarray(positions, dtype=F64)[:, None] * rope_inv_freq(d, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if interleaved:
        a, b = u[..., 0::2], u[..., 1::2]
        out = np.empty_like(u)
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = b * c + a * s
        return out
    a, b = u[..., :half], u[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


FP16_MAX = 65504.0


def int8_quantize(u):
    """Symmetric int8 with one fp16 scale per row over the last axis
    (k2-burn README, "KV cache storage", int8).

    Decisions are taken in float32:  s = fp16(fp32(amax) / 127), clamped to the
    largest finite fp16;  code = clamp(rne(fp32(u) / s), -127, 127);  s == 0
    gives code 0.  Returns (codes int8 [..., d], scales float16 [...]).
    """
    u32 = np.asarray(u, dtype=np.float32)
    amax = np.max(np.abs(u32), axis=-1)
    s32 = (amax / np.float32(127.0)).astype(np.float32)
    s32 = np.minimum(s32, np.float32(FP16_MAX))
    s16 = s32.astype(np.float16)
    sw = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.where(sw > 0, u32 / np.where(sw > 0, sw, np.float32(1)), np.float32(0))
    codes = np.clip(np.rint(qf), -127, 127).astype(np.int8)
    return codes, s16


def int8_dequantize(codes, scales):
    return np.asarray(codes, dtype=F64) * np.asarray(scales, dtype=F64)[..., None]


def store_kv(u, kv_dtype: str):
    """What a KV row reads back as after it was stored (k2-burn README,
    "KV cache storage": full | f16 | int8).  u: [T, n_kv, d] float64."""
    if kv_dtype == "f32":
        return np.asarray(u, dtype=np.float32).astype(F64)
    if kv_dtype == "f16":
        return np.asarray(u, dtype=np.float16).astype(F64)
    if kv_dtype == "i8":
        codes, scales = int8_quantize(u)
        return int8_dequantize(codes, scales)
    raise ValueError(f"kv dtype {kv_dtype!r}")


def gqa_attention(q, k, v, q_positions, scale: Optional[float] = None,
                  head_map_modulo: bool = False, exclude_self: bool = False):
    """Causal grouped-query attention, plain SDPA (k2-burn README,
    "Limitations": matmul + softmax, no flash attention).

    q: [T, nq, d] at absolute positions q_positions [T]; k, v: [L, nkv, d]
    holding positions 0..L-1.  Query at position p sees keys j <= p.
    Query head h reads KV head h // (nq / nkv).
    Returns [T, nq, d].
    """
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    T, nq, d = q.shape
    L, nkv, _ = k.shape
    rep = nq // nkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    heads = np.arange(nq)
    kvh = heads % nkv if head_map_modulo else heads // rep
    kk = k[:, kvh, :]  # [L, nq, d]
    vv = v[:, kvh, :]
    s = np.einsum("thd,lhd->htl", q, kk) * scale  # [nq, T, L]
    pos = np.asarray(q_positions)[:, None]
    j = np.arange(L)[None, :]
    # the mutant drops the newest row (position 0 keeps its only row)
    visible = (j < np.maximum(pos, 1)) if exclude_self else (j <= pos)
    s = np.where(visible[None, :, :], s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    p = np.exp(s - m)
    p = p / np.sum(p, axis=-1, keepdims=True)
    return np.einsum("htl,lhd->thd", p, vv)


def silu(z):
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def argmax_first(logits) -> int:
    """Greedy token: the first index of the maximum (kimi-k3-in-c, k3_run.c,
    ``argmax_`` uses a strict ``>`` scan, so ties go to the lowest index)."""
    logits = np.asarray(logits)
    if np.isnan(logits).any():
        raise ValueError("NaN logit")
    # np.argmax returns the first occurrence of the maximum, which is what a
    # strict-greater scan from index 0 returns.
    return int(np.argmax(logits))


# ---------------------------------------------------------------------------
# the model
# ---------------------------------------------------------------------------

WeightGetter = Callable[[str, int], np.ndarray]


class KVCache:
    """Per-layer preallocated cache of stored (read-back) K and V rows
    (k2-burn README, "KV cache storage": preallocated to --context)."""

    def __init__(self, n_layers, capacity, n_kv, head_dim):
        self.k = [np.zeros((capacity, n_kv, head_dim), dtype=F64) for _ in range(n_layers)]
        self.v = [np.zeros((capacity, n_kv, head_dim), dtype=F64) for _ in range(n_layers)]
        self.length = 0
        self.capacity = capacity


class OracleModel:
    """The dense GQA decoder: embed -> layers -> final norm -> lm_head
    (k2-burn README, "Project layout", model.rs; untied lm_head per
    "Model shape").

    ``get(name, layer)`` returns a weight as float32/float64 values in the
    nn.Linear [out, in] layout; names: embed, lm_head, final_norm and per
    layer attn_norm, wq, wk, wv, wo, mlp_norm, w_gate, w_up, w_down.
    """

    def __init__(self, shape, get: WeightGetter, kv_dtype: str, mutant: Optional[str] = None):
        assert mutant in MUTANTS, mutant
        self.s = shape
        self.get = get
        self.kv_dtype = kv_dtype
        self.mutant = mutant
        assert shape.n_heads % shape.n_kv_heads == 0
        assert shape.head_dim % 2 == 0

    def _w(self, name, layer=-1):
        return np.asarray(self.get(name, layer), dtype=F64)

    def _norm(self, x, gain):
        groups = 1 if self.mutant == "one_norm_group" else self.s.norm_groups
        return grouped_rms_norm(x, gain, groups, self.s.eps)

    def layer(self, l: int, x, positions, cache: KVCache):
        """One decoder layer over rows x [T, H] at absolute positions
        (k2-burn README, "Project layout", layer.rs: norm+attn residual,
        norm+mlp residual).  Appends the rows' K/V to ``cache`` and attends
        causally over everything cached so far."""
        s = self.s
        T = x.shape[0]
        d = s.head_dim
        positions = np.asarray(positions)
        if self.mutant == "skip_last_layer" and l == s.n_layers - 1:
            for p in positions:
                cache.k[l][p] = 0.0
                cache.v[l][p] = 0.0
            return x
        xn = self._norm(x, self._w("attn_norm", l))
        q = (xn @ self._w("wq", l).T).reshape(T, s.n_heads, d)
        k = (xn @ self._w("wk", l).T).reshape(T, s.n_kv_heads, d)
        v = (xn @ self._w("wv", l).T).reshape(T, s.n_kv_heads, d)
        inter = self.mutant == "rope_interleaved"
        q = rope_split_half(q, positions, s.rope_theta, interleaved=inter)
        kpos = positions + 1 if self.mutant == "k_pos_shift" else positions
        k = rope_split_half(k, kpos, s.rope_theta, interleaved=inter)
        cache.k[l][positions] = store_kv(k, self.kv_dtype)
        cache.v[l][positions] = store_kv(v, self.kv_dtype)
        L = int(positions.max()) + 1
        attn = gqa_attention(
            q, cache.k[l][:L], cache.v[l][:L], positions,
            scale=1.0 if self.mutant == "no_attn_scale" else None,
            head_map_modulo=self.mutant == "head_map_modulo",
            exclude_self=self.mutant == "attend_excludes_self")
        x = x + attn.reshape(T, s.n_heads * d) @ self._w("wo", l).T
        xn = self._norm(x, self._w("mlp_norm", l))
        g = xn @ self._w("w_gate", l).T
        u = xn @ self._w("w_up", l).T
        if self.mutant == "swiglu_swapped":
            g, u = u, g
        a = (g if self.mutant == "no_silu" else silu(g)) * u
        return x + a @ self._w("w_down", l).T

    def embed(self, tokens):
        E = self.get("embed", -1)
        return np.asarray(E[np.asarray(tokens)], dtype=F64)

    def head(self, x, chunk: int = 32768):
        """Final GroupedRMSNorm then the untied lm_head; x [T, H] -> logits [T, V]."""
        xn = self._norm(x, self._w("final_norm"))
        W = self.get("lm_head", -1)
        V = W.shape[0]
        out = np.empty((xn.shape[0], V), dtype=F64)
        for lo in range(0, V, chunk):
            out[:, lo:lo + chunk] = xn @ np.asarray(W[lo:lo + chunk], dtype=F64).T
        return out

    # -- sequence-level entry points ------------------------------------------

    def new_cache(self, capacity: int) -> KVCache:
        s = self.s
        return KVCache(s.n_layers, capacity, s.n_kv_heads, s.head_dim)

    def run(self, tokens, cache: KVCache, logits_rows=("last",)):
        """Append ``tokens`` at positions cache.length.. and run them through
        every layer.  Returns (final residual rows [T, H], logits of the rows
        asked for).  With a fresh cache this is full-prefix recompute; called
        one token at a time it is incremental decode."""
        tokens = np.asarray(tokens)
        T = tokens.shape[0]
        if cache.length + T > cache.capacity:
            raise ValueError("context full")  # rejected, not truncated (README, "KV cache storage")
        positions = np.arange(cache.length, cache.length + T)
        x = self.embed(tokens)
        for l in range(self.s.n_layers):
            x = self.layer(l, x, positions, cache)
        cache.length += T
        if logits_rows == ("last",):
            rows = [T - 1]
        elif logits_rows is None:
            rows = []
        else:
            rows = list(logits_rows)
        logits = self.head(x[rows]) if rows else None
        return x, logits

    def forward_full(self, tokens):
        """Full-prefix recompute: logits of the last position only
        (kimi-k3-in-c, k3_run.c, ``forward`` returns last-position logits)."""
        cache = self.new_cache(len(tokens))
        _, logits = self.run(tokens, cache)
        return logits[0]

    def generate_greedy(self, prompt, n_new: int, capacity: Optional[int] = None):
        """Prefill the prompt, then ``n_new`` single-token decode steps
        (k2-burn README, "Status: v0": prefill + single-token decode;
        temperature 0 = greedy argmax).  The first new token comes from the
        prefill; each decode step consumes the previous token.  Returns
        (tokens [n_new + 1], logits per emitted token [n_new + 1, V])."""
        cap = capacity or (len(prompt) + n_new)
        cache = self.new_cache(cap)
        _, lg = self.run(prompt, cache)
        toks = [argmax_first(lg[0])]
        all_logits = [lg[0]]
        for _ in range(n_new):
            _, lg = self.run([toks[-1]], cache)
            toks.append(argmax_first(lg[0]))
            all_logits.append(lg[0])
        return np.array(toks, dtype=np.int64), np.stack(all_logits)

    def teacher_forced(self, seq, first_row: int):
        """One causal pass over ``seq``; returns (argmax, logits, final residual)
        for rows first_row..T-1 (kimi-k3-in-c, k3_run.c, --tf-check: prediction
        i is the argmax after tokens 0..i)."""
        cache = self.new_cache(len(seq))
        rows = list(range(first_row, len(seq)))
        x, logits = self.run(seq, cache, logits_rows=rows)
        am = np.array([argmax_first(r) for r in logits], dtype=np.int64)
        return am, logits, x[rows]


# ---------------------------------------------------------------------------
# a single decoder layer on a given hidden state against a given cache
# ---------------------------------------------------------------------------

def layer_decode_step(shape, w: Dict[str, np.ndarray], x, pos: int, k_prefix, v_prefix,
                      kv_dtype: str):
    """One decoder layer for one new token at position ``pos``, reading a cache
    whose rows 0..pos-1 hold ``k_prefix``/``v_prefix`` [pos, nkv, d] (already
    stored values).  Returns (x_out [H], stored k row, stored v row)."""
    m = OracleModel(shape.replace(n_layers=1), lambda n, l: w[n], kv_dtype)
    cache = m.new_cache(pos + 1)
    cache.k[0][:pos] = k_prefix
    cache.v[0][:pos] = v_prefix
    y = m.layer(0, np.asarray(x, dtype=F64)[None, :], np.array([pos]), cache)
    return y[0], cache.k[0][pos], cache.v[0][pos]
