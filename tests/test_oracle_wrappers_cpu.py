"""Pins of the oracle's entry points that wrap its pinned core:

  * layer_decode_step (one layer for one new token over a given cache prefix)
    reproduces the residual and the stored K/V row of a full-prefix pass of a
    1-layer model at that position;
  * fp8_weights / q4_weights touch only the Linear weights (the projections
    and the lm_head: k2-burn README, "Quantization"), and what they return is
    a representable code times its scale within half a quantization step;
  * generate_sampled with top-k = 1 is greedy decoding, whatever the
    temperature and seed (k2-burn README, "Sampling + greedy generation").
"""
import numpy as np
import pytest

import k2_inputs as ki
from oracle import k2_fp8 as Q8
from oracle import k2_oracle as O
from oracle import k2_q4 as Q4
from oracle import k2_sampling as S

F32 = np.float32
LAYER_NAMES = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


def tiny_weights(shape, seed):
    rng = np.random.default_rng(seed)
    H, d, I, V = shape.hidden, shape.head_dim, shape.intermediate, shape.vocab
    dims = {"wq": (shape.n_heads * d, H), "wk": (shape.n_kv_heads * d, H), "wv": (shape.n_kv_heads * d, H),
            "wo": (H, shape.n_heads * d), "w_gate": (I, H), "w_up": (I, H), "w_down": (H, I),
            "embed": (V, H), "lm_head": (V, H)}
    w = {}
    for name, dim in dims.items():
        w[name] = (rng.standard_normal(dim) * 0.05).astype(F32)
    for name in ("attn_norm", "mlp_norm", "final_norm"):
        w[name] = (1.0 + 0.1 * rng.standard_normal(H)).astype(F32)
    return w


@pytest.mark.parametrize("pos", [0, 1, 7])
def test_layer_decode_step_is_the_full_prefix_pass(pos):
    s = ki.TINY.replace(n_layers=1)
    w = tiny_weights(s, 21)
    model = O.OracleModel(s, lambda n, l: w[n], "f32")
    toks = np.random.default_rng(22).integers(0, s.vocab, pos + 1)
    cache = model.new_cache(pos + 1)
    x_full, _ = model.run(toks, cache, logits_rows=None)
    x_in = w["embed"][toks[pos]].astype(np.float64)
    x_out, k_row, v_row = O.layer_decode_step(s, {n: w[n] for n in LAYER_NAMES}, x_in, pos,
                                              cache.k[0][:pos], cache.v[0][:pos], "f32")
    np.testing.assert_allclose(x_out, x_full[pos], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(k_row, cache.k[0][pos])
    np.testing.assert_array_equal(v_row, cache.v[0][pos])


def check_wrapper(wrap, representable):
    s = ki.TINY
    w = tiny_weights(s, 23)
    get = wrap(lambda n, l: w[n])
    for name in ("embed", "attn_norm", "mlp_norm", "final_norm"):
        assert get(name, 0) is w[name]  # passed through untouched
    for name in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "lm_head"):
        q = np.asarray(get(name, 0), dtype=np.float64)
        assert q.shape == w[name].shape and not np.array_equal(q, w[name].astype(np.float64))
        representable(w[name].astype(np.float64), q)
        assert get(name, 0) is get(name, 0)  # quantized once


def test_fp8_wrapper_quantizes_only_the_linear_weights():
    finite = Q8.E4M3_VALUES[~np.isnan(Q8.E4M3_VALUES)]

    def representable(w, q):
        s = np.max(np.abs(w), axis=1) / 448.0  # the row scale, up to float32 rounding
        for r in range(w.shape[0]):
            code = q[r] / s[r]
            nearest = finite[np.argmin(np.abs(code[:, None] - finite[None, :]), axis=1)]
            assert np.allclose(code, nearest, rtol=1e-6, atol=0)
            step = np.maximum(np.abs(nearest) * 2.0 ** -3, 2.0 ** -9)  # an E4M3 step at that value
            assert np.all(np.abs(w[r] - q[r]) <= step * s[r] * (0.5 + 1e-6))

    check_wrapper(Q8.fp8_weights, representable)


def test_int4_wrapper_quantizes_only_the_linear_weights():
    def representable(w, q):
        rows, cols = w.shape
        for b in range(0, cols, 64):
            s = np.max(np.abs(w[:, b:b + 64]), axis=1) / 7.0
            code = q[:, b:b + 64] / s[:, None]
            assert np.allclose(code, np.rint(code), rtol=0, atol=1e-5) and np.all(np.abs(code) <= 7 + 1e-5)
            assert np.all(np.abs(w[:, b:b + 64] - q[:, b:b + 64]) <= s[:, None] * (0.5 + 1e-5))

    check_wrapper(Q4.q4_weights, representable)


@pytest.mark.parametrize("temperature,seed", [(0.7, 1), (1.5, 2), (3.0, 3)])
def test_sampling_with_top_k_one_is_greedy_decoding(temperature, seed):
    s = ki.TINY
    w = tiny_weights(s, 24)
    model = O.OracleModel(s, lambda n, l: w[n], "f32")
    prompt = np.random.default_rng(25).integers(0, s.vocab, 6)
    greedy, _ = model.generate_greedy(prompt, 5, capacity=16)
    sampled = S.generate_sampled(model, prompt, 5, {"temperature": temperature, "top_k": 1, "seed": seed},
                                 capacity=16)
    assert sampled.tolist() == greedy.tolist()
