"""Pins of the CPU oracle against things other than itself: closed forms,
library routines the definitions reduce to, pure-Python brute force on tiny
inputs, and invariants.  Each test names the mistake it is there to catch.
No GPU is used."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import k2_inputs as ki
from oracle import k2_oracle as O

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------------------
# GroupedRMSNorm
# ---------------------------------------------------------------------------

def test_grouped_norm_groups_have_unit_rms_closed_form():
    # gain 1: each group's output RMS is exactly sqrt(ms / (ms + eps))
    x = RNG.standard_normal((5, 64)) * 3.0
    eps = 1e-6
    y = O.grouped_rms_norm(x, np.ones(64), 2, eps)
    for g in range(2):
        xs, ys = x[:, 32 * g:32 * (g + 1)], y[:, 32 * g:32 * (g + 1)]
        ms = np.mean(xs ** 2, axis=-1)
        np.testing.assert_allclose(np.sqrt(np.mean(ys ** 2, axis=-1)), np.sqrt(ms / (ms + eps)), rtol=1e-12)
        # and before eps it is 1 to within the eps correction
        np.testing.assert_allclose(np.sqrt(np.mean(ys ** 2, axis=-1)), 1.0, atol=1e-6)


def test_grouped_norm_one_group_is_library_rms_norm():
    x = RNG.standard_normal((3, 48))
    w = RNG.standard_normal(48)
    ref = F.rms_norm(torch.tensor(x), (48,), torch.tensor(w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.grouped_rms_norm(x, w, 1, 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_grouped_norm_groups_are_contiguous_halves():
    # two groups = library rms_norm applied to each contiguous half on its own
    x = RNG.standard_normal((4, 40))
    x[:, 20:] *= 50.0  # very different group scales: interleaved groups would fail
    w = RNG.standard_normal(40)
    ref = np.concatenate([
        F.rms_norm(torch.tensor(x[:, :20]), (20,), torch.tensor(w[:20]), eps=1e-6).numpy(),
        F.rms_norm(torch.tensor(x[:, 20:]), (20,), torch.tensor(w[20:]), eps=1e-6).numpy()], axis=-1)
    np.testing.assert_allclose(O.grouped_rms_norm(x, w, 2, 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_grouped_norm_scale_invariant():
    x = RNG.standard_normal((2, 32))
    a = O.grouped_rms_norm(x, np.ones(32), 2, 1e-6)
    b = O.grouped_rms_norm(1000.0 * x, np.ones(32), 2, 1e-6)
    np.testing.assert_allclose(a, b, rtol=1e-5)


# ---------------------------------------------------------------------------
# split-half RoPE
# ---------------------------------------------------------------------------

def test_rope_hand_example():
    # d=4, theta=10000, pos=1: theta_0 = 1, theta_1 = 0.01.  Element 0 pairs
    # with element 2 (split half), rotated by +1 rad.
    u = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    out = O.rope_split_half(u, np.array([1]), 10000.0)[0, 0]
    np.testing.assert_allclose(out, [math.cos(1.0), 0.0, math.sin(1.0), 0.0], atol=1e-15)
    u = np.array([[[0.0, 1.0, 0.0, 0.0]]])
    out = O.rope_split_half(u, np.array([3]), 10000.0)[0, 0]
    np.testing.assert_allclose(out, [0.0, math.cos(0.03), 0.0, math.sin(0.03)], atol=1e-15)


def test_rope_matches_rotate_half_textbook_form():
    # q*cos + rotate_half(q)*sin with rotate_half(q) = cat(-q2, q1) and the
    # angle table duplicated over both halves
    d = 16
    u = RNG.standard_normal((7, 3, d))
    pos = RNG.integers(0, 5000, size=7)
    inv = 1.0 / (10000.0 ** (np.arange(0, d, 2) / d))
    ang = pos[:, None] * inv[None, :]
    emb = np.concatenate([ang, ang], axis=-1)[:, None, :]
    rot = np.concatenate([-u[..., d // 2:], u[..., :d // 2]], axis=-1)
    ref = u * np.cos(emb) + rot * np.sin(emb)
    np.testing.assert_allclose(O.rope_split_half(u, pos, 10000.0), ref, rtol=1e-12, atol=1e-12)


def test_rope_invariants():
    d = 128
    q = RNG.standard_normal((1, 1, d))
    k = RNG.standard_normal((1, 1, d))
    # position 0 is the identity
    np.testing.assert_allclose(O.rope_split_half(q, np.array([0]), 1e4), q, atol=0)
    # norm preserved
    r = O.rope_split_half(q, np.array([4097]), 1e4)
    np.testing.assert_allclose(np.linalg.norm(r), np.linalg.norm(q), rtol=1e-12)
    # <R_m q, R_n k> depends only on m - n
    def dot(m, n):
        return float(np.sum(O.rope_split_half(q, np.array([m]), 1e4) * O.rope_split_half(k, np.array([n]), 1e4)))
    for (m, n, dm) in [(7, 3, 100), (30000, 2, 17), (5, 5, 999)]:
        assert abs(dot(m, n) - dot(m + dm, n + dm)) < 1e-9
    assert abs(dot(7, 3) - dot(3, 7)) > 1e-3  # and it is not symmetric (sign of sin matters)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _brute_attention(q, k, v, q_positions):
    T, nq, d = q.shape
    L, nkv, _ = k.shape
    rep = nq // nkv
    out = np.zeros_like(q)
    for t in range(T):
        for h in range(nq):
            g = h // rep
            ss = []
            for j in range(q_positions[t] + 1):
                ss.append(sum(q[t, h, i] * k[j, g, i] for i in range(d)) / math.sqrt(d))
            m = max(ss)
            e = [math.exp(s - m) for s in ss]
            z = sum(e)
            for i in range(d):
                out[t, h, i] = sum(e[j] / z * v[j, g, i] for j in range(len(e)))
    return out


def test_attention_brute_force_gqa():
    nq, nkv, d, L = 4, 2, 8, 9
    q = RNG.standard_normal((3, nq, d))
    k = RNG.standard_normal((L, nkv, d))
    v = RNG.standard_normal((L, nkv, d))
    pos = np.array([0, 4, 8])
    np.testing.assert_allclose(O.gqa_attention(q, k, v, pos), _brute_attention(q, k, v, pos), rtol=1e-11, atol=1e-12)


def test_attention_is_library_sdpa_causal_gqa():
    T, nq, nkv, d = 13, 8, 2, 16
    q = RNG.standard_normal((T, nq, d))
    k = RNG.standard_normal((T, nkv, d))
    v = RNG.standard_normal((T, nkv, d))
    ref = F.scaled_dot_product_attention(
        torch.tensor(q).transpose(0, 1), torch.tensor(k).transpose(0, 1), torch.tensor(v).transpose(0, 1),
        is_causal=True, enable_gqa=True).transpose(0, 1).numpy()
    np.testing.assert_allclose(O.gqa_attention(q, k, v, np.arange(T)), ref, rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    q = RNG.standard_normal((1, 4, 8))
    k = RNG.standard_normal((1, 2, 8))
    v = RNG.standard_normal((1, 2, 8))
    # one key: the output is that key's value row
    o = O.gqa_attention(q, k, v, np.array([0]))
    np.testing.assert_allclose(o[0], v[0, [0, 0, 1, 1]], rtol=1e-14)
    # constant V rows: the weights sum to one, so the output is that constant
    k = RNG.standard_normal((20, 2, 8))
    v = np.full((20, 2, 8), 3.25)
    o = O.gqa_attention(RNG.standard_normal((2, 4, 8)), k, v, np.array([5, 19]))
    np.testing.assert_allclose(o, 3.25, rtol=1e-13)
    # the decode row equals the last row of the full causal pass
    T = 11
    q = RNG.standard_normal((T, 4, 8))
    k = RNG.standard_normal((T, 2, 8))
    v = RNG.standard_normal((T, 2, 8))
    full = O.gqa_attention(q, k, v, np.arange(T))
    dec = O.gqa_attention(q[-1:], k, v, np.array([T - 1]))
    np.testing.assert_allclose(dec[0], full[-1], rtol=1e-13)


# ---------------------------------------------------------------------------
# SwiGLU, storage, argmax
# ---------------------------------------------------------------------------

def test_silu_is_library():
    z = RNG.standard_normal(100) * 10
    np.testing.assert_allclose(O.silu(z), F.silu(torch.tensor(z)).numpy(), rtol=1e-13)
    assert O.silu(0.0) == 0.0


def test_int8_quant_hand_example_and_bound():
    u = np.zeros((1, 1, 8))
    u[0, 0, :4] = [127.0, -63.5, 0.4, 64.5]
    codes, s = O.int8_quantize(u)
    assert float(s[0, 0]) == 1.0
    # round half to even: -63.5 -> -64, 64.5 -> 64
    assert codes[0, 0, :4].tolist() == [127, -64, 0, 64]
    # zero row: scale 0, all codes 0
    c0, s0 = O.int8_quantize(np.zeros((2, 16)))
    assert np.all(c0 == 0) and np.all(s0 == 0)
    x = RNG.standard_normal((50, 3, 128)) * 4
    codes, s = O.int8_quantize(x)
    deq = O.int8_dequantize(codes, s)
    sf = s.astype(np.float64)[..., None]
    assert np.all(np.abs(x.astype(np.float32) - deq) <= sf / 2 * (1 + 1e-6) + 1e-12)
    # the largest magnitude of each row maps to +-127
    idx = np.argmax(np.abs(x), axis=-1)
    top = np.take_along_axis(codes, idx[..., None], -1)[..., 0]
    assert np.all(np.abs(top) == 127)


def test_store_kv_roundings():
    u = np.array([[[1.0, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 65504.0]]])
    # fp16 has 10 fraction bits: 1 + 2^-11 is a tie -> even (1.0); 1 + 3*2^-11 -> 1 + 2^-9
    np.testing.assert_array_equal(O.store_kv(u, "f16"), [[[1.0, 1.0, 1.0 + 2 ** -9, 65504.0]]])
    np.testing.assert_array_equal(O.store_kv(np.array([[[0.1]]]), "f32"), [[[float(np.float32(0.1))]]])


def test_argmax_first_index_on_ties():
    for _ in range(50):
        v = RNG.integers(0, 4, size=37).astype(np.float64)
        best = 0
        for i in range(1, len(v)):  # the strict-greater scan
            if v[i] > v[best]:
                best = i
        assert O.argmax_first(v) == best
    with pytest.raises(ValueError):
        O.argmax_first(np.array([0.0, np.nan]))


def test_bf16_input_rounding_is_library():
    x = (RNG.standard_normal(10000) * 0.02).astype(np.float32)
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ki.bf16_bits(x), ref)


# ---------------------------------------------------------------------------
# whole model
# ---------------------------------------------------------------------------

def _tiny(kv="f32", mutant=None, **shape_kw):
    s = ki.TINY.replace(**shape_kw)
    cache = {}

    def get(n, l):
        if (n, l) not in cache:
            cache[(n, l)] = ki.weight(s, n, l, gain_scale=0.0).values
        return cache[(n, l)]
    return s, O.OracleModel(s, get, kv, mutant=mutant), get


@pytest.mark.parametrize("kv", ["f32", "f16", "i8"])
def test_gate3_incremental_equals_full_recompute(kv):
    # kimi-k3-in-c GATE 3: incremental decode gives the same tokens as
    # full-prefix recompute (and, here, the same logits to rounding)
    s, m, _ = _tiny(kv)
    prompt = ki.prompt_ids(s.vocab, 16)
    toks, logits = m.generate_greedy(prompt, 16)
    seq = np.concatenate([prompt, toks])
    for i in range(len(toks)):
        full = m.forward_full(seq[:16 + i])
        np.testing.assert_allclose(full, logits[i], rtol=0, atol=1e-10)
        assert O.argmax_first(full) == toks[i]
    # teacher-forced pass over the emitted sequence reproduces the tokens
    am, _, _ = m.teacher_forced(seq[:-1], 15)
    np.testing.assert_array_equal(am, toks)


def test_residual_path_closed_form():
    # with o_proj and down_proj zero every layer is the identity on the
    # residual stream: logits = lm_head . final_norm(embed[token])
    s, _, get = _tiny()

    def get0(n, l):
        if n in ("wo", "w_down"):
            return np.zeros(ki.tensor_shape(s, n))
        return get(n, l)
    m = O.OracleModel(s, get0, "f32")
    prompt = ki.prompt_ids(s.vocab, 5)
    lg = m.forward_full(prompt)
    x = get("embed", -1)[prompt[-1]].astype(np.float64)
    ms = [np.mean(x[:32] ** 2), np.mean(x[32:] ** 2)]
    xn = np.concatenate([x[:32] / math.sqrt(ms[0] + 1e-6), x[32:] / math.sqrt(ms[1] + 1e-6)])
    ref = get("lm_head", -1).astype(np.float64) @ xn
    np.testing.assert_allclose(lg, ref, rtol=1e-12, atol=1e-14)


def test_uniform_attention_closed_form():
    # Wq = 0 makes every score 0, so the attention output at position p is the
    # mean of the stored V rows 0..p.  With o_proj = identity and the MLP
    # removed, one layer adds exactly that mean to the residual.
    s = ki.TINY.replace(n_layers=1, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16)
    base = {}

    def get(n, l):
        if n == "wq":
            return np.zeros(ki.tensor_shape(s, n))
        if n == "wo":
            return np.eye(64)
        if n == "w_down":
            return np.zeros(ki.tensor_shape(s, n))
        if (n, l) not in base:
            base[(n, l)] = ki.weight(s, n, l).values
        return base[(n, l)]
    m = O.OracleModel(s, get, "f32")
    toks = ki.prompt_ids(s.vocab, 6)
    cache = m.new_cache(6)
    x, _ = m.run(toks, cache, logits_rows=None)
    E = get("embed", -1)[toks].astype(np.float64)
    xn = np.stack([O.grouped_rms_norm(e, np.ones(64), 2, 1e-6) for e in E])
    vrows = (xn @ get("wv", 0).astype(np.float64).T).astype(np.float32).astype(np.float64).reshape(6, 2, 16)
    for p in range(6):
        mean_v = vrows[:p + 1].mean(axis=0)  # [2, 16]
        expect = E[p] + np.concatenate([mean_v[0], mean_v[0], mean_v[1], mean_v[1]])
        np.testing.assert_allclose(x[p], expect, rtol=1e-12, atol=1e-13)


def test_swiglu_branch_closed_form():
    # With Wq = 0 and Wo = 0 the attention adds nothing, so the layer's update
    # is Wd . (silu(Wg . xn) * (Wu . xn)) with xn the post-attention norm of
    # the embedding row.  Wg picks xn[0] * 3 / xn[0], Wu picks -xn[0] / xn[0],
    # i.e. gate g = 3 and up u = -1 in channel 0 (zero elsewhere), and Wd
    # copies channel 0 into hidden element 5.  The update is silu(3) * (-1) =
    # -3 / (1 + e^-3) = -2.857722..., while silu on the up branch gives
    # silu(-1) * 3 = -0.806824... and no silu at all gives -3.
    s = ki.TINY.replace(n_layers=1)
    H, I = s.hidden, s.intermediate
    base = {}

    def w(n, l):
        if (n, l) not in base:
            base[(n, l)] = ki.weight(s, n, l).values
        return base[(n, l)]
    tok = ki.prompt_ids(s.vocab, 1, seed=5)
    e = w("embed", -1)[tok[0]].astype(np.float64)
    xn = O.grouped_rms_norm(e, np.ones(H), 2, s.eps)
    wg = np.zeros((I, H))
    wg[0, 0] = 3.0 / xn[0]
    wu = np.zeros((I, H))
    wu[0, 0] = -1.0 / xn[0]
    wd = np.zeros((H, I))
    wd[5, 0] = 1.0

    def get(n, l):
        if n in ("wq", "wo"):
            return np.zeros(ki.tensor_shape(s, n))
        if n in ("attn_norm", "mlp_norm", "final_norm"):
            return np.ones(H)
        mlp = {"w_gate": wg, "w_up": wu, "w_down": wd}
        return mlp[n] if n in mlp else w(n, l)
    expect = e.copy()
    expect[5] += -3.0 / (1.0 + math.exp(-3.0))
    assert abs(expect[5] - e[5] - (-2.8577223804673)) < 1e-12
    got = {}
    for m in (None, "swiglu_swapped", "no_silu"):
        x, _ = O.OracleModel(s, get, "f32", mutant=m).run(tok, O.KVCache(1, 1, s.n_kv_heads, s.head_dim), logits_rows=None)
        got[m] = x[0]
    np.testing.assert_allclose(got[None], expect, rtol=0, atol=1e-12)
    # the two plausible mistakes give the hand-computed wrong values
    assert abs(got["swiglu_swapped"][5] - e[5] - (-1.0 / (1.0 + math.exp(1.0))) * 3.0) < 1e-12
    assert abs(got["no_silu"][5] - e[5] - (-3.0)) < 1e-12


@pytest.mark.parametrize("mutant", [m for m in O.MUTANTS if m is not None])
def test_planted_mutants_break_parity(mutant):
    # cpu_weights.rs, `Ablation`: a known-bad graph must move the output by far
    # more than the fp32 parity tolerance (1e-4 max-abs; here > 10x it), or the parity test
    # could not see it
    s, good, _ = _tiny()
    _, bad, _ = _tiny(mutant=mutant)
    prompt = ki.prompt_ids(s.vocab, 16)
    toks, lg = good.generate_greedy(prompt, 4)
    seq = np.concatenate([prompt, toks[:-1]])
    _, lg_bad, _ = bad.teacher_forced(seq, 15)
    assert np.max(np.abs(lg_bad - lg)) > 1e-3, mutant
