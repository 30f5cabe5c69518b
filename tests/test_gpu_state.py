"""Saved cache state on the GPU (k2_kv_save / k2_kv_load).

A sequence is saved, restored into a fresh context of another size, and
decoding continues: the tokens and logits must be bit-identical to the run
that was never interrupted, and (tiny fp32 model) equal to the oracle's
greedy continuation of the whole conversation (kimi-k3-in-c k3_run.c,
"conversation state": a resumed session pays only for its new tokens).  A
state written for another model or KV format, or one that does not fit, is
refused before anything changes."""
import numpy as np
import pytest
import torch

import k2_inputs as ki
from oracle import k2_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


@pytest.fixture(scope="module")
def mio():
    from dense_gqa_decoder_gb300 import model_io
    return model_io


def greedy(ctx, prompt, n_new, vocab):
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(vocab, dtype=torch.float32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits)
    toks, lgs = [int(nxt.item())], [logits.cpu().numpy().copy()]
    toks2, lgs2 = decode(ctx, toks[0], n_new, vocab)
    return toks + toks2, lgs + lgs2


def decode(ctx, tok, n, vocab):
    nxt = torch.tensor([tok], dtype=torch.int32, device="cuda")
    logits = torch.empty(vocab, dtype=torch.float32, device="cuda")
    toks, lgs = [], []
    for _ in range(n):
        ctx.decode_step(nxt, 1, nxt, logits)
        toks.append(int(nxt.item()))
        lgs.append(logits.cpu().numpy().copy())
    return toks, lgs


def cache_rows(k2, ctx, layer, n, kv):
    """K, V (and int8 scales) rows 0..n-1 of sequence 0 of a layer, as bytes."""
    info = ctx.info()
    cap, nkv, d = info.kv_capacity, ctx.cfg.n_kv_heads, ctx.cfg.head_dim
    kp, vp, ksp, vsp, _ = ctx.kv_view(layer, 0)
    dt = {"f32": torch.float32, "f16": torch.float16, "i8": torch.int8}[kv]
    out = []
    for p in (kp, vp):
        out.append(k2.device_view(p, nkv * cap * d, dt).view(nkv, cap, d)[:, :n].contiguous().cpu())
    if kv == "i8":
        for p in (ksp, vsp):
            out.append(k2.device_view(p, nkv * cap, torch.float16).view(nkv, cap)[:, :n].contiguous().cpu())
    return out


@pytest.mark.parametrize("shape,kv", [("tiny", "f32"), ("medium", "f16"), ("medium", "i8")])
def test_resume_continues_bit_identically(k2, mio, shape, kv, tmp_path):
    s = ki.SHAPES[shape]
    gs = 0.0 if shape == "tiny" else 0.1
    prompt = list(ki.prompt_ids(s.vocab, 21, seed=71))
    ctx, host = mio.build_context(s, max_context=64, kv_dtype=kv, gain_scale=gs, keep_host=True)
    first, _ = greedy(ctx, prompt, 5, s.vocab)
    history = prompt + first[:-1]           # the tokens whose K/V rows are cached
    conversation = history + [first[-1]]    # and the next input
    state = ctx.kv_save(0, conversation)
    assert state.numel() == ctx.kv_state_bytes(0, len(conversation))
    assert k2.peek_state(ctx.cfg, state) == (len(history), len(conversation))
    saved_rows = [cache_rows(k2, ctx, l, len(history), kv) for l in (0, s.n_layers - 1)]
    ref_toks, ref_lgs = decode(ctx, first[-1], 8, s.vocab)   # never interrupted
    assert ctx.sync_status() == k2.K2_OK

    path = str(tmp_path / "conversation.k2st")
    k2.save_state_file(path, state)
    del ctx
    torch.cuda.empty_cache()
    # another context size and batch, the same weights
    ctx2, _ = mio.build_context(s, max_context=100, max_batch=2, kv_dtype=kv, gain_scale=gs)
    ids = ctx2.kv_load(0, k2.load_state_file(path))
    assert ids == conversation
    assert ctx2.kv_view(0, 0)[4] == len(history)
    for l, rows in zip((0, s.n_layers - 1), saved_rows):
        for a, b in zip(rows, cache_rows(k2, ctx2, l, len(history), kv)):
            assert torch.equal(a, b)
    toks, lgs = decode(ctx2, ids[-1], 8, s.vocab)
    assert toks == ref_toks
    for a, b in zip(lgs, ref_lgs):
        np.testing.assert_array_equal(a, b)
    assert ctx2.sync_status() == k2.K2_OK
    if shape == "tiny":  # fp32: the oracle's greedy tokens of the whole conversation
        want, _ = O.OracleModel(s, lambda n, l: host[(n, l)], "f32").generate_greedy(
            np.array(prompt), 5 + 8, capacity=64)
        assert first + toks == [int(t) for t in want]


def test_refused_states_change_nothing(k2, mio):
    s = ki.MEDIUM
    prompt = ki.prompt_ids(s.vocab, 30, seed=72)
    ctx, _ = mio.build_context(s, max_context=64, kv_dtype="f16", gain_scale=0.1)
    greedy(ctx, list(prompt), 0, s.vocab)
    state = ctx.kv_save(0, [1, 2, 3])
    assert k2.peek_state(ctx.cfg, state) == (30, 3)

    def refused(target, data, status):
        before = target.kv_view(0, 0)[4]
        with pytest.raises(k2.K2Error) as e:
            target.kv_load(0, data)
        assert e.value.status == status, e.value
        assert target.kv_view(0, 0)[4] == before

    other_kv, _ = mio.build_context(s, max_context=64, kv_dtype="i8", gain_scale=0.1)
    refused(other_kv, state, k2.K2_ERR_STATE)
    other_model, _ = mio.build_context(s.replace(n_layers=2), max_context=64, kv_dtype="f16", gain_scale=0.1)
    refused(other_model, state, k2.K2_ERR_STATE)
    small, _ = mio.build_context(s, max_context=16, kv_dtype="f16", gain_scale=0.1)
    refused(small, state, k2.K2_ERR_CONTEXT_FULL)
    damaged = state.clone()
    damaged[12] ^= 1  # inside the fingerprint (n_layers)
    refused(ctx, damaged, k2.K2_ERR_STATE)
    refused(ctx, state[:-16].clone(), k2.K2_ERR_STATE)
    # the untouched state still loads
    assert ctx.kv_load(0, state) == [1, 2, 3]


def test_save_refuses_while_the_device_guard_is_set(k2, mio):
    s = ki.TINY
    ctx, _ = mio.build_context(s, max_context=32, kv_dtype="f32")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor([3, s.vocab + 5], dtype=torch.int32, device="cuda"), nxt)
    with pytest.raises(k2.K2Error) as e:
        ctx.kv_save(0, [])
    assert e.value.status == k2.K2_ERR_DEVICE_GUARD
    ctx.clear_status()
    ctx.kv_reset(0)
    ctx.prefill(0, torch.tensor([3, 4], dtype=torch.int32, device="cuda"), nxt)
    assert k2.peek_state(ctx.cfg, ctx.kv_save(0, [])) == (2, 0)
