"""Speculative decoding (k2_decode_speculative) against serial greedy
decoding: the emitted ids must be the same stream (kimi-k3-in-c k3_run.c,
--spec: "batched greedy verification accepts precisely the prefix the model
itself would have emitted"), with fewer passes than ids once drafts hit.
The prompt repeats a pattern so that n-gram drafts exist from the start."""
import numpy as np
import pytest
import torch

import k2_inputs as ki

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


@pytest.fixture(scope="module")
def mio():
    from dense_gqa_decoder_gb300 import model_io
    return model_io


def repetitive_prompt(vocab, seed):
    unit = list(ki.prompt_ids(vocab, 7, seed=seed))
    return unit * 4 + unit[:3]


def serial(ctx, prompt, n, vocab):
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt)
    out = [int(nxt.item())]
    while len(out) < n:
        ctx.decode_step(nxt, 1, nxt)
        out.append(int(nxt.item()))
    return out


def speculative(ctx, prompt, n, max_draft=8, stream=None):
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt)
    torch.cuda.synchronize()
    seq = list(prompt) + [int(nxt.item())]
    out = [seq[-1]]
    passes = 0
    while len(out) < n:
        got = ctx.decode_speculative(0, seq, max_draft, stream=stream)
        passes += 1
        out += got
        seq += got
        assert ctx.kv_view(0, 0)[4] == len(seq) - 1
    return out[:n], passes


@pytest.mark.parametrize("shape,kv,repeats,graph", [("medium", "f16", True, 0), ("medium", "f16", True, 1),
                                                   ("medium", "i8", True, 1), ("k2_layer", "f16", False, 1)])
def test_speculative_stream_equals_serial_greedy(k2, mio, shape, kv, repeats, graph):
    s = ki.SHAPES[shape]
    n = 48
    prompt = repetitive_prompt(s.vocab, seed=40)
    ctx, _ = mio.build_context(s, max_context=160, kv_dtype=kv, gain_scale=0.1)
    ref = serial(ctx, prompt, n, s.vocab)
    ctx.kv_reset(0)
    # graphs: every block size is recorded once and replayed at later positions
    ctx.set_option(k2.K2_OPT_GRAPH, graph)
    stream = torch.cuda.Stream() if graph else None
    got, passes = speculative(ctx, prompt, n, stream=stream)
    assert got == ref
    assert ctx.sync_status() == k2.K2_OK
    # this medium model's greedy continuation repeats the prompt's pattern, so
    # drafts are accepted; the one-layer model's does not (its stream must
    # still be the serial one)
    if repeats:
        assert passes < n - 1, passes


def test_speculative_without_drafts_is_a_decode_step(k2, mio):
    s = ki.MEDIUM
    prompt = list(ki.prompt_ids(s.vocab, 20, seed=41))  # no repeats
    ctx, _ = mio.build_context(s, max_context=64, kv_dtype="f16", gain_scale=0.1)
    ref = serial(ctx, prompt, 4, s.vocab)
    ctx.kv_reset(0)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt)
    seq = prompt + [int(nxt.item())]
    assert ctx.decode_speculative(0, seq, 8) == [ref[1]]


def test_speculative_refusals(k2, mio):
    s = ki.MEDIUM
    ctx, _ = mio.build_context(s, max_context=64, kv_dtype="f16", gain_scale=0.1)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda"), nxt)
    with pytest.raises(k2.K2Error) as e:
        ctx.decode_speculative(0, [1, 2], 8)  # must be the 3 cached ids + the input
    assert e.value.status == k2.K2_ERR_ARG
    ctx.set_sampling(k2.sampling(temperature=1.0))
    with pytest.raises(k2.K2Error) as e:
        ctx.decode_speculative(0, [1, 2, 3, int(nxt.item())], 8)
    assert e.value.status == k2.K2_ERR_UNSUPPORTED
