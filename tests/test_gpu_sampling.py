"""The sampler (k2_sample.cu) against the sampling oracle (oracle/k2_sampling.py).

Both sides take every decision in the same precision (float32 operations,
the sampler's own exp, integer masses), so on the same fp32 logits the drawn
ids must be identical: seeded synthetic logit rows at the tiny vocabulary
and at the 3.7B shape's 250624, with ties, -inf and NaN entries, every
filter alone and together.  Then sampled decoding of the tiny fp32 model
against the oracle's own forward pass, temperature 0 against greedy, and the
same draws after a cache save / restore (k2-burn README, "Sampling + greedy
generation": a seeded RNG; temperature 0 = greedy argmax)."""
import numpy as np
import pytest
import torch

import k2_inputs as ki
from oracle import k2_oracle as O
from oracle import k2_sampling as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


@pytest.fixture(scope="module")
def mio():
    from dense_gqa_decoder_gb300 import model_io
    return model_io


def test_philox_matches_the_oracle(k2):
    for first, c1, key in ((0, 0, 0), (4093, 7, 0x0123456789ABCDEF), (0xFFFFFF00, 0xFFFFFFFF, 2 ** 64 - 1)):
        got = k2.philox(first, 300, c1=c1, c2=3, c3=0xDEADBEEF, key=key).numpy()
        for i in (0, 1, 17, 255, 299):
            want = S.philox4x32_10(((first + i) & 0xFFFFFFFF, c1, 3, 0xDEADBEEF), (key & 0xFFFFFFFF, key >> 32))
            assert tuple(int(v) for v in got[i]) == want
    assert tuple(int(v) for v in k2.philox(0, 1).numpy()[0]) == (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)


PARAMS = [
    dict(temperature=1.0),
    dict(temperature=0.7, top_k=40),
    dict(temperature=1.3, top_p=0.9),
    dict(temperature=0.9, min_p=0.05),
    dict(temperature=1.0, repetition_penalty=1.3),
    dict(temperature=0.8, top_k=50, top_p=0.95, min_p=0.02, repetition_penalty=1.2),
    dict(temperature=2.0, top_k=1),
    dict(temperature=0.05, top_p=0.5),
]


def sampler_ctx(mio, vocab, rows=4):
    s = ki.TINY.replace(vocab=vocab)
    ctx, _ = mio.build_context(s, max_context=64, max_batch=rows, kv_dtype="f32")
    return ctx


@pytest.mark.parametrize("vocab", [512, 250624])
def test_sampler_draws_the_oracles_ids(k2, mio, vocab):
    rows = 4
    ctx = sampler_ctx(mio, vocab, rows)
    stride = 40
    seen = np.stack([ki.prompt_ids(vocab, stride, seed=200 + r) for r in range(rows)]).astype(np.int32)
    seen_len = np.array([0, 5, 17, 40], np.int32)
    d_seen = torch.tensor(seen, device="cuda")
    d_seen_len = torch.tensor(seen_len, device="cuda")
    nxt = torch.zeros(rows, dtype=torch.int32, device="cuda")
    checked = 0
    for pi, prm in enumerate(PARAMS):
        for case, kw in enumerate((dict(), dict(ties=3, neg_inf=5, nan=2))):
            lg = ki.logit_rows(rows, vocab, seed=1000 + 10 * pi + case, scale=3.0, **kw)
            seed = 77 + pi
            pos = np.array([9, 100, 4096, 123456], np.int32)
            ctx.set_sampling(k2.sampling(seed=seed, **prm))
            ctx.sample_logits(torch.tensor(lg, device="cuda"), rows, torch.tensor(pos, device="cuda"), nxt,
                              seen=d_seen, seen_len=d_seen_len, first_seq=2)
            got = nxt.cpu().tolist()
            for r in range(rows):
                want = S.sample_row(lg[r], prm["temperature"], prm.get("top_k", 0), prm.get("top_p", 1.0),
                                    prm.get("min_p", 0.0), prm.get("repetition_penalty", 1.0),
                                    seen[r, :seen_len[r]].tolist(), seed, int(pos[r]), 2 + r)
                assert got[r] == want, (prm, case, r)
                checked += 1
    assert checked == len(PARAMS) * 2 * rows
    assert ctx.sync_status() == k2.K2_OK


def test_sampled_decoding_matches_the_oracle(k2, mio):
    s = ki.TINY
    prm = dict(temperature=0.9, top_k=60, top_p=0.95, repetition_penalty=1.3, seed=5)
    ctx, host = mio.build_context(s, max_context=64, kv_dtype="f32", keep_host=True)
    ctx.set_sampling(k2.sampling(**prm))
    prompt = ki.prompt_ids(s.vocab, 12, seed=8)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt)
    toks = [int(nxt.item())]
    for _ in range(20):
        ctx.decode_step(nxt, 1, nxt)
        toks.append(int(nxt.item()))
    assert ctx.sync_status() == k2.K2_OK
    want = S.generate_sampled(O.OracleModel(s, lambda n, l: host[(n, l)], "f32"), prompt, 20, prm, capacity=64)
    assert toks == want.tolist()
    # greedy would differ somewhere over 21 draws at temperature 0.9
    greedy, _ = O.OracleModel(s, lambda n, l: host[(n, l)], "f32").generate_greedy(prompt, 20, capacity=64)
    assert toks != greedy.tolist()


@pytest.mark.parametrize("graph", [0, 1])
def test_temperature_zero_is_the_greedy_step(k2, mio, graph):
    s = ki.MEDIUM
    prompt = ki.prompt_ids(s.vocab, 30, seed=9)
    out = []
    for mode in ("unset", "zero"):
        ctx, _ = mio.build_context(s, max_context=64, kv_dtype="f16", gain_scale=0.1)
        ctx.set_option(k2.K2_OPT_GRAPH, graph)
        # the tensor-core prefill adds split-K partials with atomics, whose order
        # varies between runs; appending the prompt step by step is bitwise repeatable
        ctx.set_option(k2.K2_OPT_TC_PREFILL, 0)
        if mode == "zero":
            ctx.set_sampling(k2.sampling(temperature=0.9, seed=3))
            ctx.set_sampling(k2.sampling(temperature=0.0, top_k=5, seed=3))  # back to greedy
        stream = torch.cuda.Stream()
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits, stream=stream)
            toks, lgs = [], []
            for _ in range(6):
                ctx.decode_step(nxt, 1, nxt, logits, stream=stream)
                toks.append(nxt.clone())
                lgs.append(logits.clone())
        stream.synchronize()
        out.append((torch.stack(toks).cpu(), torch.stack(lgs).cpu()))
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])


def test_resumed_sequence_draws_the_same_tokens(k2, mio):
    s = ki.MEDIUM
    prm = k2.sampling(temperature=1.0, top_p=0.9, repetition_penalty=1.1, seed=11)
    prompt = list(ki.prompt_ids(s.vocab, 25, seed=12))

    def run(ctx, tok, n):
        nxt = torch.tensor([tok], dtype=torch.int32, device="cuda")
        out = []
        for _ in range(n):
            ctx.decode_step(nxt, 1, nxt)
            out.append(int(nxt.item()))
        return out

    ctx, _ = mio.build_context(s, max_context=80, kv_dtype="f16", gain_scale=0.1)
    ctx.set_sampling(prm)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt)
    first = [int(nxt.item())] + run(ctx, int(nxt.item()), 4)
    state = ctx.kv_save(0, prompt + first)
    ref = run(ctx, first[-1], 10)
    ctx2, _ = mio.build_context(s, max_context=96, kv_dtype="f16", gain_scale=0.1)
    ctx2.set_sampling(prm)
    ids = ctx2.kv_load(0, state)
    assert run(ctx2, ids[-1], 10) == ref
    assert ctx2.sync_status() == k2.K2_OK


def test_batched_sampled_decoding_is_reproducible(k2, mio):
    s = ki.MEDIUM
    B = 3
    prm = k2.sampling(temperature=0.8, top_k=20, seed=21)
    runs = []
    for _ in range(2):
        ctx, _ = mio.build_context(s, max_context=64, max_batch=B, kv_dtype="f16", gain_scale=0.1)
        ctx.set_sampling(prm)
        nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
        for b in range(B):
            ctx.prefill(b, torch.tensor(ki.prompt_ids(s.vocab, 10 + b, seed=30 + b), dtype=torch.int32,
                                        device="cuda"), nxt[b:b + 1])
        toks = [nxt.cpu().clone()]
        for _ in range(6):
            ctx.decode_step(nxt, B, nxt)
            toks.append(nxt.cpu().clone())
        assert ctx.sync_status() == k2.K2_OK
        runs.append(torch.stack(toks))
    assert torch.equal(runs[0], runs[1])
    assert int(runs[0].max()) < s.vocab and int(runs[0].min()) >= 0


def test_bad_sampling_parameters_are_refused(k2, mio):
    ctx = sampler_ctx(mio, 512, 1)
    for bad in (dict(temperature=-1.0), dict(temperature=1.0, top_p=0.0), dict(temperature=1.0, top_p=1.5),
                dict(temperature=1.0, min_p=-0.1), dict(temperature=1.0, repetition_penalty=0.0),
                dict(temperature=1.0, top_k=-2), dict(temperature=float("inf"))):
        with pytest.raises(k2.K2Error) as e:
            ctx.set_sampling(k2.sampling(**bad))
        assert e.value.status == k2.K2_ERR_ARG
    lg = torch.zeros(1, 512, device="cuda")
    with pytest.raises(k2.K2Error):  # not set: greedy has no sampler
        ctx.sample_logits(lg, 1, torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.zeros(1, dtype=torch.int32, device="cuda"))
