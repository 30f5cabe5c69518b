"""k2_greedy_head_noalloc, the greedy head for callers that cannot allocate
device memory (its scratch is a static device array inside libk2).

Each call is checked against the existing path: after a k2_decode_step, the
residual it left (k2_hidden_view) goes through the no-workspace call, whose
logits must match the step's logits within the fp32 tolerance of the other
tests (1e-4 max-abs) and whose token must equal the step's token.  Two steps,
so two calls in a row share the static scratch.  A hidden state holding a NaN
must come back as token -1 (the call has no other way to report a device-side
failure), and the next ordinary call must be clean again."""
import numpy as np
import pytest
import torch

import k2_inputs as ki

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape_name,kv", [("tiny", "f32"), ("medium", "f16")])
def test_noalloc_head_matches_decode_step(shape_name, kv):
    from dense_gqa_decoder_gb300 import k2, model_io
    s = ki.SHAPES[shape_name]
    ctx, _ = model_io.build_context(s, max_context=40, kv_dtype=kv, gain_scale=0.1)
    prompt = torch.tensor(ki.prompt_ids(s.vocab, 12, seed=21), dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, prompt, tok)
    x = k2.device_view(ctx.hidden_view(0), s.hidden, torch.float32)
    step_logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    head_logits = torch.full((s.vocab,), float("nan"), dtype=torch.float32, device="cuda")
    head_tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        ctx.decode_step(tok, 1, tok, step_logits)
        xs = x.clone()
        st = k2.greedy_head_noalloc(ctx.cfg, ctx.weights["lm_head"], ctx.weights["final_norm"], xs, head_logits,
                                    head_tok)
        assert st == k2.K2_OK
        torch.cuda.synchronize()
        a, b = head_logits.cpu().numpy(), step_logits.cpu().numpy()
        assert np.max(np.abs(a - b)) <= 1e-4
        assert int(head_tok.item()) == int(tok.item())
    assert ctx.sync_status() == k2.K2_OK


def test_noalloc_head_refuses_bad_arguments():
    from dense_gqa_decoder_gb300 import k2
    s = ki.TINY
    cfg = k2.make_config(s, max_context=8, kv_dtype="f32")
    w = torch.zeros(s.vocab, s.hidden, device="cuda")
    g = torch.ones(s.hidden, device="cuda")
    x = torch.zeros(s.hidden, device="cuda")
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert k2.greedy_head_noalloc(cfg, w, g, None, None, t) == k2.K2_ERR_ARG
    bad = k2.make_config(s.replace(hidden=63), max_context=8, kv_dtype="f32")
    assert k2.greedy_head_noalloc(bad, w, g, x, None, t) == k2.K2_ERR_SHAPE
    assert k2.greedy_head_noalloc(cfg, w, g, x, None, t) == k2.K2_OK
    torch.cuda.synchronize()
    assert int(t.item()) == 0  # all logits 0: the first index wins


@pytest.mark.parametrize("where", ["one", "all"])
def test_noalloc_head_reports_nan_and_recovers(where):
    # a NaN in the hidden state makes NaN logits: the token is -1; the guard
    # bits live in the shared static scratch, so the call after it must start
    # clean and give the decode step's token again
    from dense_gqa_decoder_gb300 import k2, model_io
    s = ki.MEDIUM
    ctx, _ = model_io.build_context(s, max_context=24, kv_dtype="f16", gain_scale=0.1)
    prompt = torch.tensor(ki.prompt_ids(s.vocab, 9, seed=4), dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, prompt, tok)
    step_logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    ctx.decode_step(tok, 1, tok, step_logits)
    x = k2.device_view(ctx.hidden_view(0), s.hidden, torch.float32).clone()
    w, g = ctx.weights["lm_head"], ctx.weights["final_norm"]
    if where == "one":
        # one NaN row of the lm_head: one NaN logit among finite ones
        bad_x, bad_w = x, w.clone()
        bad_w[s.vocab // 2] = float("nan")
    else:
        bad_x, bad_w = torch.full_like(x, float("nan")), w
    head_tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    head_logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    assert k2.greedy_head_noalloc(ctx.cfg, bad_w, g, bad_x, head_logits, head_tok) == k2.K2_OK
    torch.cuda.synchronize()
    assert int(head_tok.item()) == -1
    n_nan = int(torch.isnan(head_logits).sum())
    assert n_nan == (1 if where == "one" else s.vocab)
    assert k2.greedy_head_noalloc(ctx.cfg, w, g, x, head_logits, head_tok) == k2.K2_OK
    torch.cuda.synchronize()
    assert int(head_tok.item()) == int(tok.item())
    assert np.max(np.abs(head_logits.cpu().numpy() - step_logits.cpu().numpy())) <= 1e-4
    assert ctx.sync_status() == k2.K2_OK


def test_noalloc_head_binding_checks_tensors():
    # the binding refuses tensors the C call would misread
    from dense_gqa_decoder_gb300 import k2
    s = ki.TINY
    cfg = k2.make_config(s, max_context=8, kv_dtype="f32")
    w = torch.zeros(s.vocab, s.hidden, device="cuda")
    g = torch.ones(s.hidden, device="cuda")
    x = torch.zeros(s.hidden, device="cuda")
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        k2.greedy_head_noalloc(cfg, w, g, x.to(torch.bfloat16), None, t)
    with pytest.raises(ValueError):
        k2.greedy_head_noalloc(cfg, w, g, x, None, t.to(torch.int64))
    with pytest.raises(ValueError):
        k2.greedy_head_noalloc(cfg, w.t(), g, x, None, t)
