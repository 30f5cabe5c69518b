"""The bounded waits of the persistent decode step, made to run out.

A step must never hand back output it did not finish (kimi-k3-in-c k3_run.c:
abort rather than return unwritten output).  Option K2_OPT_STALL_PHASE makes
one phase of the step wait for tagged words that no phase writes; with a short
K2_OPT_WAIT_LIMIT_US the waits run out, the kernel ends early without a trap,
and the host sees K2_ERR_DEVICE_GUARD with the timeout reason.  The step must
leave no effect that matters: no token written, the sequence length not
advanced, and the next clean step bitwise equal to the same step in a
context that never failed."""
import time

import numpy as np
import pytest
import torch

import k2_inputs as ki

pytestmark = pytest.mark.gpu


def setup(k2, mio, s, prompt):
    ctx, _ = mio.build_context(s, max_context=64, kv_dtype="f16", gain_scale=0.1)
    # the prompt through the persistent step itself (fixed reduction order),
    # so two contexts hold bitwise the same cache
    ctx.set_option(k2.K2_OPT_TC_PREFILL, 0)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt)
    torch.cuda.synchronize()
    return ctx, nxt


@pytest.mark.parametrize("phase", [1, 2, 3, 4, 6, 15])
def test_stalled_phase_times_out_without_effect(phase):
    from dense_gqa_decoder_gb300 import k2, model_io as mio
    s = ki.MEDIUM  # 3 layers: phases 1..14 inside the layers, 15 the lm_head
    prompt = ki.prompt_ids(s.vocab, 11, seed=17)
    ctx, tok = setup(k2, mio, s, prompt)
    assert ctx.info().persistent_grid > 0
    n0 = ctx.kv_view(0, 0)[4]
    ctx.set_option(k2.K2_OPT_WAIT_LIMIT_US, 500)
    ctx.set_option(k2.K2_OPT_STALL_PHASE, phase)
    out = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    ctx.decode_step(tok, 1, out)
    st = ctx.sync_status()
    elapsed = time.perf_counter() - t0
    assert st == k2.K2_ERR_DEVICE_GUARD
    assert "timeout" in ctx.last_error()
    assert elapsed < 0.5  # each CTA gives up after about one or two 500 us waits
    assert int(out.item()) == -7  # no token from a failed step
    ctx.clear_status()
    assert ctx.kv_view(0, 0)[4] == n0  # the length did not advance
    ctx.set_option(k2.K2_OPT_STALL_PHASE, -1)
    ctx.set_option(k2.K2_OPT_WAIT_LIMIT_US, 1000000)
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    ctx.decode_step(tok, 1, out, logits)
    assert ctx.sync_status() == k2.K2_OK
    assert ctx.kv_view(0, 0)[4] == n0 + 1
    # the same step in a context that never failed
    ref, rtok = setup(k2, mio, s, prompt)
    assert int(rtok.item()) == int(tok.item())
    rout = torch.zeros(1, dtype=torch.int32, device="cuda")
    rlog = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    ref.decode_step(rtok, 1, rout, rlog)
    assert ref.sync_status() == k2.K2_OK
    assert int(out.item()) == int(rout.item())
    np.testing.assert_array_equal(logits.cpu().numpy(), rlog.cpu().numpy())


def test_wait_options_are_checked():
    from dense_gqa_decoder_gb300 import k2, model_io as mio
    s = ki.TINY
    ctx, _ = mio.build_context(s, max_context=8, kv_dtype="f32")
    for opt, bad in ((k2.K2_OPT_WAIT_LIMIT_US, 0), (k2.K2_OPT_WAIT_LIMIT_US, 2_000_000),
                     (k2.K2_OPT_STALL_PHASE, 0), (k2.K2_OPT_STALL_PHASE, 5 * s.n_layers + 1)):
        with pytest.raises(k2.K2Error) as e:
            ctx.set_option(opt, bad)
        assert e.value.status == k2.K2_ERR_ARG
