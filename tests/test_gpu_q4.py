"""int4 block-64 weight-only decoding (weight_dtype K2_Q4) against the oracle.

The quantizer must produce the oracle's codes and block scales bit for bit
(oracle/k2_q4.py, symmetric codes in [-7, 7], one scale per 64 weights of a
row); a model stored in int4 must then match the oracle's forward pass over
the same quantized weights (k2-burn README, "Quantization": int4 checkpoints
with block size 64 run directly)."""
import numpy as np
import pytest
import torch

import k2_inputs as ki
from oracle import k2_oracle as O
from oracle import k2_q4 as Q4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


@pytest.fixture(scope="module")
def mio():
    from dense_gqa_decoder_gb300 import model_io
    return model_io


def bf16_round(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("rows,cols", [(257, 1000), (3, 64), (5, 2100)])
def test_quantizer_matches_the_oracle_bit_for_bit(k2, rows, cols):
    w = ki.normal_f32(6, 78, rows * cols).reshape(rows, cols) * np.float32(0.05)
    w[0, :min(64, cols)] = 0.0                   # a zero block
    w[rows - 1, cols - 1] = 40.0                 # an outlier in the ragged last block
    w[1 % rows] *= np.float32(1e-6)              # tiny values
    if cols >= 64:  # exact ties: a block with scale 1/8 and quotients k / 2
        w[2 % rows, :64] = (np.arange(64) % 29 - 14) / 16.0
        w[2 % rows, 0] = 0.875
    w = bf16_round(w)
    dev = torch.tensor(w).to(torch.bfloat16).cuda()
    codes, scales = k2.quantize_q4(dev)
    want_c, want_s = Q4.quantize_rows(w)
    np.testing.assert_array_equal(scales.cpu().numpy(), want_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_c)


@pytest.mark.parametrize("shape,kv", [("medium", "f16"), ("medium", "i8"), ("k2_layer", "f16")])
def test_q4_model_matches_the_oracle(k2, mio, shape, kv):
    s = ki.SHAPES[shape]
    ctx, host = mio.build_context(s, max_context=96, kv_dtype=kv, gain_scale=0.1, keep_host=True, weights="q4")
    assert ctx.info().persistent_grid > 0
    prompt = ki.prompt_ids(s.vocab, 20, seed=91)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits)
    toks, lgs = [int(nxt.item())], [logits.cpu().numpy().copy()]
    for _ in range(8):
        ctx.decode_step(nxt, 1, nxt, logits)
        toks.append(int(nxt.item()))
        lgs.append(logits.cpu().numpy().copy())
    assert ctx.sync_status() == k2.K2_OK
    model = O.OracleModel(s, Q4.q4_weights(lambda n, l: host[(n, l)]), kv)
    seq = np.concatenate([prompt, toks[:-1]])
    am, ref, _ = model.teacher_forced(seq, len(prompt) - 1)
    got = np.stack(lgs).astype(np.float64)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel <= (2e-4 if kv == "f16" else 5e-2), rel
    assert np.mean(am == np.array(toks)) >= (1.0 if kv == "f16" else 0.85)
    # and the int4 model is not the bf16 one
    _, ref16, _ = O.OracleModel(s, lambda n, l: host[(n, l)], kv).teacher_forced(seq, len(prompt) - 1)
    assert float(np.linalg.norm(got - ref16) / np.linalg.norm(ref16)) > 1e-3


def test_q4_refuses_the_kernel_chain(k2, mio):
    ctx, _ = mio.build_context(ki.MEDIUM, max_context=32, kv_dtype="f16", weights="q4")
    with pytest.raises(k2.K2Error) as e:
        ctx.set_option(k2.K2_OPT_PERSISTENT, 0)
    assert e.value.status == k2.K2_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,first,n", [("medium", 0, 300), ("k2_layer", 37, 2100)])
def test_q4_tensor_core_prefill_against_stepwise_and_oracle(k2, mio, shape, first, n):
    """The int4 prefill on the tensor cores (each layer's codes * scales
    dequantized into bf16 high and low halves, three MMAs per K step) against
    the same prompt appended one persistent step per token (K2_OPT_TC_PREFILL
    = 0) and the oracle's full recompute over the same quantized weights; the
    3.7B layer's prompt spans two 2048-token blocks after `first` cached rows."""
    s = ki.SHAPES[shape]
    pre = ki.prompt_ids(s.vocab, first, seed=93) if first else None
    prompt = ki.prompt_ids(s.vocab, n, seed=94)
    out = {}
    for tc in (1, 0):
        ctx, host = mio.build_context(s, max_context=first + n + 8, kv_dtype="f16", gain_scale=0.1, keep_host=True,
                                      weights="q4")
        assert ctx.info().tc_prefill == 1
        ctx.set_option(k2.K2_OPT_TC_PREFILL, tc)
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
        if pre is not None:
            ctx.prefill(0, torch.tensor(pre, dtype=torch.int32, device="cuda"), nxt, logits)
        ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits)
        torch.cuda.synchronize()
        assert ctx.sync_status() == k2.K2_OK
        out[tc] = (int(nxt.item()), logits.cpu().numpy().astype(np.float64))
        del ctx
        torch.cuda.empty_cache()
    seq = prompt if pre is None else np.concatenate([pre, prompt])
    ref = O.OracleModel(s, Q4.q4_weights(lambda nm, l: host[(nm, l)]), "f16").forward_full(seq)
    (t1, l1), (t0, l0) = out[1], out[0]
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))  # noqa: E731
    assert rel(l0, ref) <= 2e-4
    assert rel(l1, ref) <= 2e-4
    # the two GPU paths round differently (fp32 dot products against ~16-bit
    # halves of weights and inputs): their distance is the sum of their errors
    # (1.1e-4 measured on the 2137-token case), within the same bar
    assert rel(l1, l0) <= 2e-4
    assert t1 == t0 == O.argmax_first(ref)
