"""fp8 (E4M3) weight-only decoding (weight_dtype K2_F8) against the oracle.

The quantizer must produce the oracle's codes and scales bit for bit
(oracle/k2_fp8.py, written from the E4M3 definition); a model stored in fp8
must then match the oracle's forward pass over the same quantized weights
(k2-burn README, "Post-training quantization": fp8 checkpoints run directly)."""
import numpy as np
import pytest
import torch

import k2_inputs as ki
from oracle import k2_fp8 as Q8
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


def bf16_round(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def test_quantizer_matches_the_oracle_bit_for_bit(k2):
    rows, cols = 257, 1000
    w = ki.normal_f32(5, 77, rows * cols).reshape(rows, cols) * np.float32(0.05)
    w[3] = 0.0
    w[10, 17] = 300.0
    w[11] *= np.float32(1e-6)
    w = bf16_round(w)
    dev = torch.tensor(w).to(torch.bfloat16).cuda()
    codes, scales = k2.quantize_fp8(dev)
    want_c, want_s = Q8.quantize_rows(w)
    np.testing.assert_array_equal(scales.cpu().numpy(), want_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_c)


@pytest.mark.parametrize("shape,kv", [("medium", "f16"), ("medium", "i8"), ("k2_layer", "f16")])
def test_fp8_model_matches_the_oracle(k2, mio, shape, kv):
    s = ki.SHAPES[shape]
    ctx, host = mio.build_context(s, max_context=96, kv_dtype=kv, gain_scale=0.1, keep_host=True, weights="f8")
    assert ctx.info().persistent_grid > 0
    prompt = ki.prompt_ids(s.vocab, 20, seed=90)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits)
    toks, lgs = [int(nxt.item())], [logits.cpu().numpy().copy()]
    for _ in range(8):
        ctx.decode_step(nxt, 1, nxt, logits)
        toks.append(int(nxt.item()))
        lgs.append(logits.cpu().numpy().copy())
    assert ctx.sync_status() == k2.K2_OK
    model = O.OracleModel(s, Q8.fp8_weights(lambda n, l: host[(n, l)]), kv)
    seq = np.concatenate([prompt, toks[:-1]])
    am, ref, _ = model.teacher_forced(seq, len(prompt) - 1)
    got = np.stack(lgs).astype(np.float64)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel <= (2e-4 if kv == "f16" else 5e-2), rel
    assert np.mean(am == np.array(toks)) >= (1.0 if kv == "f16" else 0.85)
    # and the fp8 model is not the bf16 one
    _, ref16, _ = O.OracleModel(s, lambda n, l: host[(n, l)], kv).teacher_forced(seq, len(prompt) - 1)
    assert float(np.linalg.norm(got - ref16) / np.linalg.norm(ref16)) > 1e-3


def test_fp8_refuses_the_kernel_chain(k2, mio):
    ctx, _ = mio.build_context(ki.MEDIUM, max_context=32, kv_dtype="f16", weights="f8")
    with pytest.raises(k2.K2Error) as e:
        ctx.set_option(k2.K2_OPT_PERSISTENT, 0)
    assert e.value.status == k2.K2_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,kv,n", [("medium", "f16", 40), ("medium", "i8", 9), ("k2_layer", "f16", 300)])
def test_fp8_tensor_core_prefill_matches_stepwise(k2, mio, shape, kv, n):
    """A prompt of fp8 weights on the tensor cores (bf16 copies of the codes, the
    row scales in the GEMM epilogue, the last token on the persistent step)
    against the same prompt appended one persistent step per token, and against
    the oracle's full recompute over the same quantized weights.  The bar is the
    bf16 tensor-core prefill's: its activations enter the MMAs as bf16 hi + lo
    halves (~16 significant bits), 2e-4 relative on the logits."""
    s = ki.SHAPES[shape]
    ids = ki.prompt_ids(s.vocab, n, seed=94)
    prompt = torch.tensor(ids, dtype=torch.int32, device="cuda")
    runs = []
    for tc in (1, 0):
        ctx, host = mio.build_context(s, max_context=n + 16, kv_dtype=kv, gain_scale=0.1, keep_host=True,
                                      weights="f8")
        info = ctx.info()
        assert info.tc_prefill == 1 and info.tc_batched == 0
        ctx.set_option(k2.K2_OPT_TC_PREFILL, tc)
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
        ctx.prefill(0, prompt, nxt, logits)
        toks, lgs = [int(nxt.item())], [logits.cpu().numpy().copy()]
        for _ in range(4):
            ctx.decode_step(nxt, 1, nxt, logits)
            toks.append(int(nxt.item()))
            lgs.append(logits.cpu().numpy().copy())
        assert ctx.sync_status() == k2.K2_OK
        runs.append((toks, np.stack(lgs).astype(np.float64)))
    (t_tc, l_tc), (t_st, l_st) = runs
    rel = float(np.linalg.norm(l_tc - l_st) / np.linalg.norm(l_st))
    assert rel <= (2e-4 if kv == "f16" else 2e-2), rel
    ref = O.OracleModel(s, Q8.fp8_weights(lambda nm, l: host[(nm, l)]), kv).forward_full(ids)
    rel_o = float(np.linalg.norm(l_tc[0] - ref) / np.linalg.norm(ref))
    assert rel_o <= (2e-4 if kv == "f16" else 5e-2), rel_o
    if kv == "f16":
        assert t_tc == t_st
        assert t_tc[0] == O.argmax_first(ref)
