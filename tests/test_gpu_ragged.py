"""Reduction lengths that end inside a packed chunk, for every weight format
of the persistent step, against the oracle (k2-burn README, "Status: v0":
the decoder's forward pass; "Quantization": fp8 / int4 checkpoints).

hidden 640 = 2.5 bf16 chunks of 256, 1.25 fp8 chunks of 512 and 1.25 int4
chunks of 512 weights; intermediate 1664 = 6.5 bf16 chunks and 3.25 chunks
for fp8 / int4 (down projection), so every GEMV streams zero-padded tails
(zero codes, zero block scales) and its input vector is zero past K.  The
20-token prompt takes the tensor-core prefill for bf16 and fp8 weights, one
step per token for int4."""
import numpy as np
import pytest
import torch

import k2_inputs as ki
from oracle import k2_fp8 as Q8
from oracle import k2_oracle as O
from oracle import k2_q4 as Q4

pytestmark = pytest.mark.gpu

RAGGED = ki.ModelShape(hidden=640, n_layers=2, n_heads=8, n_kv_heads=2, head_dim=64, intermediate=1664,
                       norm_groups=2, vocab=1000, eps=1e-6, rope_theta=10000.0, weight_dtype="bf16")


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


@pytest.fixture(scope="module")
def mio():
    from dense_gqa_decoder_gb300 import model_io
    return model_io


# hidden 200 (three full 64-weight blocks and a partial one), intermediate 328,
# an odd vocab of 301 (the last 16-row tile holds 13 rows, the last pair one)
ODD = ki.ModelShape(hidden=200, n_layers=2, n_heads=4, n_kv_heads=1, head_dim=64, intermediate=328,
                    norm_groups=2, vocab=301, eps=1e-6, rope_theta=10000.0, weight_dtype="bf16")


@pytest.mark.parametrize("shape", ["ragged", "odd"])
@pytest.mark.parametrize("weights", ["bf16", "f8", "q4"])
def test_ragged_reduction_lengths_match_the_oracle(k2, mio, weights, shape):
    """Every packed format (pair units, and the fp8 / int4 tile units of
    gate/up and the lm_head) over reduction lengths and row counts that end
    inside a chunk, a 64-weight block or a 16-row tile, against the oracle
    over the same (quantized) weights."""
    s = RAGGED if shape == "ragged" else ODD
    ctx, host = mio.build_context(s, max_context=64, kv_dtype="f16", gain_scale=0.1, keep_host=True,
                                  weights=None if weights == "bf16" else weights, prefill_split=1)
    assert ctx.info().persistent_grid > 0
    prompt = ki.prompt_ids(s.vocab, 20, seed=95)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits)
    toks, lgs = [int(nxt.item())], [logits.cpu().numpy().copy()]
    for _ in range(6):
        ctx.decode_step(nxt, 1, nxt, logits)
        toks.append(int(nxt.item()))
        lgs.append(logits.cpu().numpy().copy())
    assert ctx.sync_status() == k2.K2_OK
    get = lambda n, l: host[(n, l)]  # noqa: E731
    wts = {"bf16": get, "f8": Q8.fp8_weights(get), "q4": Q4.q4_weights(get)}[weights]
    seq = np.concatenate([prompt, toks[:-1]])
    am, ref, _ = O.OracleModel(s, wts, "f16").teacher_forced(seq, len(prompt) - 1)
    got = np.stack(lgs).astype(np.float64)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel <= 2e-4, rel
    assert np.mean(am == np.array(toks)) == 1.0
