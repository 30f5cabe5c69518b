"""The full 36-layer 3.7B-shape model (bf16 random-init weights, vocab 250624,
untied lm_head, fp16 KV): prefill of 512 random token ids, then 256 greedy
decode steps, against the oracle's teacher-forced pass over the emitted
sequence (kimi-k3-in-c k3_run.c, --tf-check: prediction i is the argmax after
tokens 0..i).

Bars: teacher-forced argmax agreement >= 99 % and logits relative L2 <= 2e-2
(the bf16 + fp16-KV bars).  The GPU keeps fp32 activations, so the logits are
also held to 1e-3: over 36 layers the remaining differences are fp32
summation order and K/V values that round to neighbouring fp16 numbers on the
two sides (one fp16 ulp is 2^-11 relative); measured 4.3e-4."""
import numpy as np
import pytest
import torch

import k2_inputs as ki
from oracle import k2_oracle as O

pytestmark = pytest.mark.gpu


_ORACLE = {}


def _teacher_forced(s, host, seq, start):
    key = tuple(int(t) for t in seq)
    if key not in _ORACLE:
        _ORACLE[key] = O.OracleModel(s, lambda n, l: host[(n, l)], "f16").teacher_forced(seq, start)
    return _ORACLE[key]


@pytest.mark.parametrize("split", [1, 0, 2, 3])
def test_full_3p7b_prefill512_decode256_teacher_forced(split):
    """split = 0 (K2_OPT_PREFILL_SPLIT off): the 512-token prefill feeds the
    GEMMs single bf16 activations and the attention single fp16 queries and
    probabilities; the decode steps keep fp32 activations.  That mode does not
    hold the bf16 bars on this 36-layer model -- measured: agreement 0.949-0.965,
    logits relative L2 1.1e-2 over the 257 predictions and 2.1e-2 on the
    prefill's own logits -- which is why the split is the default.  The test
    keeps the measured cost of dropping it bounded (agreement >= 0.9, relative
    L2 <= 3e-2), holds split = 1 to the bars and to 1e-3, and split = 2 (the
    GEMMs split, the attention single) and split = 3 (single fp16 operands
    throughout: fp16 copies of the weights, fp16 activations) to the bars."""
    from dense_gqa_decoder_gb300 import k2, model_io
    s = ki.K2_3P7B
    n_prompt, n_new = 512, 256
    ctx, host = model_io.build_context(s, max_context=n_prompt + n_new + 8, kv_dtype="f16", keep_host=True)
    ctx.set_option(k2.K2_OPT_PREFILL_SPLIT, split)
    prompt = ki.prompt_ids(s.vocab, n_prompt, seed=1)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits)
    toks, lgs = [int(nxt.item())], [logits.cpu().numpy().copy()]
    for _ in range(n_new):
        ctx.decode_step(nxt, 1, nxt, logits)
        toks.append(int(nxt.item()))
        lgs.append(logits.cpu().numpy().copy())
    assert ctx.sync_status() == k2.K2_OK
    del ctx
    torch.cuda.empty_cache()
    seq = np.concatenate([prompt, toks[:-1]])
    am, lg_ref, _ = _teacher_forced(s, host, seq, n_prompt - 1)
    got = np.stack(lgs).astype(np.float64)
    rel = float(np.linalg.norm(got - lg_ref) / np.linalg.norm(lg_ref))
    rel_first = float(np.linalg.norm(got[0] - lg_ref[0]) / np.linalg.norm(lg_ref[0]))
    agree = float(np.mean(am == np.array(toks)))
    print(f"split={split} rel_l2={rel:.3e} rel_l2_prefill_logits={rel_first:.3e} agreement={agree:.4f}")
    if split == 1:
        assert agree >= 0.99, agree
        assert rel <= 2e-2
        assert rel <= 1e-3, rel
    elif split in (2, 3):
        # 2: the GEMMs split, the attention's queries and probabilities single
        # fp16; 3: every prefill contraction on single fp16 operands
        assert agree >= 0.99, agree
        assert rel <= 2e-2, rel
    else:
        # this mode's ~1e-2 error lets a last-bit difference (the order of the
        # stream-K GEMMs' fp32 atomic additions) flip a greedy token, and the
        # sequence generated from there differs run to run: 0.949 - 0.965 measured
        assert agree >= 0.9, agree
        assert rel <= 3e-2, rel
