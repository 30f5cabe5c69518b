"""Tensor-core prefill (k2_prefill with bf16 weights) against the oracle and
against the same library appending the prompt one decode step per token.

Both GPU paths keep fp32 activations (the GEMM splits each activation into two
bf16 halves), so they agree far more tightly than the bf16 parity bars; the
oracle comparisons use the bars of tests/test_gpu_decode.py."""
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


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def prefill(k2, ctx, prompt, vocab, tc, split=1):
    """split: K2_OPT_PREFILL_SPLIT; 1 (bf16 hi + lo activations) unless a test
    asks for another mode: the 2e-4 bars of this file are that mode's."""
    ctx.set_option(k2.K2_OPT_TC_PREFILL, 1 if tc else 0)
    ctx.set_option(k2.K2_OPT_PREFILL_SPLIT, split)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(vocab, dtype=torch.float32, device="cuda")
    ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt, logits)
    torch.cuda.synchronize()
    return int(nxt.item()), logits.cpu().numpy()


def cache_rows(k2, ctx, s, kv, n):
    """K and V rows 0..n-1 of every layer, dequantised, as float64."""
    cap = ctx.info().kv_capacity
    nkv, d = s.n_kv_heads, s.head_dim
    out = []
    for layer in range(s.n_layers):
        kp, vp, ksp, vsp, _ = ctx.kv_view(layer, 0)
        for ptr, sptr in ((kp, ksp), (vp, vsp)):
            if kv == "i8":
                codes = k2.device_view(ptr, nkv * cap * d, torch.int8).view(nkv, cap, d)[:, :n].float()
                sc = k2.device_view(sptr, nkv * cap, torch.float16).view(nkv, cap)[:, :n].float()
                out.append((codes * sc[..., None]).cpu().numpy())
            else:
                dt = torch.float16 if kv == "f16" else torch.float32
                out.append(k2.device_view(ptr, nkv * cap * d, dt).view(nkv, cap, d)[:, :n].float().cpu().numpy())
    return np.stack(out).astype(np.float64)


@pytest.mark.parametrize("kv", ["f16", "i8", "f32"])
def test_tc_prefill_matches_stepwise_and_oracle(k2, mio, kv):
    s = ki.MEDIUM
    n = 200  # two 128-token tiles, the second ragged
    prompt = ki.prompt_ids(s.vocab, n, seed=31)
    res = {}
    for tc in (True, False):
        ctx, host = mio.build_context(s, max_context=256, kv_dtype=kv, gain_scale=0.1, keep_host=True)
        tok, lg = prefill(k2, ctx, prompt, s.vocab, tc)
        hid = k2.device_view(ctx.hidden_view(0), s.hidden, torch.float32).cpu().numpy().copy()
        res[tc] = (tok, lg, hid, cache_rows(k2, ctx, s, kv, n))
        assert ctx.info().kv_capacity >= n
        assert ctx.sync_status() == k2.K2_OK
        if tc:
            ref = O.OracleModel(s, lambda nm, l: host[(nm, l)], kv).forward_full(prompt)
    (t1, l1, h1, c1), (t0, l0, h0, c0) = res[True], res[False]
    assert t1 == t0 == O.argmax_first(ref)
    assert rel_l2(l1, ref) <= (2e-4 if kv != "i8" else 5e-2)
    # int8: the two paths' fp32 values (~1e-6 apart) pick different codes where
    # a value sits on a rounding boundary; one code step is 1/127 of the row max
    close = 1e-4 if kv != "i8" else 5e-3
    assert rel_l2(l1, l0) <= close
    assert rel_l2(h1, h0) <= close
    if kv == "i8":
        # codes may differ by one step where a value sits on a rounding boundary
        assert rel_l2(c1, c0) <= 2e-2
    elif kv == "f16":
        # fp16 storage: values ~1e-6 apart round to neighbouring halves now and
        # then; one ulp is 2^-11 relative, so even all of them flipping stays below
        assert rel_l2(c1, c0) <= 2.0 ** -11
    else:
        assert rel_l2(c1, c0) <= 1e-5


def test_tc_prefill_in_blocks_after_existing_rows(k2, mio):
    """A second prompt appended to a non-empty cache, longer than one 2048-token
    block, against the step-by-step path."""
    s = ki.MEDIUM
    first = ki.prompt_ids(s.vocab, 37, seed=41)
    second = ki.prompt_ids(s.vocab, 2100, seed=42)
    out = {}
    for tc in (True, False):
        ctx, _ = mio.build_context(s, max_context=2200, kv_dtype="f16", gain_scale=0.1)
        prefill(k2, ctx, first, s.vocab, tc)
        tok, lg = prefill(k2, ctx, second, s.vocab, tc)
        out[tc] = (tok, lg)
        assert ctx.kv_view(0, 0)[4] == len(first) + len(second)
        assert ctx.sync_status() == k2.K2_OK
    assert out[True][0] == out[False][0]
    assert rel_l2(out[True][1], out[False][1]) <= 2e-4


def test_tc_prefill_3p7b_layer_against_oracle(k2, mio):
    """One decoder layer of the 3.7B shape: a 300-token prompt through the
    tensor-core path against the oracle's full recompute."""
    s = ki.K2_LAYER
    n = 300
    prompt = ki.prompt_ids(s.vocab, n, seed=51)
    ctx, host = mio.build_context(s, max_context=512, kv_dtype="f16", keep_host=True)
    tok, lg = prefill(k2, ctx, prompt, s.vocab, True)
    ref = O.OracleModel(s, lambda nm, l: host[(nm, l)], "f16").forward_full(prompt)
    assert rel_l2(lg, ref) <= 2e-4
    assert tok == O.argmax_first(ref)
    assert ctx.sync_status() == k2.K2_OK


@pytest.mark.parametrize("kv", ["f16", "i8"])
def test_batched_decode_matches_one_token_at_a_time_and_oracle(k2, mio, kv):
    """Batch-4 decode (weights read once per step for all four sequences)
    against the same steps taken one sequence at a time, and sequences 0 and 3
    against the oracle teacher-forced."""
    s = ki.MEDIUM
    B, steps = 4, 10
    prompts = [ki.prompt_ids(s.vocab, n, seed=60 + b) for b, n in enumerate((23, 40, 9, 71))]
    runs = {}
    for batched in (True, False):
        ctx, host = mio.build_context(s, max_context=128, max_batch=B, kv_dtype=kv, gain_scale=0.1, keep_host=True,
                                      prefill_split=1)
        ctx.set_option(k2.K2_OPT_TC_DECODE, 1 if batched else 0)
        nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
        logits = torch.empty(B * s.vocab, dtype=torch.float32, device="cuda")
        for b, p in enumerate(prompts):
            ctx.prefill(b, torch.tensor(p, dtype=torch.int32, device="cuda"), nxt[b:b + 1])
        toks, lgs = [nxt.cpu().numpy().copy()], []
        for _ in range(steps):
            ctx.decode_step(nxt, B, nxt, logits)
            toks.append(nxt.cpu().numpy().copy())
            lgs.append(logits.view(B, s.vocab).cpu().numpy().copy())
        assert ctx.sync_status() == k2.K2_OK
        runs[batched] = (np.stack(toks), np.stack(lgs))
    (t1, l1), (t0, l0) = runs[True], runs[False]
    assert np.array_equal(t1, t0)
    assert rel_l2(l1, l0) <= (1e-4 if kv == "f16" else 5e-3)
    model = O.OracleModel(s, lambda nm, l: host[(nm, l)], kv)
    for b in (0, 3):
        seq = np.concatenate([prompts[b], t1[:-1, b]])
        am, ref, _ = model.teacher_forced(seq, len(prompts[b]))
        assert rel_l2(l1[:, b], ref) <= (2e-4 if kv == "f16" else 5e-2)
        assert np.mean(am == t1[1:, b]) >= (0.99 if kv == "f16" else 0.9)


@pytest.mark.parametrize("n", [8, 12, 16, 17])
def test_short_prompts_through_the_small_block_path(k2, mio, n):
    """Prompts of 8..16 tokens stream the weights with the 16-token-tile GEMMs
    (17 takes the 128-token tiles): against the step-by-step path."""
    s = ki.MEDIUM
    prompt = ki.prompt_ids(s.vocab, n, seed=70 + n)
    out = {}
    for tc in (True, False):
        ctx, _ = mio.build_context(s, max_context=64, kv_dtype="f16", gain_scale=0.1)
        out[tc] = prefill(k2, ctx, prompt, s.vocab, tc)
        assert ctx.sync_status() == k2.K2_OK
    assert out[True][0] == out[False][0]
    assert rel_l2(out[True][1], out[False][1]) <= 1e-4


@pytest.mark.parametrize("shape,first,n", [("k2_layer", 50, 1000), ("medium", 0, 333), ("medium", 129, 64)])
def test_tcgen05_prefill_attention_against_mma_sync_and_oracle(k2, mio, shape, first, n):
    """The prefill attention on the 5th-generation tensor cores (option
    K2_OPT_PREFILL_ATTN = 1, the default for fp16 caches) against the mma.sync
    kernel (= 0) and the oracle's full recompute: a prompt after `first` cached
    rows, so query blocks start mid-tile and the last key tile is partial."""
    s = ki.SHAPES[shape]
    pre = ki.prompt_ids(s.vocab, first, seed=91) if first else None
    prompt = ki.prompt_ids(s.vocab, n, seed=92)
    out = {}
    for tc_attn in (1, 0):
        ctx, host = mio.build_context(s, max_context=first + n + 8, kv_dtype="f16", gain_scale=0.1, keep_host=True)
        ctx.set_option(k2.K2_OPT_PREFILL_ATTN, tc_attn)
        if pre is not None:
            prefill(k2, ctx, pre, s.vocab, True)
        out[tc_attn] = prefill(k2, ctx, prompt, s.vocab, True)
        assert ctx.sync_status() == k2.K2_OK
    seq = prompt if pre is None else np.concatenate([pre, prompt])
    ref = O.OracleModel(s, lambda nm, l: host[(nm, l)], "f16").forward_full(seq)
    (t1, l1), (t0, l0) = out[1], out[0]
    assert rel_l2(l1, ref) <= 2e-4
    assert rel_l2(l0, ref) <= 2e-4
    assert rel_l2(l1, l0) <= 1e-4
    assert t1 == t0 == O.argmax_first(ref)


@pytest.mark.parametrize("kv", ["f16", "i8"])
@pytest.mark.parametrize("shape,first,n", [("k2_layer", 50, 1000), ("medium", 0, 333), ("medium", 129, 64)])
def test_prefill_without_split_against_oracle(k2, mio, kv, shape, first, n):
    """K2_OPT_PREFILL_SPLIT = 0: the prefill GEMMs take single bf16 activations
    and the tcgen05 attention (fp16 caches) single fp16 queries and
    probabilities.  Held to the bf16 bars (relative L2 <= 2e-2 with fp16 KV,
    5e-2 with int8) against the oracle's full recompute, and to the same
    argmax; the split run of the same prompt is printed beside it."""
    s = ki.SHAPES[shape]
    pre = ki.prompt_ids(s.vocab, first, seed=91) if first else None
    prompt = ki.prompt_ids(s.vocab, n, seed=92)
    out = {}
    for split in (1, 0):
        ctx, host = mio.build_context(s, max_context=first + n + 8, kv_dtype=kv, gain_scale=0.1, keep_host=True)
        if pre is not None:
            prefill(k2, ctx, pre, s.vocab, True, split)
        out[split] = prefill(k2, ctx, prompt, s.vocab, True, split)
        assert ctx.sync_status() == k2.K2_OK
    seq = prompt if pre is None else np.concatenate([pre, prompt])
    ref = O.OracleModel(s, lambda nm, l: host[(nm, l)], kv).forward_full(seq)
    (t1, l1), (t0, l0) = out[1], out[0]
    r1, r0 = rel_l2(l1, ref), rel_l2(l0, ref)
    print(f"{shape} kv={kv} first={first} n={n}: split rel_l2={r1:.3e}, single rel_l2={r0:.3e}")
    assert r0 <= (2e-2 if kv == "f16" else 5e-2)
    assert t0 == O.argmax_first(ref)


@pytest.mark.parametrize("split", [1, 3])
@pytest.mark.parametrize("shape,first,n", [("k2_layer", 50, 1000), ("medium", 0, 333), ("medium", 129, 2100)])
def test_persistent_prefill_gemm_against_per_tile_and_oracle(k2, mio, shape, first, n, split):
    """K2_OPT_PREFILL_GEMM: QKV and gate/up on the persistent kernel over whole
    tiles (1, the default: the SwiGLU epilogue of one tile overlaps the next
    tile's K steps; 256-token tiles for fp16 blocks over 512 tokens) against
    one CTA per tile (0) and the oracle's full recompute; ragged token tiles,
    and a prompt longer than one 2048-token block after cached rows.  split:
    the bf16 hi + lo activations (1) or single fp16 operands (3, whose bars are
    those of test_fp16_operand_prefill_against_oracle)."""
    s = ki.SHAPES[shape]
    pre = ki.prompt_ids(s.vocab, first, seed=93) if first else None
    prompt = ki.prompt_ids(s.vocab, n, seed=94)
    out = {}
    for mode in (1, 0):
        ctx, host = mio.build_context(s, max_context=first + n + 8, kv_dtype="f16", gain_scale=0.1, keep_host=True)
        ctx.set_option(k2.K2_OPT_PREFILL_GEMM, mode)
        if pre is not None:
            prefill(k2, ctx, pre, s.vocab, True, split)
        tok, lg = prefill(k2, ctx, prompt, s.vocab, True, split)
        hid = k2.device_view(ctx.hidden_view(0), s.hidden, torch.float32).cpu().numpy().copy()
        out[mode] = (tok, lg, hid)
        assert ctx.sync_status() == k2.K2_OK
    seq = prompt if pre is None else np.concatenate([pre, prompt])
    ref = O.OracleModel(s, lambda nm, l: host[(nm, l)], "f16").forward_full(seq)
    (t1, l1, h1), (t0, l0, h0) = out[1], out[0]
    bar = 2e-4 if split == 1 else 5e-3
    assert rel_l2(l1, ref) <= bar
    assert rel_l2(l0, ref) <= bar
    # the same products; the tile shapes, the order of the fp32 additions and
    # (fp16) the activations they round differ: well inside the bars' margin
    close = 1e-4 if split == 1 else 2e-3
    assert rel_l2(l1, l0) <= close
    assert rel_l2(h1, h0) <= close
    assert t1 == t0 == O.argmax_first(ref)


@pytest.mark.parametrize("shape,first,n", [("k2_layer", 50, 1000), ("medium", 0, 333), ("medium", 129, 2100),
                                           ("medium", 0, 512), ("medium", 7, 513)])
def test_fp16_operand_prefill_against_oracle(k2, mio, shape, first, n):
    """K2_OPT_PREFILL_SPLIT = 3: every prefill contraction on single fp16
    operands (each weight matrix converted to fp16 per layer, fp16 activations,
    queries and probabilities).  fp16 keeps 11 significant bits (unit roundoff
    2^-11 = 4.9e-4); each layer rounds its four GEMM inputs and the attention's
    queries and probabilities once, so the logits are held to 5e-3 of the
    oracle's full recompute (10 roundoffs) and to the same argmax; the split
    run (1) of the same prompt stays within 2e-4.  Blocks of more than 512
    tokens take 256-token GEMM tiles: 512 and 513 tokens sit on either side."""
    s = ki.SHAPES[shape]
    pre = ki.prompt_ids(s.vocab, first, seed=95) if first else None
    prompt = ki.prompt_ids(s.vocab, n, seed=96)
    out = {}
    for split in (3, 1):
        ctx, host = mio.build_context(s, max_context=first + n + 8, kv_dtype="f16", gain_scale=0.1, keep_host=True)
        if pre is not None:
            prefill(k2, ctx, pre, s.vocab, True, split)
        out[split] = prefill(k2, ctx, prompt, s.vocab, True, split)
        assert ctx.sync_status() == k2.K2_OK
    seq = prompt if pre is None else np.concatenate([pre, prompt])
    ref = O.OracleModel(s, lambda nm, l: host[(nm, l)], "f16").forward_full(seq)
    (t3, l3), (t1, l1) = out[3], out[1]
    r3, r1 = rel_l2(l3, ref), rel_l2(l1, ref)
    print(f"{shape} first={first} n={n}: fp16 rel_l2={r3:.3e}, split rel_l2={r1:.3e}")
    assert r3 <= 5e-3
    assert r1 <= 2e-4
    assert t3 == t1 == O.argmax_first(ref)


def test_fp16_operand_prefill_flags_weights_beyond_fp16(k2, mio):
    """A weight beyond fp16's range (1e5 in one W_up entry): the fp16-operand
    prefill raises the device guard ("beyond-fp16-range") instead of running on
    an infinity; the split prefill of the same model does not."""
    s = ki.MEDIUM
    prompt = ki.prompt_ids(s.vocab, 100, seed=97)
    for split in (3, 1):
        dev, _ = mio.device_weights(s, gain_scale=0.1)
        dev["w_up"][0][0, 0] = 1.0e5
        ctx = k2.Context(k2.make_config(s, max_context=128, kv_dtype="f16"), dev)
        ctx.set_option(k2.K2_OPT_PREFILL_SPLIT, split)
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        ctx.prefill(0, torch.tensor(prompt, dtype=torch.int32, device="cuda"), nxt)
        torch.cuda.synchronize()
        st = ctx.sync_status()
        if split == 3:
            assert st == k2.K2_ERR_DEVICE_GUARD
            assert "beyond-fp16-range" in ctx.last_error()
        else:
            assert st == k2.K2_OK
