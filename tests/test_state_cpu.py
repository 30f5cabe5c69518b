"""Saved cache state: the header check of k2_kv_peek, without a GPU.

A state is written here by hand from the layout documented in include/k2.h
(not by the library), so these tests pin the format itself: the fingerprint
of the model architecture and KV format, the size arithmetic, and every
refusal (kimi-k3-in-c k3_run.c, "conversation state": a state written for a
different architecture is refused; only occupied positions are stored, so the
restoring context may size its cache differently)."""
import struct

import pytest

import k2_inputs as ki

HDR = 96


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import build
    build.build()
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


def fingerprint(cfg):
    f2i = lambda x: struct.unpack("<i", struct.pack("<f", x))[0]
    return [cfg.hidden, cfg.n_layers, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate,
            cfg.norm_groups, cfg.vocab, cfg.weight_dtype, cfg.kv_dtype, f2i(cfg.eps), f2i(cfg.rope_theta)]


def layout(cfg, cached, n_tokens):
    """(row bytes, scale bytes, offset of layer 0, bytes per layer, total)."""
    elt = {0: 4, 1: 2, 2: 2, 3: 1}[cfg.kv_dtype]
    row = cfg.head_dim * elt
    scale = 2 if cfg.kv_dtype == 3 else 0
    kv_off = (HDR + 4 * n_tokens + 15) // 16 * 16
    rows = cfg.n_kv_heads * cached
    per_layer = (2 * rows * row + 2 * rows * scale + 15) // 16 * 16
    return row, scale, kv_off, per_layer, kv_off + cfg.n_layers * per_layer


def make_state(cfg, cached, tokens, fp=None, magic=b"K2ST", version=1, sizes=None):
    row, scale, kv_off, per_layer, total = layout(cfg, cached, len(tokens))
    if sizes is not None:
        row, scale, total = sizes
    h = magic + struct.pack("<i", version) + struct.pack("<12i", *(fp or fingerprint(cfg)))
    h += struct.pack("<ii", cached, len(tokens)) + struct.pack("<qqq", row, scale, total) + struct.pack("<ii", 0, 0)
    assert len(h) == HDR
    body = bytes(range(256)) * ((total - HDR) // 256 + 1)
    data = h + struct.pack(f"<{len(tokens)}i", *tokens) + body
    return bytearray(data[:layout(cfg, cached, len(tokens))[4]])


def peek(k2, cfg, data):
    import torch
    return k2.peek_state(cfg, torch.frombuffer(bytearray(data), dtype=torch.uint8) if len(data) else
                         torch.zeros(0, dtype=torch.uint8))


@pytest.mark.parametrize("kv", ["f16", "i8", "f32"])
def test_peek_accepts_a_state_written_from_the_documented_layout(k2, kv):
    cfg = k2.make_config(ki.MEDIUM, max_context=300, kv_dtype=kv)
    data = make_state(cfg, 123, [5, 7, 11])
    assert peek(k2, cfg, data) == (123, 3)
    # the restoring context may have another max_context / max_batch (not in the fingerprint)
    other = k2.make_config(ki.MEDIUM, max_context=64, max_batch=4, kv_dtype=kv)
    assert peek(k2, other, data) == (123, 3)
    # an empty cache with no tokens is a valid state too
    assert peek(k2, cfg, make_state(cfg, 0, [])) == (0, 0)


def test_layout_sizes_of_the_3p7b_shape(k2):
    # 36 layers x 8 KV heads x 4096 rows x (K + V) x 256 bytes = the fp16 KV of a 4096-token context
    cfg = k2.make_config(ki.K2_3P7B, max_context=4200, kv_dtype="f16")
    row, scale, kv_off, per_layer, total = layout(cfg, 4096, 10)
    assert (row, scale, kv_off) == (256, 0, 144)
    assert total - kv_off == 147456 * 4096
    cfg8 = k2.make_config(ki.K2_3P7B, max_context=4200, kv_dtype="i8")
    assert layout(cfg8, 4096, 0)[4] - HDR == 36 * 8 * 4096 * 2 * (128 + 2)


@pytest.mark.parametrize("field,value", [(1, 35), (3, 4), (4, 128), (7, 1001), (8, 0), (9, 2), (10, 0), (11, 0)])
def test_peek_refuses_another_architecture_or_kv_format(k2, field, value):
    cfg = k2.make_config(ki.MEDIUM, max_context=300, kv_dtype="i8")
    fp = fingerprint(cfg)
    assert fp[field] != value
    fp[field] = value
    assert peek(k2, cfg, make_state(cfg, 40, [1], fp=fp)) == (-1, -1)


def test_peek_refuses_damaged_or_foreign_buffers(k2):
    cfg = k2.make_config(ki.MEDIUM, max_context=300, kv_dtype="f16")
    good = make_state(cfg, 40, [1, 2])
    assert peek(k2, cfg, good) == (40, 2)
    assert peek(k2, cfg, make_state(cfg, 40, [1, 2], magic=b"K3ST")) == (-1, -1)
    assert peek(k2, cfg, make_state(cfg, 40, [1, 2], version=2)) == (-1, -1)
    assert peek(k2, cfg, good[:-1]) == (-1, -1)           # truncated body
    assert peek(k2, cfg, good[:HDR - 1]) == (-1, -1)      # truncated header
    assert peek(k2, cfg, b"") == (-1, -1)
    row, scale, _, _, total = layout(cfg, 40, 2)
    assert peek(k2, cfg, make_state(cfg, 40, [1, 2], sizes=(row + 2, scale, total))) == (-1, -1)
    assert peek(k2, cfg, make_state(cfg, 40, [1, 2], sizes=(row, 2, total))) == (-1, -1)
    assert peek(k2, cfg, make_state(cfg, 40, [1, 2], sizes=(row, scale, total + 16))) == (-1, -1)
    bad = bytearray(good)
    bad[56:60] = struct.pack("<i", -1)                      # negative row count
    assert peek(k2, cfg, bad) == (-1, -1)
    bad = bytearray(good)
    bad[88:92] = struct.pack("<i", 1)                       # reserved word set
    assert peek(k2, cfg, bad) == (-1, -1)
