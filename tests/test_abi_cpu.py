"""Host-side checks of the C ABI: the library loads, exports every call that
include/k2.h declares, and validates configs and arguments before touching a
GPU.  No GPU is needed."""
import ctypes as C
import os
import re

import pytest

import k2_inputs as ki

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import build
    build.build()
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


def declared_calls():
    text = open(os.path.join(ROOT, "include", "k2.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(k2_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_call_is_exported(k2):
    names = declared_calls()
    assert len(names) >= 16
    for n in names:
        assert hasattr(k2.LIB, n), n
    assert set(k2.EXPORTED) == set(names)


def test_workspace_bytes_valid_and_invalid(k2):
    cfg = k2.make_config(ki.K2_3P7B, max_context=4096 + 256, max_batch=1, kv_dtype="f16")
    n = k2.workspace_bytes(cfg)
    # packed projections (every weight but the embedding) + fp16 KV
    # 36 x 2 x 8 x cap x 128 x 2 bytes
    cap = (4096 + 256 + 8 + 63) // 64 * 64
    kv = 36 * 2 * 8 * cap * 128 * 2
    packed = (36 * ((6144 + 2 * 10240) * 2560 + 2560 * 4096 + 2560 * 10240) + 250624 * 2560) * 2
    # tensor-core prefill buffers for blocks of 2048 tokens: fp32 residual,
    # bf16 hi/lo GEMM inputs (normed input / attention output, SwiGLU output),
    # fp32 QKV output and rotated queries
    P = 2048
    prefill = P * (2560 * 4 + 2 * 4096 * 2 + 2 * 10240 * 2 + 6144 * 4 + 4096 * 4)
    # and two layers' projections as fp16 (the fp16-operand prefill converts a layer ahead)
    prefill += 2 * (6144 * 2560 + 2560 * 4096 + 20480 * 2560 + 2560 * 10240) * 2
    assert packed + kv + prefill < n < packed + kv + prefill + 64 * 2 ** 20
    for bad in (dict(head_dim=96), dict(n_heads=30), dict(hidden=2561), dict(norm_groups=0),
                dict(vocab=0), dict(head_dim=127)):
        c = k2.make_config(ki.K2_3P7B.replace(**bad), max_context=4096)
        assert k2.workspace_bytes(c) == 0, bad
        assert k2.LIB.k2_last_error(None).decode() != ""
    c = k2.make_config(ki.K2_3P7B, max_context=4096, max_batch=65)
    assert k2.workspace_bytes(c) == 0


def test_init_refuses_bad_config_and_weights_without_a_gpu(k2):
    ctx = C.c_void_p()
    bad = k2.make_config(ki.K2_3P7B.replace(n_heads=30), max_context=64)
    w = k2.Weights()
    st = k2.LIB.k2_init_weights(C.byref(bad), C.byref(w), None, 0, None, C.byref(ctx))
    assert st == k2.K2_ERR_SHAPE and not ctx.value
    st = k2.LIB.k2_init_weights(C.byref(k2.make_config(ki.TINY.replace(head_dim=12), 64)), C.byref(w), None, 0,
                                None, C.byref(ctx))
    assert st == k2.K2_ERR_UNSUPPORTED
    good = k2.make_config(ki.TINY, max_context=64, kv_dtype="f32")
    st = k2.LIB.k2_init_weights(C.byref(good), C.byref(w), None, 0, None, C.byref(ctx))
    assert st == k2.K2_ERR_ARG and "embed" in k2.LIB.k2_last_error(None).decode()
    st = k2.LIB.k2_init_weights(C.byref(good), None, None, 0, None, C.byref(ctx))
    assert st == k2.K2_ERR_ARG


def test_calls_on_null_context_are_refused(k2):
    assert k2.LIB.k2_prefill(None, 0, None, 1, None, None, None) == k2.K2_ERR_ARG
    assert k2.LIB.k2_decode_step(None, None, 1, None, None, None) == k2.K2_ERR_ARG
    assert k2.LIB.k2_kv_reset(None, -1, None) == k2.K2_ERR_ARG
    assert k2.LIB.k2_sync_status(None, None) == k2.K2_ERR_ARG
    k2.LIB.k2_free(None)


def header_enum(name):
    """name -> value of the members of the typedef enum `name` in include/k2.h."""
    text = open(os.path.join(ROOT, "include", "k2.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef enum\s*\{([^}]*)\}\s*" + name + r"\s*;", text, flags=re.S).group(1)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(K2_[A-Z0-9_]+)\s*=\s*(\d+)", body)}


@pytest.mark.parametrize("enum", ["k2_status", "k2_dtype", "k2_option"])
def test_binding_constants_match_the_header(k2, enum):
    """Every status, dtype and option number the header declares has the same
    value in the Python binding (the binding passes bare integers)."""
    members = header_enum(enum)
    assert len(members) >= 6
    for n, v in members.items():
        assert getattr(k2, n) == v, n
