"""Thin ctypes binding of libk2 (include/k2.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of libk2.so.  torch is used for device memory and streams.  If the
library is missing the import fails loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libk2.so")

K2_OK, K2_ERR_ARG, K2_ERR_SHAPE, K2_ERR_UNSUPPORTED, K2_ERR_TOKEN_RANGE, K2_ERR_CONTEXT_FULL, \
    K2_ERR_WORKSPACE, K2_ERR_CUDA, K2_ERR_DEVICE_GUARD, K2_ERR_STATE = range(10)
K2_STATE_HEADER_BYTES = 96
K2_F32, K2_BF16, K2_F16, K2_I8, K2_F8, K2_Q4 = range(6)
(K2_OPT_PDL, K2_OPT_GRAPH, K2_OPT_ATTN_SPLITS, K2_OPT_PERSISTENT, K2_OPT_TC_PREFILL, K2_OPT_TC_DECODE,
 K2_OPT_WAIT_LIMIT_US, K2_OPT_STALL_PHASE, K2_OPT_L2_AHEAD, K2_OPT_L2_AHEAD_PHASES, K2_OPT_TRACE,
 K2_OPT_PREFILL_ATTN, K2_OPT_PREFILL_SPLIT, K2_OPT_PREFILL_GEMM) = range(14)
KERNEL_CLASSES = ("embed", "qkv", "attn", "o_proj", "gate_up", "down", "lm_head", "step", "sample")
DTYPES = {"f32": K2_F32, "bf16": K2_BF16, "f16": K2_F16, "i8": K2_I8, "f8": K2_F8, "q4": K2_Q4}


class K2Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"k2 status {status}: {msg}")
        self.status = status


class Config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "hidden", "n_layers", "n_heads", "n_kv_heads", "head_dim", "intermediate", "norm_groups", "vocab",
        "max_context", "max_batch")] + [("eps", C.c_float), ("rope_theta", C.c_float),
                                        ("weight_dtype", C.c_int32), ("kv_dtype", C.c_int32)]


_PP = C.POINTER(C.c_void_p)


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p)] + [
        (n, _PP) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")]


class Info(C.Structure):
    _fields_ = [("kv_capacity", C.c_int32), ("num_sms", C.c_int32), ("attn_splits", C.c_int32),
                ("gemv_grid", C.c_int32), ("kv_bytes", C.c_int64), ("repack_bytes", C.c_int64),
                ("scratch_bytes", C.c_int64), ("persistent_grid", C.c_int32), ("persistent_splits", C.c_int32),
                ("tc_prefill", C.c_int32), ("tc_batched", C.c_int32)]


class Sampling(C.Structure):
    _fields_ = [("temperature", C.c_float), ("top_k", C.c_int32), ("top_p", C.c_float), ("min_p", C.c_float),
                ("repetition_penalty", C.c_float), ("seed", C.c_uint64)]


def sampling(temperature=0.0, top_k=0, top_p=1.0, min_p=0.0, repetition_penalty=1.0, seed=0) -> Sampling:
    return Sampling(temperature=temperature, top_k=top_k, top_p=top_p, min_p=min_p,
                    repetition_penalty=repetition_penalty, seed=seed)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libk2.so is not built ({LIB_PATH}); run dense_gqa_decoder_gb300.build")
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
    sig = {
        "k2_workspace_bytes": (C.c_size_t, [C.POINTER(Config)]),
        "k2_init_weights": (C.c_int, [C.POINTER(Config), C.POINTER(Weights), vp, C.c_size_t, vp, C.POINTER(vp)]),
        "k2_free": (None, [vp]),
        "k2_last_error": (C.c_char_p, [vp]),
        "k2_get_info": (C.c_int, [vp, C.POINTER(Info)]),
        "k2_prefill": (C.c_int, [vp, i32, vp, i32, vp, vp, vp]),
        "k2_decode_step": (C.c_int, [vp, vp, i32, vp, vp, vp]),
        "k2_decode_layers": (C.c_int, [vp, vp, i32, vp]),
        "k2_kv_reset": (C.c_int, [vp, i32, vp]),
        "k2_kv_set_len": (C.c_int, [vp, i32, i32, vp]),
        "k2_kv_view": (C.c_int, [vp, i32, i32, C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), C.POINTER(vp),
                                 C.POINTER(i32)]),
        "k2_hidden_view": (C.c_int, [vp, i32, C.POINTER(vp)]),
        "k2_sync_status": (C.c_int, [vp, vp]),
        "k2_clear_status": (C.c_int, [vp, vp]),
        "k2_set_option": (C.c_int, [vp, i32, i64]),
        "k2_profile_decode": (C.c_int, [vp, vp, i32, vp, C.POINTER(C.c_float), C.POINTER(i32), vp]),
        "k2_greedy_head_noalloc": (C.c_int, [C.POINTER(Config), vp, vp, vp, vp, vp, vp]),
        "k2_kv_state_bytes": (C.c_int, [vp, i32, i32, C.POINTER(C.c_size_t)]),
        "k2_kv_save": (C.c_int, [vp, i32, vp, i32, vp, C.c_size_t, C.POINTER(C.c_size_t), vp]),
        "k2_kv_peek": (C.c_int, [C.POINTER(Config), vp, C.c_size_t, C.POINTER(i32), C.POINTER(i32)]),
        "k2_kv_load": (C.c_int, [vp, i32, vp, C.c_size_t, vp, i32, vp]),
        "k2_set_sampling": (C.c_int, [vp, C.POINTER(Sampling)]),
        "k2_sample_logits": (C.c_int, [vp, vp, i32, vp, i32, vp, vp, i32, vp, vp]),
        "k2_philox": (C.c_int, [C.c_uint32, i32, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint64, vp, vp]),
        "k2_spec_draft": (i32, [vp, i32, i32, vp]),
        "k2_quantize_fp8": (C.c_int, [vp, i32, i32, vp, vp, vp]),
        "k2_quantize_q4": (C.c_int, [vp, i32, i32, vp, vp, vp]),
        "k2_decode_speculative": (C.c_int, [vp, i32, vp, i32, i32, vp, C.POINTER(i32), vp]),
        "k2_spec_logits_view": (C.c_int, [vp, C.POINTER(vp), C.POINTER(i32)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


LIB = _load()
EXPORTED = ("k2_workspace_bytes", "k2_init_weights", "k2_free", "k2_last_error", "k2_get_info", "k2_prefill",
            "k2_decode_step", "k2_decode_layers", "k2_kv_reset", "k2_kv_set_len", "k2_kv_view", "k2_hidden_view",
            "k2_sync_status", "k2_clear_status", "k2_set_option", "k2_profile_decode", "k2_greedy_head_noalloc",
            "k2_kv_state_bytes", "k2_kv_save", "k2_kv_peek", "k2_kv_load", "k2_set_sampling", "k2_sample_logits",
            "k2_philox", "k2_spec_draft", "k2_decode_speculative", "k2_quantize_fp8",
            "k2_quantize_q4", "k2_spec_logits_view")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_config(shape, max_context: int, max_batch: int = 1, kv_dtype: str = "f16", weights: str = None) -> Config:
    """weights: the stored weight dtype, default the shape's; "f8" stores the
    shape's bf16 weights as fp8 E4M3 rows with per-row scales, "q4" as int4
    codes with one scale per 64 weights of a row."""
    return Config(hidden=shape.hidden, n_layers=shape.n_layers, n_heads=shape.n_heads, n_kv_heads=shape.n_kv_heads,
                  head_dim=shape.head_dim, intermediate=shape.intermediate, norm_groups=shape.norm_groups,
                  vocab=shape.vocab, max_context=max_context, max_batch=max_batch, eps=shape.eps,
                  rope_theta=shape.rope_theta, weight_dtype=DTYPES[weights or shape.weight_dtype],
                  kv_dtype=DTYPES[kv_dtype])


def workspace_bytes(cfg: Config) -> int:
    return int(LIB.k2_workspace_bytes(C.byref(cfg)))


class Context:
    """Owns a k2_ctx plus the torch tensors whose memory it uses (workspace,
    weights).  Methods mirror the C calls of the same name (k2_ prefix dropped)."""

    def __init__(self, cfg: Config, weights: dict, stream=None):
        self.cfg = cfg
        self.weights = weights  # keeps device memory alive
        nbytes = workspace_bytes(cfg)
        if nbytes == 0:
            raise K2Error(K2_ERR_ARG, "invalid config: " + (LIB.k2_last_error(None) or b"").decode())
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        L = cfg.n_layers
        arrs = {}
        for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"):
            arrs[n] = (C.c_void_p * L)(*[_ptr(weights[n][l]) for l in range(L)])
        self._arrs = arrs
        w = Weights(embed=_ptr(weights["embed"]), lm_head=_ptr(weights["lm_head"]),
                    final_norm=_ptr(weights["final_norm"]),
                    **{n: C.cast(a, _PP) for n, a in arrs.items()})
        ctx = C.c_void_p()
        st = LIB.k2_init_weights(C.byref(cfg), C.byref(w), _ptr(self.workspace), nbytes, _stream(stream),
                                 C.byref(ctx))
        if st != K2_OK:
            raise K2Error(st, (LIB.k2_last_error(None) or b"").decode())
        self.ctx = ctx

    def __del__(self):
        ctx = getattr(self, "ctx", None)
        if ctx:
            LIB.k2_free(ctx)
            self.ctx = None

    def _check(self, st):
        if st != K2_OK:
            raise K2Error(st, LIB.k2_last_error(self.ctx).decode())

    def last_error(self) -> str:
        return LIB.k2_last_error(self.ctx).decode()

    def info(self) -> Info:
        i = Info()
        self._check(LIB.k2_get_info(self.ctx, C.byref(i)))
        return i

    def prefill(self, seq, tokens, next_token, logits=None, stream=None):
        self._check(LIB.k2_prefill(self.ctx, seq, _ptr(tokens), tokens.numel(), _ptr(next_token), _ptr(logits),
                                   _stream(stream)))

    def decode_step(self, tokens, batch, next_tokens, logits=None, stream=None):
        self._check(LIB.k2_decode_step(self.ctx, _ptr(tokens), batch, _ptr(next_tokens), _ptr(logits),
                                       _stream(stream)))

    def decode_layers(self, x, batch, stream=None):
        self._check(LIB.k2_decode_layers(self.ctx, _ptr(x), batch, _stream(stream)))

    def kv_reset(self, seq=-1, stream=None):
        self._check(LIB.k2_kv_reset(self.ctx, seq, _stream(stream)))

    def kv_set_len(self, seq, n, stream=None):
        self._check(LIB.k2_kv_set_len(self.ctx, seq, n, _stream(stream)))

    def kv_view(self, layer, seq):
        k, v, ks, vs = C.c_void_p(), C.c_void_p(), C.c_void_p(), C.c_void_p()
        n = C.c_int32()
        self._check(LIB.k2_kv_view(self.ctx, layer, seq, C.byref(k), C.byref(v), C.byref(ks), C.byref(vs),
                                   C.byref(n)))
        return k.value, v.value, ks.value, vs.value, n.value

    def hidden_view(self, b=0):
        p = C.c_void_p()
        self._check(LIB.k2_hidden_view(self.ctx, b, C.byref(p)))
        return p.value

    def spec_logits(self):
        """k2_spec_logits_view: the logits of the last speculative step as a
        [rows, vocab] float32 CUDA tensor view (not a copy)."""
        p, rows = C.c_void_p(), C.c_int32(0)
        self._check(LIB.k2_spec_logits_view(self.ctx, C.byref(p), C.byref(rows)))
        if rows.value == 0:
            return torch.empty(0, self.cfg.vocab, dtype=torch.float32, device="cuda")
        return device_view(p.value, rows.value * self.cfg.vocab, torch.float32).view(rows.value, self.cfg.vocab)

    def sync_status(self, stream=None):
        return LIB.k2_sync_status(self.ctx, _stream(stream))

    def clear_status(self, stream=None):
        self._check(LIB.k2_clear_status(self.ctx, _stream(stream)))

    def set_option(self, opt, value):
        self._check(LIB.k2_set_option(self.ctx, opt, value))

    def set_sampling(self, params=None):
        """k2_set_sampling: a Sampling (see sampling()) or None for greedy."""
        self._check(LIB.k2_set_sampling(self.ctx, C.byref(params) if params is not None else None))

    def sample_logits(self, logits, rows, positions, next_tokens, seen=None, seen_len=None, first_seq=0,
                      stream=None):
        """k2_sample_logits on device tensors: logits [rows, vocab] fp32, positions
        and next_tokens [rows] int32, seen [rows, stride] / seen_len [rows] int32."""
        stride = seen.shape[-1] if seen is not None else 0
        self._check(LIB.k2_sample_logits(self.ctx, _ptr(logits), rows, _ptr(seen), stride, _ptr(seen_len),
                                         _ptr(positions), first_seq, _ptr(next_tokens), _stream(stream)))

    def decode_speculative(self, seq, tokens, max_draft=8, stream=None):
        """k2_decode_speculative: `tokens` = the cached ids + the next input (a
        contiguous numpy int32 array is passed without a copy); returns the
        emitted greedy ids (the last one is the next input)."""
        import numpy as np
        if isinstance(tokens, np.ndarray) and tokens.dtype == np.int32 and tokens.flags.c_contiguous:
            ids, n_ids = tokens.ctypes.data, tokens.size
        else:
            arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
            ids, n_ids = arr.ctypes.data, arr.size
        out = (C.c_int32 * (max(max_draft, 0) + 1))()
        n = C.c_int32(0)
        self._check(LIB.k2_decode_speculative(self.ctx, seq, ids, n_ids, max_draft, out, C.byref(n),
                                              _stream(stream)))
        return list(out[:n.value])

    def kv_state_bytes(self, seq, n_tokens=0):
        n = C.c_size_t()
        st = LIB.k2_kv_state_bytes(self.ctx, seq, n_tokens, C.byref(n))
        if st != K2_OK:
            raise K2Error(st, "kv_state_bytes: bad seq or n_tokens")
        return n.value

    def kv_save(self, seq, tokens=(), out=None, stream=None):
        """k2_kv_save into `out` (a uint8 CPU tensor, pinned copies fastest) or
        a new pinned buffer; returns the uint8 tensor holding the state."""
        ids = torch.as_tensor(list(tokens) if not torch.is_tensor(tokens) else tokens.cpu(),
                              dtype=torch.int32).contiguous()
        n = self.kv_state_bytes(seq, ids.numel())
        if out is None:
            out = torch.empty(n, dtype=torch.uint8).pin_memory()
        wrote = C.c_size_t()
        self._check(LIB.k2_kv_save(self.ctx, seq, ids.data_ptr() if ids.numel() else None, ids.numel(),
                                   out.data_ptr(), out.numel(), C.byref(wrote), _stream(stream)))
        return out[:wrote.value]

    def kv_load(self, seq, state, stream=None):
        """k2_kv_load from a uint8 CPU tensor; returns the saved token ids."""
        state = state.contiguous()
        cached, n_tok = peek_state(self.cfg, state)  # sizes the token buffer; the load re-checks
        ids = torch.empty(max(n_tok, 0), dtype=torch.int32)
        self._check(LIB.k2_kv_load(self.ctx, seq, state.data_ptr(), state.numel(),
                                   ids.data_ptr() if n_tok > 0 else None, max(n_tok, 0), _stream(stream)))
        return ids.tolist()

    def profile_decode(self, tokens, batch, next_tokens, stream=None):
        ms = (C.c_float * len(KERNEL_CLASSES))()
        n = (C.c_int32 * len(KERNEL_CLASSES))()
        self._check(LIB.k2_profile_decode(self.ctx, _ptr(tokens), batch, _ptr(next_tokens), ms, n,
                                          _stream(stream)))
        return dict(zip(KERNEL_CLASSES, ms)), dict(zip(KERNEL_CLASSES, n))


def greedy_head_noalloc(cfg: Config, lm_head, final_norm, x, logits, token, stream=None) -> int:
    """k2_greedy_head_noalloc: returns the k2 status (no context, no workspace).

    The tensors are checked here, since the C call reads raw pointers: x
    float32, logits float32 or None, token int32, lm_head and final_norm in
    the config's weight dtype, all contiguous CUDA tensors holding at least
    the elements the call touches (x and final_norm: hidden, lm_head:
    vocab * hidden, logits: vocab, token: 1); the call itself checks the
    config's shape.  A token of -1 after the call means a NaN logit or a
    bounded wait that ran out on the device.  ``x = None`` passes a null
    pointer through (the call refuses it)."""
    wdt = {K2_F32: torch.float32, K2_BF16: torch.bfloat16}.get(cfg.weight_dtype)

    def want(t, name, dtype, numel):
        if t is None:
            return
        if not (t.is_cuda and t.is_contiguous() and t.dtype == dtype and t.numel() >= numel):
            raise ValueError(f"greedy_head_noalloc: {name} must be a contiguous CUDA {dtype} tensor "
                             f"of at least {numel} elements, got {t.dtype} {tuple(t.shape)} on {t.device}")
    if wdt is not None:
        want(lm_head, "lm_head", wdt, cfg.vocab * cfg.hidden)
        want(final_norm, "final_norm", wdt, cfg.hidden)
    if cfg.hidden > 0 and cfg.vocab > 0:
        want(x, "x", torch.float32, cfg.hidden)
        want(logits, "logits", torch.float32, cfg.vocab)
    want(token, "token", torch.int32, 1)
    return LIB.k2_greedy_head_noalloc(C.byref(cfg), _ptr(lm_head), _ptr(final_norm), _ptr(x), _ptr(logits),
                                      _ptr(token), _stream(stream))


def philox(first: int, n: int, c1=0, c2=0, c3=0, key=0, stream=None) -> torch.Tensor:
    """k2_philox: [n, 4] uint32 words (as int64) of Philox4x32-10 for counters
    (first + i, c1, c2, c3) under the 64-bit key."""
    out = torch.empty(4 * n, dtype=torch.int32, device="cuda")
    st = LIB.k2_philox(first, n, c1, c2, c3, key, _ptr(out), _stream(stream))
    if st != K2_OK:
        raise K2Error(st, "k2_philox failed")
    return out.view(n, 4).cpu().to(torch.int64) & 0xFFFFFFFF


def quantize_fp8(src, stream=None):
    """k2_quantize_fp8 on a [rows, cols] bf16 device tensor: (codes uint8, scales fp32)."""
    rows, cols = src.shape
    codes = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    st = LIB.k2_quantize_fp8(_ptr(src), rows, cols, _ptr(codes), _ptr(scales), _stream(stream))
    if st != K2_OK:
        raise K2Error(st, "k2_quantize_fp8 failed")
    return codes, scales


def quantize_q4(src, stream=None):
    """k2_quantize_q4 on a [rows, cols] bf16 device tensor: (codes int8 [rows, cols],
    scales fp32 [rows, ceil(cols / 64)])."""
    rows, cols = src.shape
    codes = torch.empty(rows, cols, dtype=torch.int8, device="cuda")
    scales = torch.empty(rows, (cols + 63) // 64, dtype=torch.float32, device="cuda")
    st = LIB.k2_quantize_q4(_ptr(src), rows, cols, _ptr(codes), _ptr(scales), _stream(stream))
    if st != K2_OK:
        raise K2Error(st, "k2_quantize_q4 failed")
    return codes, scales


def spec_draft(tokens, max_draft=8) -> list:
    """k2_spec_draft (host only)."""
    ids = (C.c_int32 * max(len(tokens), 1))(*[int(t) for t in tokens])
    out = (C.c_int32 * 8)()
    n = LIB.k2_spec_draft(ids, len(tokens), max_draft, out)
    return list(out[:n])


def peek_state(cfg: Config, state) -> tuple:
    """k2_kv_peek: (cached rows, token ids) of a state in a uint8 CPU tensor,
    or (-1, -1) if it cannot be loaded into a context of cfg's model."""
    state = state.contiguous()
    cached, n_tok = C.c_int32(-1), C.c_int32(-1)
    if LIB.k2_kv_peek(C.byref(cfg), state.data_ptr(), state.numel(), C.byref(cached), C.byref(n_tok)) != K2_OK:
        return -1, -1
    return cached.value, n_tok.value


def save_state_file(path: str, state) -> None:
    with open(path, "wb") as f:
        f.write(state.numpy().tobytes())


def load_state_file(path: str) -> torch.Tensor:
    with open(path, "rb") as f:
        data = f.read()
    return torch.frombuffer(bytearray(data), dtype=torch.uint8)


def device_view(ptr: int, numel: int, dtype: torch.dtype) -> torch.Tensor:
    """A torch tensor over device memory inside a k2 workspace (test hooks)."""
    storage_bytes = numel * torch.empty((), dtype=dtype).element_size()

    class _Holder:
        __cuda_array_interface__ = {
            "shape": (storage_bytes,), "typestr": "|u1", "data": (ptr, False), "version": 3}
    return torch.as_tensor(_Holder(), device="cuda").view(dtype)[:numel]
