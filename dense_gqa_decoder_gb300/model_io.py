"""Uploads seeded synthetic weights (k2_inputs) to the device as torch tensors
and builds a libk2 context over them.  Marshalling only."""
from __future__ import annotations

import numpy as np
import torch

import k2_inputs as ki

from . import k2

LAYER_NAMES = ki.LAYER_TENSORS


def upload(t: ki.Tensor) -> torch.Tensor:
    a = np.ascontiguousarray(t.stored)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def device_weights(shape: ki.ModelShape, seed: int = 0, gain_scale: float = 0.0, keep_host: bool = False):
    """Returns (device dict for k2.Context, host dict of float32 values or None)."""
    dev = {n: [] for n in LAYER_NAMES}
    host = {} if keep_host else None
    for name in ("embed", "final_norm", "lm_head"):
        t = ki.weight(shape, name, -1, seed=seed, gain_scale=gain_scale)
        dev[name] = upload(t)
        if keep_host:
            host[(name, -1)] = t.values
    for l in range(shape.n_layers):
        for name in LAYER_NAMES:
            t = ki.weight(shape, name, l, seed=seed, gain_scale=gain_scale)
            dev[name].append(upload(t))
            if keep_host:
                host[(name, l)] = t.values
    return dev, host


def build_context(shape: ki.ModelShape, max_context: int, max_batch: int = 1, kv_dtype: str = "f16",
                  seed: int = 0, gain_scale: float = 0.0, keep_host: bool = False, weights: str = None,
                  prefill_split: int = None):
    """weights="f8" / "q4": the shape's bf16 weights stored as fp8 / int4 by the library.
    prefill_split: K2_OPT_PREFILL_SPLIT for the context (None: the library's default)."""
    dev, host = device_weights(shape, seed=seed, gain_scale=gain_scale, keep_host=keep_host)
    cfg = k2.make_config(shape, max_context=max_context, max_batch=max_batch, kv_dtype=kv_dtype, weights=weights)
    ctx = k2.Context(cfg, dev)
    if prefill_split is not None:
        ctx.set_option(k2.K2_OPT_PREFILL_SPLIT, prefill_split)
    return ctx, host
