#!/usr/bin/env python
"""Batch-1 greedy decode throughput of the K2-Horizon-3.7B-shape dense GQA
decoder (bf16 weights, fp16 KV) at context 4096 on one GB300, through libk2.

One step = one token: embedding, 36 decoder layers (QKV + RoPE, attention +
KV append, o_proj, gate/up + SwiGLU, down), final norm, lm_head, argmax.
Weights are random-init of the published shape (no checkpoint exists here);
the KV cache is filled by prefilling 4096 seeded random token ids.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]

Prints one JSON line.  With --gpus N > 1 (under torchrun) every rank runs an
independent replica (weak scaling; the path has no cross-GPU exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tok/s (3.7B dense GQA, bf16) and achieved HBM GB/s vs peak"
WORKLOAD = "k2-horizon-3.7b-shape greedy decode, batch 1, context 4096, fp16 KV, bf16 weights"
WEIGHT_DESC = {"bf16": "bf16", "f8": "fp8 E4M3 (per-row scales)", "q4": "int4 (one fp32 scale per 64 weights)"}
CTX = 4096
SHAPE_NAME = "k2_3p7b"
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=128)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--ctx", type=int, default=CTX)
    p.add_argument("--profile-steps", type=int, default=4)
    p.add_argument("--e2e-steps", type=int, default=32)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--layers", type=int, default=0, help="override layer count (debug)")
    p.add_argument("--kv", default="f16", choices=["f16", "i8"], help="KV cache storage")
    p.add_argument("--weights", default="bf16", choices=["bf16", "f8", "q4"],
                   help="stored projection weights: bf16, fp8 E4M3 rows with per-row scales, or int4 codes with "
                        "one scale per 64 weights of a row (both quantized at init)")
    p.add_argument("--temperature", type=float, default=0.0,
                   help="> 0: sample each token (with --top-k / --top-p / --min-p / --repetition-penalty / "
                        "--seed) instead of the greedy argmax")
    p.add_argument("--top-k", type=int, default=0)
    p.add_argument("--top-p", type=float, default=1.0)
    p.add_argument("--min-p", type=float, default=0.0)
    p.add_argument("--repetition-penalty", type=float, default=1.0)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--speculate", type=int, default=0,
                   help="> 0: greedy decode by k2_decode_speculative with up to this many drafted ids per pass "
                        "(wall clock; each pass waits for the device)")
    p.add_argument("--spec-unit", type=int, default=0,
                   help="with --speculate: the prompt repeats a random unit of this many ids (0: random ids)")
    p.add_argument("--kv-state", action="store_true",
                   help="time saving and restoring the cache state of a --ctx-token sequence (k2_kv_save / "
                        "k2_kv_load, pinned host memory) instead of decoding")
    p.add_argument("--batch", type=int, default=1,
                   help="> 1: aggregate decode throughput of that many sequences per step (each prefilled "
                        "with --ctx random tokens); the default 1 is the batch-1 metric")
    p.add_argument("--prefill-split", type=int, default=3, choices=[0, 1, 2, 3],
                   help="K2_OPT_PREFILL_SPLIT for the prefill: 3 = single fp16 operands throughout (weights "
                        "converted to fp16 per layer; the library's default), 1 = activations as bf16 hi + lo "
                        "halves and the attention's queries / probabilities as fp16 hi + lo, 0 = all single "
                        "(bf16 GEMMs), 2 = GEMM activations split, attention single")
    p.add_argument("--prefill-gemm", type=int, default=1, choices=[0, 1],
                   help="K2_OPT_PREFILL_GEMM: 1 = QKV and gate/up on the persistent kernel over whole tiles "
                        "(the default), 0 = one CTA per tile")
    p.add_argument("--phase-timeline", default="",
                   help="after the timed steps, trace a few persistent steps (K2_OPT_TRACE: per-CTA clock stamps "
                        "at every phase's start, input ready, last slot and end), write the per-phase table to "
                        "this path and add a summary to the JSON line; the traced steps are not timed")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the sub-records of the int8-KV context-8192 and batch-16 context-8192 workloads "
                        "that the default run adds to its line")
    return p.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
PHASE_KINDS = ("qkv", "attention", "o_proj", "gate_up", "down")


def phase_timeline(ctx, s, tok, stream, sm_mhz, path, steps=6):
    """Per-phase timeline of the persistent step from K2_OPT_TRACE stamps.

    Each CTA c stamps its SM clock at phase q's start, input ready, last slot
    consumed and end, plus one (globaltimer, clock) pair at its own start that
    places its clock on the common time axis.  Per phase: the critical time
    (the phase's last end minus the previous phase's last end) and, over CTAs,
    the head (start to input ready: waiting for the previous phase's words and
    the norm), body (the weight or K/V slots) and tail (combining and writing
    the outputs).  The stamps cost time themselves: read the shares, not the
    absolute step time."""
    import numpy as np
    import torch
    from dense_gqa_decoder_gb300 import k2
    G = ctx.info().persistent_grid
    nq = 5 * s.n_layers + 1
    buf = torch.zeros((nq + 1) * G * 4, dtype=torch.int64, device="cuda")
    ctx.set_option(k2.K2_OPT_TRACE, buf.data_ptr())
    runs = []
    for _ in range(steps):
        buf.zero_()
        with torch.cuda.stream(stream):
            ctx.decode_step(tok, 1, tok, stream=stream)
        stream.synchronize()
        runs.append(buf.view(nq + 1, G, 4).cpu().numpy().astype(np.float64))
    ctx.set_option(k2.K2_OPT_TRACE, 0)
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard in the traced steps: " + ctx.last_error())
    ghz = sm_mhz / 1e3
    kinds = list(PHASE_KINDS) + ["lm_head"]
    acc = {k: {"crit": [], "head_med": [], "head_max": [], "body_med": [], "body_max": [], "tail_med": [],
               "tail_max": []} for k in kinds}
    step_us = []
    for R in runs[2:]:  # the first traced steps re-capture the graph
        T = (R[:-1] - R[-1:, :, 1:2]) / ghz + R[-1:, :, 0:1]  # ns on the common axis
        T -= T[0, :, 0].min()
        prev = 0.0
        for q in range(nq):
            k = kinds[q % 5] if q < nq - 1 else "lm_head"
            st, rd, bd, en = T[q, :, 0], T[q, :, 1], T[q, :, 2], T[q, :, 3]
            d = acc[k]
            d["crit"].append(en.max() - prev)
            prev = en.max()
            for name, v in (("head", rd - st), ("body", bd - rd), ("tail", en - bd)):
                d[name + "_med"].append(float(np.median(v)))
                d[name + "_max"].append(float(v.max()))
        step_us.append(prev / 1e3)
    out = {"traced_step_us": float(np.mean(step_us)), "sm_mhz": sm_mhz, "per_layer_us": {}, "lm_head_us": {}}
    lines = ["| phase | critical (us) | share of step | head med / max | body med / max | tail med / max |",
             "|---|---|---|---|---|---|"]
    total = float(np.mean(step_us))
    for k in kinds:
        d = {n: float(np.mean(v)) / 1e3 for n, v in acc[k].items()}
        reps = s.n_layers if k != "lm_head" else 1
        share = d["crit"] * reps / total
        lines.append(f"| {k} | {d['crit']:.2f} | {100 * share:.1f} % | {d['head_med']:.2f} / {d['head_max']:.2f} | "
                     f"{d['body_med']:.2f} / {d['body_max']:.2f} | {d['tail_med']:.2f} / {d['tail_max']:.2f} |")
        (out["lm_head_us"] if k == "lm_head" else out["per_layer_us"])[k] = round(d["crit"], 3)
    if path:
        with open(path, "w") as f:
            f.write(f"traced step {total:.1f} us (SM clock {sm_mhz:.0f} MHz), {s.n_layers} layers; "
                    f"times per phase in us, the layer phases averaged over layers\n\n" + "\n".join(lines) + "\n")
    return out


def prefill_note(args):
    if args.weights == "f8":
        return ("fp8: the same tensor-core GEMMs over bf16 copies of the E4M3 codes, each row's scale applied in "
                "the GEMM epilogue; the last prompt token takes the fp8 decode step")
    if args.weights == "q4":
        return ("int4: each layer's codes * block scales dequantized into bf16 high and low halves, then the "
                "tensor-core GEMMs with three MMAs per K step (w_hi x_hi, w_hi x_lo, w_lo x_hi); the last prompt "
                "token takes the int4 decode step")
    if args.prefill_split == 3:
        return ("useful FLOPs (2 per weight x token + causal attention); every contraction on single fp16 "
                "operands (the bf16 weights converted to fp16 per layer, exact in fp16's normal range; fp16 "
                "activations, queries and probabilities), one MMA per K step, S and O in tensor memory")
    if args.prefill_split:
        return ("useful FLOPs (2 per weight x token + causal attention); the GEMMs issue twice the linear MMAs "
                "(activations as bf16 hi + lo halves); attention (fp16 KV) issues tcgen05 MMAs on fp16 hi + lo "
                "halves of the queries and probabilities, S and O in tensor memory")
    return ("useful FLOPs (2 per weight x token + causal attention); single bf16 activations into the GEMMs and "
            "single fp16 queries and probabilities into the tcgen05 attention (fp16 KV), S and O in tensor memory")



def algorithmic_bytes(s, ctx_len: int, kv: str = "f16", weights_store: str = "bf16") -> dict:
    """Bytes the decode step must move at context ctx_len (weights once, the
    KV history once, plus the small activations).  fp8 weights: one byte per
    weight plus a 4-byte scale per row; int4: half a byte per weight plus a
    4-byte scale per 64 weights; gains and the embedding row stay bf16."""
    H, d, I, V = s.hidden, s.head_dim, s.intermediate, s.vocab
    qkv_n = (s.n_heads + 2 * s.n_kv_heads) * d
    gb = 2 if s.weight_dtype == "bf16" else 4
    def mat(N, K):  # bytes of one stored projection matrix [N, K]
        if weights_store == "f8":  # one byte per weight, one fp32 scale per row
            return N * K + 4 * N
        if weights_store == "q4":  # half a byte per weight, one fp32 scale per 64 weights of a row
            return N * K // 2 + 4 * N * ((K + 63) // 64)
        return N * K * gb

    per_layer = mat(qkv_n, H) + mat(H, s.n_heads * d) + mat(2 * I, H) + mat(H, I) + 2 * H * gb
    weights = s.n_layers * per_layer + mat(V, H) + H * gb
    # K and V of one position, one layer: fp16, or int8 codes + one fp16 scale per head
    kv_row = 2 * s.n_kv_heads * d * 2 if kv == "f16" else 2 * s.n_kv_heads * (d + 2)
    kv = s.n_layers * kv_row * ctx_len
    return {
        "weights": weights,
        "kv": kv,
        "total": weights + kv,
        # the gate/up GEMV: W [2I, H] + x [H] fp32 + gain [H] + act [I] fp32
        "gate_up_launch": mat(2 * I, H) + H * 4 + H * gb + I * 4,
        # the persistent step kernel: weights, the KV history, the new K/V rows
        "step_launch": weights + kv + s.n_layers * kv_row,
    }


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def traffic_from_profiles(kernel_sources, kernel):
    """dram bytes per launch of `kernel` from the committed ncu summary, only
    if the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    h = hashlib.sha256()
    for src in kernel_sources:
        with open(src, "rb") as f:
            h.update(f.read())
    sha = h.hexdigest()[:16]
    try:
        for line in open(path):
            kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
            if kv.get("kernel") == kernel and kv.get("source_sha") == sha:
                return float(kv["dram_bytes_per_launch"]), sha
    except OSError:
        pass
    return None, sha


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.out.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, value: float) -> float:
    """The largest of a per-rank number over all ranks (the slowest rank's
    time); the number itself on a single rank."""
    if pg is None:
        return value
    import torch
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (every rank does the same fixed work: weak scaling)."""
    return world * units_per_rank / seconds


def step_stats(per_step_ms) -> dict:
    """Median and 90th percentile (nearest rank) of the per-step times."""
    v = sorted(per_step_ms)
    if not v:
        return {"p50_ms": None, "p90_ms": None}
    k = max(0, -(-9 * len(v) // 10) - 1)
    return {"p50_ms": statistics.median(v), "p90_ms": v[k]}


def timed_decode(ctx, tok, batch, steps, stream, local, pg):
    """`steps` decode steps (CUDA graph replays) on `stream`, an event before
    the first and after every step, between a barrier and a synchronize on
    both sides, with the SM clocks sampled meanwhile.  Returns (ms of all
    steps, max over ranks; per-step ms on this rank; clock summary)."""
    import torch
    clocks = ClockSampler(local)
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        ctx.decode_step(tok, batch, tok, stream=stream)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clk = clocks.stop()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return max_over_ranks(pg, ev[0].elapsed_time(ev[-1])), per, clk


# ---------------------------------------------------------------------------
# CPU oracle legs (the oracle as it stands, on this host's cores)
# ---------------------------------------------------------------------------

def oracle_decode_sample(n_layers_sample: int = 2, vocab_fraction: float = 1.0, ctx_len: int = CTX):
    """Times the oracle's single-token decode at context ctx_len on a sample of
    the model: n_layers_sample layers (each with its own weights) and a
    fraction of the lm_head rows; returns seconds per full token (the sample
    scaled to 36 layers and the whole vocab) and a description."""
    import numpy as np

    import k2_inputs as ki
    from oracle import k2_oracle as O

    s = ki.K2_3P7B
    rng = np.random.default_rng(5)
    kv = rng.standard_normal((ctx_len, s.n_kv_heads, s.head_dim)).astype(np.float16).astype(np.float64)
    x = ki.hidden_f32(s.hidden, seed=3).astype(np.float64)
    t_layers = 0.0
    for l in range(n_layers_sample):
        w = {n: ki.weight(s, n, l).values for n in ki.LAYER_TENSORS}
        t0 = time.perf_counter()
        x, _, _ = O.layer_decode_step(s, w, x, ctx_len, kv, kv, "f16")
        t_layers += time.perf_counter() - t0
    rows = max(1, int(s.vocab * vocab_fraction))
    W = ki.weight(s, "lm_head", -1).values[:rows]
    fn = np.ones(s.hidden, np.float32)
    m = O.OracleModel(s.replace(vocab=rows), lambda n, l: {"final_norm": fn, "lm_head": W}[n], "f16")
    t0 = time.perf_counter()
    lg = m.head(x[None, :])
    O.argmax_first(lg[0])
    t_head = time.perf_counter() - t0
    per_token = t_layers / n_layers_sample * s.n_layers + t_head / (rows / s.vocab)
    desc = (f"oracle single-token decode at context {ctx_len}: {n_layers_sample} of {s.n_layers} layers and "
            f"{rows} of {s.vocab} lm_head rows timed, scaled to one full token")
    return per_token, desc, t_layers + t_head


def host_cpu() -> dict:
    """The host the oracle ran on: logical CPUs and the model name."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                name = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"nproc": os.cpu_count(), "model": name}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, world, rank, pg):
    if rank != 0:
        return
    import numpy as np  # noqa: F401
    # each step: one oracle decode over one layer and 1/36 of the lm_head rows
    # (a 36th of a token); value = tokens per second of the whole model
    for _ in range(args.warmup):
        oracle_decode_sample(1, 1.0 / 36, args.ctx)
    per_tok, times = [], []
    for _ in range(args.steps):
        pt, desc, wall = oracle_decode_sample(1, 1.0 / 36, args.ctx)
        per_tok.append(pt)
        times.append(wall)
    sec_per_token = statistics.mean(per_tok)
    value = 1.0 / sec_per_token
    cores = blas_threads()
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(times) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": WORKLOAD, "batch": 1, "context": args.ctx},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": desc + "; each step is 1/36 of a token", "host": host_cpu()},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def random_device_weights(s, seed: int = 0):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    dt = torch.bfloat16 if s.weight_dtype == "bf16" else torch.float32

    def rnd(*shape):
        return (torch.randn(*shape, generator=g, device="cuda", dtype=torch.float32) * 0.02).to(dt)

    H, d = s.hidden, s.head_dim
    w = {"embed": rnd(s.vocab, H), "lm_head": rnd(s.vocab, H), "final_norm": torch.ones(H, device="cuda", dtype=dt)}
    for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"):
        w[n] = []
    for _ in range(s.n_layers):
        w["attn_norm"].append(torch.ones(H, device="cuda", dtype=dt))
        w["mlp_norm"].append(torch.ones(H, device="cuda", dtype=dt))
        w["wq"].append(rnd(s.n_heads * d, H))
        w["wk"].append(rnd(s.n_kv_heads * d, H))
        w["wv"].append(rnd(s.n_kv_heads * d, H))
        w["wo"].append(rnd(H, s.n_heads * d))
        w["w_gate"].append(rnd(s.intermediate, H))
        w["w_up"].append(rnd(s.intermediate, H))
        w["w_down"].append(rnd(H, s.intermediate))
    return w


def run_ours(args, world, rank, local, pg):
    import numpy as np
    import torch

    import k2_inputs as ki
    from dense_gqa_decoder_gb300 import k2

    torch.cuda.set_device(local)
    s = ki.SHAPES[SHAPE_NAME]
    if args.layers:
        s = s.replace(n_layers=args.layers)
    budget = args.ctx + args.warmup + args.steps + args.profile_steps + args.e2e_steps + 16
    cfg = k2.make_config(s, max_context=budget, max_batch=1, kv_dtype=args.kv,
                         weights=None if args.weights == "bf16" else args.weights)
    wdev = random_device_weights(s, seed=1234 + rank)
    ctx = k2.Context(cfg, wdev)
    stream = torch.cuda.Stream()
    sampled = args.temperature > 0
    if sampled:
        ctx.set_sampling(k2.sampling(temperature=args.temperature, top_k=args.top_k, top_p=args.top_p,
                                     min_p=args.min_p, repetition_penalty=args.repetition_penalty, seed=args.seed))
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    prompt = torch.from_numpy(ki.prompt_ids(s.vocab, args.ctx, seed=1 + rank)).cuda()
    # prefill: one untimed warm-up on a short prompt, then the timed prompt
    ctx.set_option(k2.K2_OPT_PREFILL_SPLIT, args.prefill_split)
    ctx.set_option(k2.K2_OPT_PREFILL_GEMM, args.prefill_gemm)
    with torch.cuda.stream(stream):
        ctx.prefill(0, prompt[:256], tok, stream=stream)
    stream.synchronize()
    ctx.kv_reset(0, stream=stream)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    with torch.cuda.stream(stream):
        ctx.prefill(0, prompt, tok, stream=stream)
    p1.record(stream)
    stream.synchronize()
    prefill_ms = p0.elapsed_time(p1)
    ctx.set_option(k2.K2_OPT_GRAPH, 1)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            ctx.decode_step(tok, 1, tok, stream=stream)
    stream.synchronize()
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard after warm-up: " + ctx.last_error())

    ctx_start = ctx.kv_view(0, 0)[4]
    ms, per_step, clk = timed_decode(ctx, tok, 1, args.steps, stream, local, pg)
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard after the timed steps: " + ctx.last_error())
    ms_per_step = ms / args.steps
    value = job_throughput(world, args.steps, ms / 1e3)
    mean_ctx = ctx_start + (args.steps - 1) / 2 + 1
    by = algorithmic_bytes(s, int(round(mean_ctx)), args.kv, args.weights)

    # per-kernel durations: one un-graphed step with an event pair per kernel
    ms_k = {k: 0.0 for k in k2.KERNEL_CLASSES}
    n_k = {k: 0 for k in k2.KERNEL_CLASSES}
    for _ in range(args.profile_steps):
        a, b = ctx.profile_decode(tok, 1, tok, stream=stream)
        for k in ms_k:
            ms_k[k] += a[k]
            n_k[k] += b[k]
    persistent = n_k["step"] > 0
    peak, peak_src = measured_peaks()
    csrc = os.path.join(ROOT, "dense_gqa_decoder_gb300", "csrc")
    k_ms_profile = None
    if persistent and not sampled:
        # the whole token is one kernel, the only launch of a timed step: its
        # average duration over the timed region is the mean of the per-step
        # event pairs around the graph replays (on the launching stream); the
        # un-graphed profiling launch (which includes its launch) is kept beside it
        k_name, k_desc, k_bytes = "mega_decode", "mega_decode_kernel (whole decode step)", by["step_launch"]
        k_ms = statistics.mean(per_step)
        k_ms_profile = ms_k["step"] / n_k["step"]
        src = [os.path.join(csrc, f) for f in ("k2_mega.cu", "k2_common.cuh", "k2_kernels.h")]
        launches_per_step = 1
    elif persistent:
        # sampling adds the sampler kernel to every step: the profiling launch of the step kernel alone
        k_name, k_desc, k_bytes = "mega_decode", "mega_decode_kernel (whole decode step)", by["step_launch"]
        k_ms = ms_k["step"] / n_k["step"]
        src = [os.path.join(csrc, f) for f in ("k2_mega.cu", "k2_common.cuh", "k2_kernels.h")]
        launches_per_step = 2 if sampled else 1  # the step, and the sampler when sampling
    else:
        k_name, k_desc, k_bytes = "gemv_gate_up", "gemv_gate_up (norm + gate/up GEMV + SwiGLU)", by["gate_up_launch"]
        k_ms = ms_k["gate_up"] / max(1, n_k["gate_up"])
        src = [os.path.join(csrc, f) for f in ("k2_gemv_packed.cu", "k2_common.cuh", "k2_kernels.h")]
        launches_per_step = 1 + 5 * s.n_layers + 1
    achieved = k_bytes / (k_ms * 1e-3) / 1e9
    traffic, sha = traffic_from_profiles(src, k_name)
    if not (args.kv == "f16" and args.ctx == CTX and args.weights == "bf16" and not sampled and not args.layers):
        traffic = None  # the committed capture is of the default workload only

    # end to end through the C ABI with host buffers: token H2D, step, token D2H
    host_in = torch.zeros(1, dtype=torch.int32).pin_memory()
    host_out = torch.zeros(1, dtype=torch.int32).pin_memory()
    host_in.copy_(tok.cpu())
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        with torch.cuda.stream(stream):
            tok.copy_(host_in, non_blocking=True)
            ctx.decode_step(tok, 1, tok, stream=stream)
            host_out.copy_(tok, non_blocking=True)
        stream.synchronize()
        host_in.copy_(host_out)
    e2e_s = time.perf_counter() - t0
    e2e_value = world * args.e2e_steps / e2e_s

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        per_token, desc, _ = oracle_decode_sample(2, 1.0, args.ctx)
        cpu = {"value": 1.0 / per_token, "unit": "tok/s", "cores": blas_threads(), "kind": "oracle", "sample": desc,
               "host": host_cpu()}

    T = args.ctx
    pf_linear = 2.0 * s.n_layers * ((s.n_heads + 2 * s.n_kv_heads) * s.head_dim * s.hidden
                                    + s.hidden * s.n_heads * s.head_dim + 3 * s.intermediate * s.hidden) * T
    pf_attn = 2.0 * 2 * s.n_layers * s.n_heads * s.head_dim * T * (T + 1) / 2
    pf_tflops = (pf_linear + pf_attn) / (prefill_ms * 1e-3) / 1e12
    tc_peak = measured_bf16_peak()
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"bf16": "bf16", "f8": "f8e4m3", "q4": "i4"}[args.weights], "data": "synthetic",
        "config": {"workload": WORKLOAD if (args.kv == "f16" and args.ctx == CTX and not sampled and
                                            args.weights == "bf16") else
                   f"k2-horizon-3.7b-shape {'sampled' if sampled else 'greedy'} decode, batch 1, context {args.ctx}, "
                   f"{args.kv} KV, {WEIGHT_DESC[args.weights]} weights",
                   "sampling": ({"temperature": args.temperature, "top_k": args.top_k, "top_p": args.top_p,
                                 "min_p": args.min_p, "repetition_penalty": args.repetition_penalty,
                                 "seed": args.seed} if sampled else None),
                   "batch": 1, "context": args.ctx, "layers": s.n_layers,
                   "kv_dtype": args.kv, "activations": "fp32", "cuda_graph": True,
                   "persistent_kernel": persistent, "pdl": not persistent,
                   "l2": "no flush: every step streams 8.8 GB of weights, far above the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "hbm": {"bytes_per_step": by["total"], "achieved_gbs": by["total"] / (ms_per_step * 1e-3) / 1e9,
                "peak_gbs": peak, "frac": by["total"] / (ms_per_step * 1e-3) / 1e9 / peak,
                "frac_of_8tbs_nominal": by["total"] / (ms_per_step * 1e-3) / 1e9 / 8000.0},
        "step_ms": step_stats(per_step),
        "roofline": {"bound": "hbm", "kernel": k_desc,
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": peak_src, "algorithmic_bytes": k_bytes,
                     "launch_ms": k_ms, "launch_ms_ungraphed": k_ms_profile, "source_sha": sha},
        "kernel_ms_per_step": {k: ms_k[k] / args.profile_steps for k in ms_k},
        "gpu_launches": launches_per_step * args.steps,
        "prefill": {"tokens": T, "ms": prefill_ms, "tok_per_s": T / (prefill_ms * 1e-3),
                    "algorithmic_tflop": (pf_linear + pf_attn) / 1e12,
                    "achieved_tflops": pf_tflops, "peak_tflops": tc_peak, "frac": pf_tflops / tc_peak,
                    "split_mode": args.prefill_split, "persistent_gemm": bool(args.prefill_gemm),
                    "note": prefill_note(args)},
        "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4},
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    if args.phase_timeline and persistent:
        line["phase_timeline"] = phase_timeline(ctx, s, tok, stream, clk.get("sm_mhz") or 2070.0,
                                                args.phase_timeline)
    default = (args.kv == "f16" and args.ctx == CTX and args.weights == "bf16" and not sampled and not args.layers)
    if default and not args.no_configs:
        # the two larger workloads, each on a fresh context over the same weights
        del ctx
        torch.cuda.empty_cache()
        line["configs"] = {
            "int8_kv_ctx8192": sub_int8_ctx8192(args, s, wdev, world, local, pg),
            "batch16_ctx8192": sub_batch16_ctx8192(args, s, wdev, world, local, pg),
        }
    if rank == 0:
        print(json.dumps(line), flush=True)


def sub_int8_ctx8192(args, s, wdev, world, local, pg):
    """The int8-KV workload: allocation 32768 positions, prefill of 8192
    random ids, then 512 greedy decode steps (after the warm-up), batch 1."""
    import torch

    import k2_inputs as ki
    from dense_gqa_decoder_gb300 import k2
    T, steps = 8192, 512
    ctx = k2.Context(k2.make_config(s, max_context=32768, max_batch=1, kv_dtype="i8"), wdev)
    stream = torch.cuda.Stream()
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    with torch.cuda.stream(stream):
        ctx.prefill(0, torch.from_numpy(ki.prompt_ids(s.vocab, T, seed=1)).cuda(), tok, stream=stream)
    p1.record(stream)
    stream.synchronize()
    ctx.set_option(k2.K2_OPT_GRAPH, 1)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            ctx.decode_step(tok, 1, tok, stream=stream)
    stream.synchronize()
    c0 = ctx.kv_view(0, 0)[4]
    ms, per, clk = timed_decode(ctx, tok, 1, steps, stream, local, pg)
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard (int8 KV workload): " + ctx.last_error())
    by = algorithmic_bytes(s, int(round(c0 + (steps - 1) / 2 + 1)), "i8")
    peak, peak_src = measured_peaks()
    mps = ms / steps
    achieved = by["step_launch"] / (mps * 1e-3) / 1e9
    del ctx
    torch.cuda.empty_cache()
    return {"workload": f"k2-horizon-3.7b-shape greedy decode, batch 1, int8 KV (allocation 32768), prefill {T} "
                        f"random ids, then {steps} timed steps (context {c0} -> {c0 + steps})",
            "value": job_throughput(world, steps, ms / 1e3), "unit": "tok/s", "ms_per_step": mps,
            "step_ms": step_stats(per), "prefill_ms": p0.elapsed_time(p1),
            "roofline": {"bound": "hbm", "kernel": "mega_decode_kernel (whole decode step, graph replay)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "peak_source": peak_src, "algorithmic_bytes": by["step_launch"]},
            "clocks": clk}


def sub_batch16_ctx8192(args, s, wdev, world, local, pg):
    """The batch-16 workload: 16 independent sequences, each prefilled with
    8192 random ids (distinct seeds), then 128 greedy decode steps of all 16
    (after the warm-up)."""
    import torch

    import k2_inputs as ki
    from dense_gqa_decoder_gb300 import k2
    B, T, steps = 16, 8192, 128
    ctx = k2.Context(k2.make_config(s, max_context=T + args.warmup + steps + 16, max_batch=B, kv_dtype="f16"), wdev)
    stream = torch.cuda.Stream()
    tok = torch.zeros(B, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for b in range(B):
            ctx.prefill(b, torch.from_numpy(ki.prompt_ids(s.vocab, T, seed=1 + b)).cuda(), tok[b:b + 1],
                        stream=stream)
    ctx.set_option(k2.K2_OPT_GRAPH, 1)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            ctx.decode_step(tok, B, tok, stream=stream)
    stream.synchronize()
    c0 = ctx.kv_view(0, 0)[4]
    ms, per, clk = timed_decode(ctx, tok, B, steps, stream, local, pg)
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard (batch-16 workload): " + ctx.last_error())
    one = algorithmic_bytes(s, 1, "f16")
    step_bytes = one["weights"] + B * one["kv"] * (c0 + (steps - 1) / 2 + 1)
    peak, peak_src = measured_peaks()
    mps = ms / steps
    achieved = step_bytes / (mps * 1e-3) / 1e9
    del ctx
    torch.cuda.empty_cache()
    return {"workload": f"k2-horizon-3.7b-shape greedy decode, {B} sequences, fp16 KV, each prefilled with {T} "
                        f"random ids, then {steps} timed steps (context {c0} -> {c0 + steps})",
            "value": job_throughput(world, B * steps, ms / 1e3), "unit": "tok/s", "ms_per_step": mps,
            "step_ms": step_stats(per),
            "roofline": {"bound": "hbm", "kernel": "batched decode step (tensor-core GEMMs with N = 16, decode "
                                                   "attention, row kernels; graph replay)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "peak_source": peak_src, "algorithmic_bytes": step_bytes},
            "clocks": clk}


def run_speculative(args, world, rank, local, pg):
    """Greedy decoding with n-gram drafts verified in one pass: --steps
    emitted tokens timed after --warmup, from a --ctx-token random prompt."""
    import numpy as np
    import torch

    import k2_inputs as ki
    from dense_gqa_decoder_gb300 import k2

    torch.cuda.set_device(local)
    s = ki.SHAPES[SHAPE_NAME]
    if args.layers:
        s = s.replace(n_layers=args.layers)
    cfg = k2.make_config(s, max_context=args.ctx + args.warmup + args.steps + 32, max_batch=1, kv_dtype=args.kv)
    ctx = k2.Context(cfg, random_device_weights(s, seed=1234 + rank))
    stream = torch.cuda.Stream()
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    if args.spec_unit > 0:
        unit = [int(x) for x in ki.prompt_ids(s.vocab, args.spec_unit, seed=1 + rank)]
        ids = (unit * (args.ctx // args.spec_unit + 1))[:args.ctx]
    else:
        ids = [int(x) for x in ki.prompt_ids(s.vocab, args.ctx, seed=1 + rank)]
    with torch.cuda.stream(stream):
        ctx.prefill(0, torch.tensor(ids, dtype=torch.int32, device="cuda"), tok, stream=stream)
    stream.synchronize()
    ctx.set_option(k2.K2_OPT_GRAPH, 1)  # each (block size) is recorded once, then replayed
    buf = np.zeros(args.ctx + args.warmup + args.steps + 32, dtype=np.int32)  # the sequence, passed without copies
    buf[:len(ids)] = ids
    buf[len(ids)] = int(tok.item())
    n = len(ids) + 1

    def step():
        nonlocal n
        got = ctx.decode_speculative(0, buf[:n], args.speculate, stream=stream)
        buf[n:n + len(got)] = got
        n += len(got)
        return len(got)

    emitted = 0
    while emitted < args.warmup:
        emitted += step()
    t0 = time.perf_counter()
    emitted, passes = 0, 0
    while emitted < args.steps:
        emitted += step()
        passes += 1
    dt = time.perf_counter() - t0
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard after speculative decoding: " + ctx.last_error())
    line = {
        "metric": "speculative greedy decode tok/s (3.7B dense GQA, bf16)", "value": world * emitted / dt,
        "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"k2-horizon-3.7b-shape greedy decode with up to {args.speculate} n-gram drafts "
                               f"per pass, batch 1, from a {args.ctx}-token "
                               + (f"prompt repeating a {args.spec_unit}-id random unit" if args.spec_unit > 0
                                  else "random prompt") + f", {args.kv} KV",
                   "layers": s.n_layers, "timing": "wall clock (every pass waits for the device)"},
        "passes": passes, "tokens_per_pass": emitted / passes, "ms_per_pass": 1e3 * dt / passes,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_kv_state(args, world, rank, local, pg):
    """Save / restore of one sequence's cache: the state of a --ctx-token
    prompt (K/V rows of every layer + header + the prompt's ids) written to
    pinned host memory and read back, --steps times each after --warmup."""
    import torch

    import k2_inputs as ki
    from dense_gqa_decoder_gb300 import k2

    torch.cuda.set_device(local)
    s = ki.SHAPES[SHAPE_NAME]
    if args.layers:
        s = s.replace(n_layers=args.layers)
    cfg = k2.make_config(s, max_context=args.ctx + 16, max_batch=1, kv_dtype=args.kv)
    ctx = k2.Context(cfg, random_device_weights(s, seed=1234 + rank))
    stream = torch.cuda.Stream()
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = ki.prompt_ids(s.vocab, args.ctx, seed=1 + rank)
    with torch.cuda.stream(stream):
        ctx.prefill(0, torch.from_numpy(ids).cuda(), tok, stream=stream)
    stream.synchronize()
    n = ctx.kv_state_bytes(0, len(ids))
    buf = torch.empty(n, dtype=torch.uint8).pin_memory()
    save_s, load_s = [], []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        state = ctx.kv_save(0, ids, out=buf, stream=stream)
        t1 = time.perf_counter()
        back = ctx.kv_load(0, state, stream=stream)
        t2 = time.perf_counter()
        if i >= args.warmup:
            save_s.append(t1 - t0)
            load_s.append(t2 - t1)
    assert back == [int(x) for x in ids]
    with torch.cuda.stream(stream):
        ctx.decode_step(tok, 1, tok, stream=stream)
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard after the restored step: " + ctx.last_error())
    save_gbs = world * n / (sum(save_s) / len(save_s)) / 1e9
    line = {
        "metric": f"KV cache state save / restore, {args.ctx}-token sequence", "value": save_gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.kv, "data": "synthetic",
        "config": {"workload": f"k2-horizon-3.7b-shape cache of one sequence, context {args.ctx}, {args.kv} KV",
                   "layers": s.n_layers, "host_buffer": "pinned"},
        "state_bytes": n,
        "save": {"ms": 1e3 * sum(save_s) / len(save_s), "gbs": save_gbs},
        "load": {"ms": 1e3 * sum(load_s) / len(load_s), "gbs": world * n / (sum(load_s) / len(load_s)) / 1e9},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_batched(args, world, rank, local, pg):
    """Batched decode: --batch sequences, each prefilled with --ctx random ids,
    advanced together by one k2_decode_step per step (weights read once per
    step for all of them)."""
    import torch

    import k2_inputs as ki
    from dense_gqa_decoder_gb300 import k2

    torch.cuda.set_device(local)
    s = ki.SHAPES[SHAPE_NAME]
    if args.layers:
        s = s.replace(n_layers=args.layers)
    B = args.batch
    cfg = k2.make_config(s, max_context=args.ctx + args.warmup + args.steps + 16, max_batch=B, kv_dtype=args.kv)
    ctx = k2.Context(cfg, random_device_weights(s, seed=1234 + rank))
    stream = torch.cuda.Stream()
    tok = torch.zeros(B, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for b in range(B):
            prompt = torch.from_numpy(ki.prompt_ids(s.vocab, args.ctx, seed=1 + b + 100 * rank)).cuda()
            ctx.prefill(b, prompt, tok[b:b + 1], stream=stream)
    ctx.set_option(k2.K2_OPT_GRAPH, 1)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            ctx.decode_step(tok, B, tok, stream=stream)
    stream.synchronize()
    ms, per, clk = timed_decode(ctx, tok, B, args.steps, stream, local, pg)
    if ctx.sync_status(stream) != k2.K2_OK:
        raise RuntimeError("device guard after the timed steps: " + ctx.last_error())
    ms_per_step = ms / args.steps
    mean_ctx = args.ctx + args.warmup + (args.steps - 1) / 2 + 1
    by = algorithmic_bytes(s, 1, args.kv)
    step_bytes = by["weights"] + B * (by["kv"] * mean_ctx)  # kv of one position x mean length, per sequence
    peak, peak_src = measured_peaks()
    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": f"batch-{B} decode aggregate tok/s (3.7B dense GQA, bf16) and achieved HBM GB/s vs peak",
        "value": job_throughput(world, B * args.steps, ms / 1e3), "unit": "tok/s", "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"k2-horizon-3.7b-shape greedy decode, {B} sequences, context {args.ctx}, {args.kv} KV",
                   "batch": B, "context": args.ctx, "layers": s.n_layers, "cuda_graph": True,
                   "l2": "no flush: every step streams 8.8 GB of weights", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "decode_batched step (tensor-core GEMMs N = batch, attention, "
                                               "row kernels)", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "peak_source": peak_src,
                     "algorithmic_bytes": step_bytes},
        "step_ms": step_stats(per),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local, pg = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank, pg)
    elif args.kv_state:
        run_kv_state(args, world, rank, local, pg)
    elif args.speculate > 0:
        run_speculative(args, world, rank, local, pg)
    elif args.batch > 1:
        run_batched(args, world, rank, local, pg)
    else:
        run_ours(args, world, rank, local, pg)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
