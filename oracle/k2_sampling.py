"""CPU oracle for token sampling from logits.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/`` (and by
nothing on the product path); it imports nothing from the CUDA package and
shares no code with the kernels.

What it computes (k2-burn README, "Sampling + greedy generation" and its
"--temperature / --top-k / --top-p / --min-p / --seed / --repetition-penalty"
flags): temperature 0 is the greedy argmax; temperature > 0 draws the next
token from the logits after a repetition penalty on already-seen tokens and
the top-k / top-p / min-p truncation filters, with a seeded generator.

Readings where the page only names the knobs:
  * repetition penalty r: each distinct already-seen id has its logit l
    replaced by l / r if l > 0, else l * r (r = 1: off);
  * order: penalty, z = l / temperature, top-k, top-p, min-p, draw;
  * top-k: keep z >= the k-th largest z (ties at the k-th value all kept);
  * weights w = exp(z - z_max) (the probability relative to the most likely
    token), masses m = floor(w * 2^32) as integers;
  * top-p: keep a survivor of top-k iff the survivors strictly heavier than
    it weigh less than top_p * W (W = their total): the smallest
    most-probable set whose mass reaches top_p, ties kept together;
  * min-p: keep w >= min_p;
  * draw: x = Philox4x32-10 with counter (position the token takes, sequence,
    0, 0) and key (seed low, seed high); u = (x[0] >> 8) / 2^24; the token is
    the first index, in vocabulary order, whose running sum of kept masses
    exceeds floor(u * total).

Precision: the sampled token is an integer decided by floating point
comparisons, so every decision is taken in the precision of the CUDA
sampler: float32 for the penalty, the temperature division and the weights
(each step one IEEE float32 operation, as numpy performs them), unsigned
integers for the masses and their sums, float64 for the top-p comparison.
The weights use the sampler's own exp (``exp_neg``), a written-out method,
so both sides round identically.
"""
import numpy as np

F32 = np.float32
MASK32 = 0xFFFFFFFF

# ---- Philox4x32-10 -------------------------------------------------------------------------
# Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
# (SC 2011): the round multipliers and the Weyl key increments.
PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85


def philox4x32_10(ctr, key):
    """Ten Philox rounds on the 4-word counter under the 2-word key; each round
    multiplies words 0 and 2 by the round constants (64-bit products) and mixes
    the high halves with words 1, 3 and the key; the key grows by the Weyl
    constants between rounds."""
    c0, c1, c2, c3 = (int(v) & MASK32 for v in ctr)
    k0, k1 = (int(v) & MASK32 for v in key)
    for r in range(10):
        if r:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & MASK32, p1 & MASK32, ((p0 >> 32) ^ c3 ^ k1) & MASK32, p0 & MASK32
    return c0, c1, c2, c3


def uniform24(seed: int, position: int, seq: int) -> int:
    """The draw's 24 random bits r (u = r / 2^24)."""
    x = philox4x32_10((position, seq, 0, 0), (seed & MASK32, (seed >> 32) & MASK32))
    return x[0] >> 8


# ---- exp in float32 ----------------------------------------------------------------------------
EXP_TAYLOR = (1.38888888888888889e-3, 8.33333333333333333e-3, 4.16666666666666667e-2, 1.66666666666666667e-1,
              0.5, 1.0, 1.0)  # 1/6!, 1/5!, ..., 1/1!, 1/0! (Horner from 1/7!)


def exp_neg(x):
    """exp(x) for float32 x <= 0: Cody-Waite reduction x = n ln2 + r with ln2
    split into a 12-bit head and a tail, the degree-7 Taylor polynomial of
    exp(r) in Horner form, the exact scaling by 2^n; 0 below -87.  Every step
    is one float32 operation."""
    x = np.asarray(x, dtype=F32)
    live = x > F32(-87.0)
    x = np.where(live, x, F32(0.0)).astype(F32)  # the rest is 0 below
    n = np.rint(x * F32(1.44269504088896341))
    r = x - n * F32(0.693145751953125)
    r = r - n * F32(1.42860676533018708e-06)
    p = np.full_like(x, F32(1.98412698412698413e-4))
    for c in EXP_TAYLOR:
        p = p * r + F32(c)
    e = np.where(live, n, F32(0.0)).astype(np.int32)
    scale = ((e + 127) << 23).astype(np.uint32).view(F32)
    return np.where(live, p * scale, F32(0.0)).astype(F32)


def order_key(z):
    """Unsigned key of float32 values with the same order."""
    u = np.asarray(z, dtype=F32).view(np.uint32)
    return np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)


# ---- the filters and the draw --------------------------------------------------------------
def filter_row(logits, temperature, top_k=0, top_p=1.0, min_p=0.0, penalty=1.0, seen=()):
    """(kept mask, masses) of one row of logits after the penalty and the
    top-k, top-p and min-p filters."""
    lg = np.asarray(logits, dtype=F32).copy()
    V = lg.size
    if penalty != 1.0:
        ids = np.unique(np.array([i for i in seen if 0 <= i < V], dtype=np.int64))
        sel = lg[ids]
        lg[ids] = np.where(sel > 0, sel / F32(penalty), sel * F32(penalty))
    z = lg / F32(temperature)
    z = np.where(np.isnan(z), F32(-np.inf), z).astype(F32)
    zmax = z.max()
    keys = order_key(z)
    keep = np.ones(V, dtype=bool)
    if 0 < top_k < V:
        kth = np.sort(keys)[::-1][top_k - 1]
        keep &= keys >= kth
    w = exp_neg(z - zmax)
    mass = np.floor(w.astype(np.float64) * 2.0 ** 32).astype(np.uint64)
    if top_p < 1.0:
        total = int(mass[keep].sum(dtype=np.uint64))
        target = float(F32(top_p)) * float(total)
        wkey = w.view(np.uint32)
        cand = np.nonzero(keep)[0]
        ukeys, inv = np.unique(wkey[cand], return_inverse=True)  # ascending
        per_key = np.zeros(ukeys.size, dtype=object)
        for k, m in zip(inv, mass[cand]):
            per_key[k] += int(m)
        # mass strictly above each distinct key, from the top
        above = [0] * ukeys.size
        run = 0
        for k in range(ukeys.size - 1, -1, -1):
            above[k] = run
            run += per_key[k]
        kept_key = np.array([float(a) < target for a in above], dtype=bool)
        keep_p = np.zeros(V, dtype=bool)
        keep_p[cand] = kept_key[inv]
        keep &= keep_p
    if min_p > 0.0:
        keep &= w >= F32(min_p)
    return keep, mass


def sample_row(logits, temperature, top_k=0, top_p=1.0, min_p=0.0, penalty=1.0, seen=(), seed=0, position=0,
               seq=0):
    """The drawn token id of one row (temperature > 0)."""
    keep, mass = filter_row(logits, temperature, top_k, top_p, min_p, penalty, seen)
    m = [int(v) if k else 0 for v, k in zip(mass, keep)]
    total = sum(m)
    r = uniform24(seed, position, seq)
    target = (total >> 24) * r + (((total & 0xFFFFFF) * r) >> 24)
    run = 0
    for i, v in enumerate(m):
        run += v
        if run > target:
            return i
    return 0  # no kept mass (every logit NaN or -inf)


def generate_sampled(model, prompt, n_new, params, capacity=None, seq=0):
    """``model`` (an ``OracleModel``) prefills the prompt, then takes n_new
    decode steps; each next token is drawn from the fp32-rounded logits of the
    step with the position it takes and the cache's tokens as the seen set."""
    cap = capacity or (len(prompt) + n_new + 1)
    cache = model.new_cache(cap)
    _, lg = model.run(list(prompt), cache)
    seen = list(prompt)
    toks = []
    for _ in range(n_new + 1):
        t = sample_row(lg[0].astype(F32), params["temperature"], params.get("top_k", 0), params.get("top_p", 1.0),
                       params.get("min_p", 0.0), params.get("repetition_penalty", 1.0), seen,
                       params.get("seed", 0), position=len(seen), seq=seq)
        toks.append(t)
        if len(toks) == n_new + 1:
            break
        _, lg = model.run([t], cache)
        seen.append(t)
    return np.array(toks, dtype=np.int64)
