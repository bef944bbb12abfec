"""ORACLE — test infrastructure only.

Seeded sampling of the next token from a step's logits, written plainly
(numpy, one step at a time) for checking the device sampler.  "Metal LLM
decode", the sampled arm of the batched prefill+decode section, names the
controls (temperature, top_k, top_p, min_p, repeat / presence / frequency
penalties, seed) and fixes two rules: temperature <= 0 falls back to the
greedy decode, and top_k = 1 reproduces the greedy token sequence exactly.
Everything else is a reading of those names, in this order:

1. penalties, once per distinct token t among the sequence's inputs so far
   (count c_t): a = l_t / r if l_t > 0 else l_t * r; a = a - presence;
   a = a - frequency * c_t (each an f32 operation, in that order); NaN
   logits become -inf;
2. the order: tokens ranked by the penalised logit l descending, index
   ascending.  Division by T > 0 preserves that order, so ranking before the
   division keeps top_k = 1 equal to the greedy token even where l / T rounds
   two adjacent logits to the same f32 value;
3. top_k (1 <= k < V): the first k tokens of that order;
4. top_p (p < 1): of those, in that order, the shortest prefix whose
   probability mass reaches p of the kept mass;
5. min_p (> 0): keep z_i - z_max >= f32(ln min_p), with z = l / T in f32 and
   the difference in f32;
6. draw: u = (splitmix64 draw at the sampled token's position) top 24 bits
   * 2^-24; the token is the first kept one in index order whose running
   mass exceeds u times the kept mass.

Probabilities are exp(z_i - z_max) in double precision, z = l / T in f32.
When l_max / T overflows f32 to +-inf (a temperature so small that the
distribution is the limit T -> 0), the draw is the greedy token of the
penalised logits.
Where a float decides a kept set or a draw, the decision is taken on the same
f32 values the device uses (steps 1, 2, 3, 5); steps 4 and 6 compare masses,
which the device carries in fixed point, so ``sample`` also returns how far
the decisive masses lie from their boundaries.
"""
from __future__ import annotations

from collections import Counter

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def mix64(z: int) -> int:
    """The splitmix64 output function (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", 2014): two xor-shift-multiply rounds and
    a final xor-shift."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def draw(seed: int, k: int) -> int:
    """The k-th (0-based) output of splitmix64 seeded with `seed`: the state
    advances by the golden-ratio increment before each output."""
    return mix64((seed + (k + 1) * GOLDEN) & MASK64)


def uniform24(seed: int, pos: int) -> float:
    """u in [0, 1) from the top 24 bits of draw(seed, pos): exact in f32."""
    return (draw(seed, pos) >> 40) * 2.0 ** -24


def penalised(logits, history, repeat: float, presence: float, frequency: float) -> np.ndarray:
    """Step 1: the penalties on the distinct tokens among `history`, in f32."""
    l = np.array(logits, dtype=np.float32, copy=True)
    r, pr, fr = np.float32(repeat), np.float32(presence), np.float32(frequency)
    for t, c in Counter(int(x) for x in history).items():
        a = l[t]
        a = np.float32(a / r) if a > 0 else np.float32(a * r)
        a = np.float32(a - pr)
        a = np.float32(a - np.float32(fr * np.float32(c)))
        l[t] = a
    return l


def greedy(logits) -> int:
    """argmax, ties to the lowest index, NaN never wins."""
    x = np.asarray(logits, dtype=np.float64)
    x = np.where(np.isnan(x), -np.inf, x)
    return int(np.argmax(x))


def kept(logits, history, temperature: float, top_k: int = 0, top_p: float = 1.0, min_p: float = 0.0,
         repeat: float = 1.0, presence: float = 0.0, frequency: float = 0.0):
    """Steps 1-5 (temperature > 0): returns (w, keep, margin) with w the
    probabilities exp(z_i - z_max) (f64 [V]), keep the kept tokens (bool
    [V]) and margin the top_p boundary's distance relative to the mass it
    was taken from (inf without top_p)."""
    V = len(logits)
    l = penalised(logits, history, repeat, presence, frequency)
    l = np.where(np.isnan(l), np.float32(-np.inf), l).astype(np.float32)
    order = np.lexsort((np.arange(V), -l.astype(np.float64)))   # l descending, index ascending
    with np.errstate(over="ignore"):
        z = (l / np.float32(temperature)).astype(np.float32)
        zmax = np.float32(l[order[0]] / np.float32(temperature))
    if np.isinf(zmax) and np.isfinite(l[order[0]]):                # the T -> 0 limit: greedy on l
        w = np.zeros(V)
        w[order[0]] = 1.0
        keep = np.zeros(V, dtype=bool)
        keep[order[0]] = True
        return w, keep, np.inf
    w = np.exp(z.astype(np.float64) - np.float64(zmax))
    keep = np.ones(V, dtype=bool)
    margin = np.inf
    if 1 <= top_k < V:                                              # step 3
        keep[:] = False
        keep[order[:top_k]] = True
    if top_p < 1.0:                                                 # step 4
        ranked = order[keep[order]]
        total = w[ranked].sum()
        need = np.float64(np.float32(top_p)) * total
        cum = np.cumsum(w[ranked])
        j = min(int(np.searchsorted(cum, need, side="left")), len(ranked) - 1)  # first cum >= need
        keep[:] = False
        keep[ranked[:j + 1]] = True
        lo = cum[j - 1] if j > 0 else 0.0
        margin = min((cum[j] - need) / total, (need - lo) / total)
    if min_p > 0.0:                                                 # step 5
        ln = np.float32(np.log(np.float64(np.float32(min_p))))
        keep &= (z - zmax).astype(np.float32) >= ln
    return w, keep, margin


def sample(logits, history, pos: int, temperature: float, top_k: int = 0, top_p: float = 1.0,
           min_p: float = 0.0, repeat: float = 1.0, presence: float = 0.0, frequency: float = 0.0,
           seed: int = 0):
    """The token drawn at position `pos` from `logits` (f32 [V]) given the
    sequence's inputs so far (`history`).  Returns (token, margin): margin is
    the smallest distance, relative to the mass involved, between a mass the
    decision compared and its threshold (inf when no mass decided anything),
    so a caller can tell a unique answer from one a rounding could flip."""
    if temperature <= 0:
        return greedy(logits), np.inf
    w, keep, margin = kept(logits, history, temperature, top_k, top_p, min_p, repeat, presence, frequency)
    idx = np.nonzero(keep)[0]                                       # step 6, index order
    cum = np.cumsum(w[idx])
    total = cum[-1]
    target = uniform24(seed, pos) * total
    j = int(np.searchsorted(cum, target, side="right"))             # first running mass > target
    lo = cum[j - 1] if j > 0 else 0.0
    margin = min(margin, (cum[j] - target) / total, (target - lo) / total)
    return int(idx[j]), float(margin)
