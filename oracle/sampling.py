"""Sampling the next token beyond greedy arg-max, written as its plain
definition in float64.

Test infrastructure only (see the package docstring).

"Kernels, Fusion & CUDA Graphs", "Fix 1: kernel fusion", the "Sampling" row:
softmax, top-k / top-p and the draw in one kernel that keeps the
vocabulary-sized logits on chip. The page names the steps and nothing more;
the readings taken here (each listed in the design notes):

* temperature T > 0 divides the logits: z = logits / T;
* top-k keeps the k largest z (a tie at the boundary keeps the lower token id);
  k = 0 keeps every token;
* top-p keeps, in order of decreasing probability under softmax over the
  top-k set (equal probabilities: lower id first), the shortest prefix whose
  probabilities sum to at least p (always at least one token); p = 1 keeps the
  whole top-k set;
* the draw is from softmax(z) restricted to the kept set and renormalised,
  taken as the Gumbel-max draw: the kept token with the largest z_i + g_i,
  g_i = -log(-log(u_i)) with one uniform u_i per token (Gumbel 1954; for
  independent u_i this picks token i with probability exp(z_i) / sum_kept
  exp(z_j), so no normaliser and no sort are needed);
* u_i comes from the counter-based generator Philox4x32-10 (Salmon, Moraes,
  Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011) with
  key (seed mod 2^32, seed div 2^32) and counter (token id, row, step mod
  2^32, step div 2^32): the first output word x gives
  u = (floor(x / 512) + 1/2) / 2^23, a value with 24 significant bits that
  float32 and float64 both hold exactly.
"""
from __future__ import annotations

import numpy as np

__all__ = ["philox4x32_10", "uniforms", "gumbel", "keep_set", "sample"]

_M0, _M1 = 0xD2511F53, 0xCD9E8D57            # round multipliers
_W0, _W1 = 0x9E3779B9, 0xBB67AE85            # key increments (Weyl sequence)
_MASK = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds on numpy uint64 arrays holding 32-bit words.

    counter: 4 arrays (c0, c1, c2, c3), key: 2 arrays (k0, k1), broadcastable.
    One round: (hi0, lo0) = M0 * c0 and (hi1, lo1) = M1 * c2 as 64-bit
    products split in halves; the new counter is (hi1 ^ c1 ^ k0, lo1,
    hi0 ^ c3 ^ k1, lo0); the key then advances by (W0, W1) modulo 2^32."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK for c in counter)
    k0, k1 = (np.asarray(k, dtype=np.uint64) & _MASK for k in key)
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = np.uint64(_M0) * c0
        p1 = np.uint64(_M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & _MASK, lo1, (hi0 ^ c3 ^ k1) & _MASK, lo0
    return c0, c1, c2, c3


def uniforms(seed: int, row: int, step: int, ids) -> np.ndarray:
    """u for the given token ids of one (row, step): float64 values in (0, 1)."""
    ids = np.asarray(ids, dtype=np.uint64)
    zero = np.zeros_like(ids)
    x0, _, _, _ = philox4x32_10((ids, zero + np.uint64(row), zero + np.uint64(step & _MASK),
                                 zero + np.uint64((step >> 32) & _MASK)),
                                (zero + np.uint64(seed & _MASK), zero + np.uint64((seed >> 32) & _MASK)))
    return ((x0 >> np.uint64(9)).astype(np.float64) + 0.5) / 2.0 ** 23


def gumbel(u: np.ndarray) -> np.ndarray:
    """Standard Gumbel variates from uniforms: -log(-log(u))."""
    return -np.log(-np.log(np.asarray(u, dtype=np.float64)))


def keep_set(logits: np.ndarray, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    """Token ids kept by top-k then top-p, in order of decreasing probability."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    V = len(z)
    order = np.lexsort((np.arange(V), -z))         # decreasing z, lower id first
    cand = order[: top_k] if 0 < top_k < V else order
    p = np.exp(z[cand] - z[cand[0]])
    p /= p.sum()
    if top_p >= 1.0:
        return cand
    csum = np.cumsum(p)
    n = int(np.searchsorted(csum, top_p, side="left")) + 1   # first prefix with sum >= top_p
    return cand[: min(max(n, 1), len(cand))]


def sample(logits: np.ndarray, temperature: float, top_k: int, top_p: float, seed: int, row: int,
           step: int) -> int:
    """The sampled token id of one row (see the module docstring)."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    kept = keep_set(logits, temperature, top_k, top_p)
    score = z[kept] + gumbel(uniforms(seed, row, step, kept))
    best = np.max(score)
    return int(np.min(kept[score == best]))        # an exact tie keeps the lower id
