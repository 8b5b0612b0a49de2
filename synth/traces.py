"""Seeded synthetic routing traces for the residency-policy replays.

No real routing trace is in this repository (the kairos README replays a recorded
conversation). These traces stand in for one with the two properties the README
measures: skewed expert popularity and sticky routing between adjacent tokens
("adjacent tokens share 43% of a layer's experts"). Per layer, a Zipf(s)
popularity over a seeded permutation of the experts; each token keeps each of the
previous token's experts with probability `stick` and fills the rest of its K
distinct experts by popularity. Holds none of the layer's arithmetic; uses
numpy's PCG64 generator with a fixed seed.
"""
from __future__ import annotations

import numpy as np


def routing_trace(n_tokens: int, n_layers: int, n_experts: int, K: int, seed: int = 0, zipf_s: float = 1.1,
                  stick: float = 0.43):
    """ids [n_tokens][n_layers][K] int32: the experts each token routes to per layer."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    out = np.zeros((n_tokens, n_layers, K), dtype=np.int32)
    ranks = np.arange(1, n_experts + 1, dtype=np.float64)
    pop = ranks ** (-zipf_s)
    pop /= pop.sum()
    perms = [rng.permutation(n_experts) for _ in range(n_layers)]
    prev = [None] * n_layers
    for t in range(n_tokens):
        for l in range(n_layers):
            chosen = []
            if prev[l] is not None:
                keep = rng.random(K) < stick
                chosen = [int(e) for e, k in zip(prev[l], keep) if k]
            while len(chosen) < K:
                e = int(perms[l][rng.choice(n_experts, p=pop)])
                if e not in chosen:
                    chosen.append(e)
            out[t, l] = chosen
            prev[l] = out[t, l].copy()
    return out


def profile_ranking(trace) -> tuple[np.ndarray, np.ndarray]:
    """(layers, experts) of every pair seen in `trace`, most frequent first (equal
    counts: lower layer, then lower expert): a shipped profile."""
    T, L, K = trace.shape
    counts = {}
    for t in range(T):
        for l in range(L):
            for e in trace[t, l]:
                counts[(l, int(e))] = counts.get((l, int(e)), 0) + 1
    order = sorted(counts, key=lambda k: (-counts[k], k[0], k[1]))
    return (np.array([k[0] for k in order], dtype=np.int32), np.array([k[1] for k in order], dtype=np.int32))


def sharing(trace) -> float:
    """Mean share of a layer's experts that the next token routes to again."""
    T, L, K = trace.shape
    s = [len(set(trace[t, l]) & set(trace[t + 1, l])) / K for t in range(T - 1) for l in range(L)]
    return float(np.mean(s)) if s else 0.0
