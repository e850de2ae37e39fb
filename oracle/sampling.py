"""Sampling and speculative rejection sampling in fp64 (oracle side; test infrastructure).

Speculative pipeline decoding page 2, "Assumptions & free parameters", standard math
(section 3.5): rejection sampling preserves the target's output distribution, taken
from Leviathan et al. (2023).  The rule restated: a draft x drawn from p_D is kept with
probability min(1, p_T(x) / p_D(x)); otherwise the token is drawn from the normalised
residual max(0, p_T - p_D).  Readings where the pages are silent:
  * p = softmax(z / T) over the whole vocabulary;
  * a draw with uniform u takes the smallest index i whose running sum (in index order)
    exceeds u times the total;
  * the keep test is ``u1 < p_T(x) / p_D(x)``;
  * an all-zero residual (p_T == p_D) falls back to p_T.
"""
from __future__ import annotations

import numpy as np


def probs(z: np.ndarray, T: float) -> np.ndarray:
    s = np.asarray(z, dtype=np.float64) / T
    e = np.exp(s - s.max())
    return e / e.sum()


def inverse_cdf(w: np.ndarray, u: float) -> int:
    """Smallest i with sum(w[:i+1]) > u * sum(w), scanning in index order."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    i = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(i, len(w) - 1)


def residual(pT: np.ndarray, pD: np.ndarray) -> np.ndarray:
    r = np.maximum(pT - pD, 0.0)
    return pT if r.sum() <= 0.0 else r / r.sum()


def keep(pT: np.ndarray, pD: np.ndarray, x: int, u1: float) -> bool:
    return bool(u1 < pT[x] / pD[x])


def verify_exact(pT: np.ndarray, pD: np.ndarray) -> np.ndarray:
    """Exact output distribution of one draft-then-verify round: sum over drafts x of
    p_D(x) [keep prob * delta_x + (1 - keep prob) * residual].  Used to pin the
    distribution-preservation property on small vocabularies."""
    V = len(pT)
    out = np.zeros(V)
    r = residual(pT, pD)
    for x in range(V):
        if pD[x] == 0.0:
            continue
        a = min(1.0, pT[x] / pD[x])
        out[x] += pD[x] * a
        out += pD[x] * (1.0 - a) * r
    return out
