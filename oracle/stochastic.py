"""Stochastic prefix verifier, CPU reference in fp64 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
use this module; the CUDA library never imports it and shares no code with it.

Follows "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification",
SIII-D (Prefix verifier), step by step:

* P_r is the target policy's next-token distribution of packed row r: softmax(z_r / T) at
  temperature T > 0 (row off_i + j - 1 predicts candidate j);
* the deterministic draft candidate x_j = tokens[off_i + j] (j = 1..k_i-1) is accepted with
  probability P_{off_i+j-1}(x_j): it is accepted iff u[off_i + j] < P(x_j), in order, and the
  first rejection ends the prefix;
* at the first rejection (candidate a+1), the successor is drawn from P_{off_i+a} with
  x_{a+1} removed and the rest renormalised; if every candidate passes, from the
  unmodified P_{off_i+k_i-1}; row off_i + a_i supplies the successor either way;
* accept_len = 1 + a_i (the anchor counts), next_token = the successor; k_i = 0 gives
  accept_len 0 and next_token -1.

The random numbers are inputs: u_accept [m_cap] (entry off_i + j is the draw for candidate
j) and u_next [n] (the successor draw of request i), each uniform in [0, 1).  The successor
is the smallest token y whose cumulative renormalised probability, summed in token order,
exceeds u_next (inverse-CDF sampling).
"""
from __future__ import annotations

from typing import Tuple

import numpy as np


def row_probs(z: np.ndarray, temperature: float) -> np.ndarray:
    """softmax(z / T) of one row, fp64."""
    x = np.asarray(z, dtype=np.float64) / float(temperature)
    x = x - x.max()
    e = np.exp(x)
    return e / e.sum()


def sample(p: np.ndarray, u: float, exclude: int = -1) -> int:
    """Smallest y with sum_{y' <= y, y' != exclude} p(y') > u * (1 - p(exclude))."""
    w = p.copy()
    if exclude >= 0:
        w[exclude] = 0.0
    total = w.sum()
    c = np.cumsum(w)
    y = int(np.searchsorted(c, u * total, side="right"))
    y = min(y, len(p) - 1)
    while w[y] == 0.0 and y > 0:      # never land on the removed token or an empty tail
        y -= 1
    return y


def stochastic_accept(logits: np.ndarray, tokens: np.ndarray, cu_slots: np.ndarray,
                      temperature: float, u_accept: np.ndarray,
                      u_next: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(accept_len [n], next_token [n], p_draft [m_cap]) -- p_draft[off_i + j] is the
    acceptance probability of candidate j (NaN where no candidate is tested)."""
    z = np.asarray(logits, dtype=np.float64)
    cu = np.asarray(cu_slots, dtype=np.int64)
    n = len(cu) - 1
    acc = np.zeros(n, dtype=np.int32)
    nxt = np.full(n, -1, dtype=np.int32)
    p_draft = np.full(z.shape[0], np.nan)
    for i in range(n):
        off, k = int(cu[i]), int(cu[i + 1] - cu[i])
        if k <= 0:
            continue
        a = 0
        rejected = -1
        for j in range(1, k):
            p = row_probs(z[off + j - 1], temperature)
            x = int(tokens[off + j])
            p_draft[off + j] = p[x]
            if u_accept[off + j] < p[x]:
                a += 1
            else:
                rejected = x
                break
        p = row_probs(z[off + a], temperature)
        acc[i] = 1 + a
        nxt[i] = sample(p, float(u_next[i]), rejected)
    return acc, nxt, p_draft


def output_distribution(logits: np.ndarray, drafts: np.ndarray, temperature: float):
    """Exact joint law of (accepted drafts a, successor y) for one request whose rows are
    logits[0..k-1] and whose candidates are drafts[1..k-1] (drafts[0] is the anchor)."""
    k = len(drafts)
    ps = [row_probs(logits[r], temperature) for r in range(k)]
    law = {}
    reach = 1.0
    for a in range(k):
        p = ps[a]
        if a < k - 1:
            x = int(drafts[a + 1])
            rej = reach * (1.0 - p[x])
            for y in range(len(p)):
                if y != x and p[y] > 0:
                    law[(a, y)] = law.get((a, y), 0.0) + rej * p[y] / (1.0 - p[x])
            reach *= p[x]
        else:
            for y in range(len(p)):
                law[(a, y)] = law.get((a, y), 0.0) + reach * p[y]
    return law
