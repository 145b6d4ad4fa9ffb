"""DVL budget allocator and flat-buffer packer, CPU reference -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
use this module; the CUDA library never imports it and shares no code with it.

Follows "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification",
SIII-C (Acceptance predictor, Budget allocator, Flat-buffer packer; Algorithm 1, Fig. 6),
step by step in the page's order:

1. prefix scores: q[i, 0] = 1 for the anchor; q[i, j] = min(q[i, j-1], s[i, j-1]) for the
   acceptance scores s of draft positions j = 1..W-1 (cumulative minimum: acceptance needs
   accepted predecessors);
2. initial length: the W-1 prefix scores of a live request are summed into the estimated
   accepted draft count, rounded and clipped to [1, W] (one anchor plus candidates);
3. budget gap: delta = budget - sum(k);
4. while delta > 0: the live request whose next slot q[i, k_i] scores highest (k_i < W)
   grows by one slot;
5. while delta < 0: the live request whose last slot q[i, k_i - 1] scores lowest (k_i > 1)
   loses it; the anchor is never removed;
6. offsets: exclusive prefix sums of k; inactive requests (the bucket entries past the
   live count) have k = 0 and therefore offset = budget end;
7. packing: row offset_i + j of every field takes field[i, j] for j < k_i; rows past the
   live slots hold the field's placeholder.

Readings where the page is silent: the score sum and the
rounding are done in fp32 (the kernel's precision, because they decide integers), adding
positions 1..W-1 in order; rounding is to nearest, ties to even; ties between requests go
to the lowest request index, both when growing and when shrinking; the budget is
``budget_per_req * n_live``; growing stops early when every live request is at W, and
shrinking when every live request is at 1.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np


def prefix_scores(scores: np.ndarray) -> np.ndarray:
    """[n, W-1] acceptance scores -> [n, W] non-increasing prefix scores with q[:, 0] = 1."""
    s = np.asarray(scores, dtype=np.float32)
    n, wm1 = s.shape
    q = np.ones((n, wm1 + 1), dtype=np.float32)
    for i in range(n):
        for j in range(1, wm1 + 1):
            q[i, j] = min(q[i, j - 1], s[i, j - 1])
    return q


def initial_lengths(q: np.ndarray, n_live: int) -> np.ndarray:
    """k^(0): fp32 sum of the draft prefix scores, rounded (ties to even), clipped to [1, W]."""
    n, w = q.shape
    k0 = np.zeros(n, dtype=np.int64)
    for i in range(n_live):
        acc = np.float32(0.0)
        for j in range(1, w):
            acc = np.float32(acc + q[i, j])
        k0[i] = int(min(max(np.rint(acc), 1), w))
    return k0


def allocate(q: np.ndarray, k0: np.ndarray, n_live: int, budget: int):
    """Grow / shrink loop of Algorithm 1.  Returns (k, number of adjustments)."""
    n, w = q.shape
    k = np.array(k0, dtype=np.int64)
    delta = budget - int(k.sum())
    adjustments = 0
    while delta > 0:
        best = -1
        for i in range(n_live):
            if k[i] < w and (best < 0 or q[i, k[i]] > q[best, k[best]]):
                best = i
        if best < 0:
            break
        k[best] += 1
        delta -= 1
        adjustments += 1
    while delta < 0:
        worst = -1
        for i in range(n_live):
            if k[i] > 1 and (worst < 0 or q[i, k[i] - 1] < q[worst, k[worst] - 1]):
                worst = i
        if worst < 0:
            break
        k[worst] -= 1
        delta += 1
        adjustments += 1
    return k, adjustments


def offsets(k: np.ndarray) -> np.ndarray:
    cu = np.zeros(len(k) + 1, dtype=np.int64)
    for i in range(len(k)):
        cu[i + 1] = cu[i] + k[i]
    return cu


def pack(field: np.ndarray, k: np.ndarray, cu: np.ndarray, m_cap: int, fill: int) -> np.ndarray:
    """Row offset_i + j <- field[i, j] for j < k_i; every other row <- fill."""
    out = np.full(m_cap, fill, dtype=np.int64)
    for i in range(len(k)):
        for j in range(int(k[i])):
            out[cu[i] + j] = field[i, j]
    return out


def retention(y: np.ndarray, k: np.ndarray) -> float:
    """Accepted-token retention of windows k (anchor included) for full-width labels y
    (DScale SIV, Predictor quality and budget adjustment): sum min(y, k-1) / sum y."""
    y = np.asarray(y, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    den = int(y.sum())
    return float(np.minimum(y, k - 1).sum()) / den if den else 1.0


def dvl_allocate_pack(scores: np.ndarray, n_live: int, budget_per_req: int, m_cap: int,
                      tokens: Optional[np.ndarray] = None, positions: Optional[np.ndarray] = None,
                      kv_refs: Optional[np.ndarray] = None, fill_token: int = 0, fill_pos: int = 0,
                      fill_ref: int = -1) -> Dict[str, np.ndarray]:
    q = prefix_scores(scores)
    k0 = initial_lengths(q, n_live)
    budget = budget_per_req * n_live
    k, adj = allocate(q, k0, n_live, budget)
    cu = offsets(k)
    out = dict(q=q, k0=k0, k=k, cu=cu, adjustments=adj)
    for name, field, fill in (("tokens", tokens, fill_token), ("positions", positions, fill_pos),
                              ("kv_refs", kv_refs, fill_ref)):
        if field is not None:
            out[name] = pack(np.asarray(field), k, cu, m_cap, fill)
    return out
