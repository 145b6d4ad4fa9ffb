"""Draft-signal features and ACT truncation, CPU reference in fp64 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
use this module; the CUDA library never imports it and shares no code with it.

* ``draft_features`` -- per draft-logit row, the 18 values of "DScale: Scaling
  Block-Diffusion Speculative Decoding with Adaptive Verification", SIII-C (Acceptance
  predictor): the highest logit, its gaps to ranks 2..16 (rank r = the r-th element of the
  row sorted descending as a multiset), the top token's log-probability (top logit minus
  the row's log-sum-exp) and the distribution entropy -sum p log p, p = softmax(row).
* ``act_truncate`` -- DFlash-Mini-Lab README, DFlash7-ACT: the draft suffix is cut before
  the first draft position whose top-1/top-2 margin is below the threshold; threshold 0
  keeps the full block.  Slot count k = 1 (anchor) + the number of leading positions kept.
"""
from __future__ import annotations

import numpy as np


def draft_features(logits: np.ndarray) -> np.ndarray:
    z = np.asarray(logits, dtype=np.float64)
    rows, V = z.shape
    out = np.zeros((rows, 18), dtype=np.float64)
    for r in range(rows):
        srt = np.sort(z[r])[::-1]
        top = srt[:16]
        m = srt[0]
        e = np.exp(z[r] - m)
        s = e.sum()
        lse = m + np.log(s)
        p = e / s
        ent = -float(np.sum(p * np.where(p > 0, np.log(np.where(p > 0, p, 1.0)), 0.0)))
        out[r, 0] = top[0]
        out[r, 1:16] = top[0] - top[1:16]
        out[r, 16] = top[0] - lse
        out[r, 17] = ent
    return out


def act_truncate(margins: np.ndarray, threshold: float) -> np.ndarray:
    """margins [n, W-1] (draft positions 1..W-1 in order) -> k [n]."""
    mg = np.asarray(margins, dtype=np.float64)
    n, wm1 = mg.shape
    k = np.ones(n, dtype=np.int64)
    for i in range(n):
        for j in range(wm1):
            if mg[i, j] < threshold:
                break
            k[i] += 1
    return k
