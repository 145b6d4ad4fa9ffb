"""Pins of the draft-feature and ACT-truncation references (oracle/features.py): "DScale"
SIII-C (Acceptance predictor: top logit, 15 gaps, top log-probability, entropy) and the
DFlash-Mini-Lab README (DFlash7-ACT margin threshold, threshold 0 = full block)."""
import math

import numpy as np
import pytest

import oracle
from oracle import features as ft


def test_closed_forms():
    V = 100
    # uniform row: entropy log V, top log-prob -log V, all gaps 0
    f = ft.draft_features(np.zeros((1, V)))[0]
    assert f[17] == pytest.approx(math.log(V), abs=1e-12)
    assert f[16] == pytest.approx(-math.log(V), abs=1e-12)
    assert np.all(f[1:16] == 0)
    # two levels: one logit at L, the rest 0
    L = 3.0
    z = np.zeros((1, V)); z[0, 17] = L
    f = ft.draft_features(z)[0]
    s = math.exp(L) + V - 1
    p1 = math.exp(L) / s
    assert f[0] == L and np.all(f[1:16] == L)
    assert f[16] == pytest.approx(math.log(p1), abs=1e-12)
    ent = -(p1 * math.log(p1) + (V - 1) * (1 / s) * math.log(1 / s))
    assert f[17] == pytest.approx(ent, abs=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_against_library_routines(seed, orc):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 2, (7, 300))
    z[3, 5] = z[3, 9] = z[3].max() + 1.0          # a repeated maximum: gap_2 = 0
    f = ft.draft_features(z)
    for r in range(z.shape[0]):
        srt = -np.sort(-z[r])
        assert f[r, 0] == srt[0]
        assert f[r, 1:16].tolist() == (srt[0] - srt[1:16]).tolist()
        lse = np.logaddexp.reduce(z[r])
        assert f[r, 16] == pytest.approx(srt[0] - lse, abs=1e-12)
        p = np.exp(z[r] - lse)
        assert f[r, 17] == pytest.approx(float(-(p * np.log(p)).sum()), abs=1e-10)
    assert f[3, 1] == 0.0
    # gap_2 is the top-1/top-2 margin of the margin reference (fp32 inputs)
    z32 = z.astype(np.float32)
    _, _, _, mg = oracle.row_top2(z32)
    f32 = ft.draft_features(z32)
    assert np.allclose(f32[:, 1], mg, atol=0, rtol=0)


def test_act_truncate():
    mg = np.array([[3.0, 2.5, 0.4, 5.0], [0.1, 9.0, 9.0, 9.0], [1.0, 1.0, 1.0, 1.0]])
    assert ft.act_truncate(mg, 0.0).tolist() == [5, 5, 5]        # threshold 0: full block
    assert ft.act_truncate(mg, 1.0).tolist() == [3, 1, 5]
    assert ft.act_truncate(mg, 2.0).tolist() == [3, 1, 1]
    assert ft.act_truncate(mg, 1e9).tolist() == [1, 1, 1]
