"""Pins of the DVL budget allocator and flat-buffer packer reference (oracle/dvl.py).

"DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification", SIII-C
(Algorithm 1, Fig. 6, Complexity analysis) and SIV (retention).  The pins do not retype the
reference: Fig. 6's printed lengths and offsets, brute-force optimality of the adjusted
lengths on tiny inputs, the 7N adjustment bound, the tie rule, pack/unpack round trips
and a hand-computed retention value.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import dvl

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def _scores_from_rows(rows, w=16):
    """Acceptance scores of draft positions 1..w-1 from explicit per-request lists."""
    s = np.zeros((len(rows), w - 1), dtype=np.float32)
    for i, r in enumerate(rows):
        s[i, :len(r)] = r
    return s


# Scores built so that the rounded sums are Fig. 6's initial lengths [5, 10, 7, 9] and R1's
# next slot (0.6) beats the others (0.55, 0.52, 0.51).
FIG6_GROW = [[1, 1, 1, 1, 0.6], [1] * 9 + [0.55], [1] * 6 + [0.52], [1] * 8 + [0.51]]
# Same initial lengths, but R2's last slot (0.75) is the lowest last slot.
FIG6_SHRINK = [[1, 1, 1, 1, 0.6], [1] * 8 + [0.75, 0.75], [1] * 6 + [0.52], [1] * 8 + [0.51]]


def test_fig6_growth():
    g = GOLD["allocator_fig6"]
    r = dvl.dvl_allocate_pack(_scores_from_rows(FIG6_GROW), n_live=4, budget_per_req=8, m_cap=64)
    assert r["k0"].tolist() == g["initial"]
    assert r["k"].tolist() == g["grown"]
    assert r["cu"][:-1].tolist() == GOLD["packer_fig6"]["offsets"]
    assert int(r["cu"][-1]) == GOLD["packer_fig6"]["end"] == g["budget"]
    assert r["adjustments"] == 1


def test_fig6_alternative_shrinkage():
    g = GOLD["allocator_fig6"]
    r = dvl.dvl_allocate_pack(_scores_from_rows(FIG6_SHRINK), n_live=4, budget_per_req=8, m_cap=64)
    assert r["k0"].tolist() == g["initial"]
    # budget 30 < 31: the lowest last slot, R2's tail, is removed
    q = r["q"]
    k, adj = dvl.allocate(q, r["k0"], 4, 30)
    expect = list(g["initial"])
    expect[g["shrink_request"]] -= 1
    assert k.tolist() == expect and adj == 1


def test_prefix_scores_are_cumulative_minima():
    s = np.array([[0.9, 0.95, 0.4, 0.6, 0.1]], dtype=np.float32)
    q = dvl.prefix_scores(s)
    assert q[0].tolist() == pytest.approx([1.0, 0.9, 0.9, 0.4, 0.4, 0.1])
    assert np.all(np.diff(q[0]) <= 0)


def test_rounding_ties_to_even_and_clip():
    w = 8
    # sums 2.5 -> 2, 3.5 -> 4, 0 -> clipped to 1, 7 (all ones) -> 7 (<= W)
    rows = [[1, 1, 0.5], [1, 1, 1, 0.5], [0.0], [1] * 7]
    q = dvl.prefix_scores(_scores_from_rows(rows, w))
    assert dvl.initial_lengths(q, 4).tolist() == [2, 4, 1, 7]


def _objective(q, k):
    return sum(float(q[i, :k[i]].sum(dtype=np.float64)) for i in range(len(k)))


@pytest.mark.parametrize("seed", range(40))
def test_adjusted_lengths_are_optimal_on_tiny_inputs(seed):
    """Growing picks the best next slots, shrinking drops the worst tails: with distinct
    scores the result is the unique maximiser of the summed prefix scores among lengths on
    the same side of k0 with the budget's total."""
    rng = np.random.default_rng(seed)
    n, w = 3, 5
    s = rng.random((n, w - 1)).astype(np.float32)
    q = dvl.prefix_scores(s)
    k0 = dvl.initial_lengths(q, n)
    for budget in range(n, n * w + 1):
        k, adj = dvl.allocate(q, k0, n, budget)
        assert int(k.sum()) == budget and adj == abs(budget - int(k0.sum()))
        grow = budget >= k0.sum()
        best, best_k = None, None
        for cand in itertools.product(range(1, w + 1), repeat=n):
            if sum(cand) != budget:
                continue
            if grow and any(c < a for c, a in zip(cand, k0)):
                continue
            if not grow and any(c > a for c, a in zip(cand, k0)):
                continue
            v = _objective(q, cand)
            if best is None or v > best + 1e-12:
                best, best_k = v, cand
        assert _objective(q, k) == pytest.approx(best, abs=1e-9)
        if len(set(q[:, 1:].ravel().tolist())) == q[:, 1:].size:
            assert tuple(k.tolist()) == best_k


def test_ties_go_to_the_lowest_request():
    w = 6
    s = np.full((3, w - 1), 0.5, dtype=np.float32)        # equal scores everywhere
    q = dvl.prefix_scores(s)
    k0 = np.array([2, 2, 2])
    k, _ = dvl.allocate(q, k0, 3, 7)                       # one slot to give
    assert k.tolist() == [3, 2, 2]
    k, _ = dvl.allocate(q, k0, 3, 5)                       # one slot to take
    assert k.tolist() == [1, 2, 2]


@pytest.mark.parametrize("seed", range(20))
def test_adjustment_bound_for_w16(seed):
    b = GOLD["adjustment_bound"]
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 200))
    w = b["W"]
    for s in (rng.random((n, w - 1)), np.ones((n, w - 1)), np.zeros((n, w - 1)),
              rng.beta(0.3, 0.3, (n, w - 1))):
        r = dvl.dvl_allocate_pack(s.astype(np.float32), n_live=n, budget_per_req=b["per_request_budget"],
                                  m_cap=w * n)
        assert r["adjustments"] <= b["max_adjustments_per_request"] * n
        assert int(r["k"].sum()) == b["per_request_budget"] * n
        assert r["k"].min() >= 1 and r["k"].max() <= w


def test_pack_round_trip_inactive_and_tail():
    rng = np.random.default_rng(7)
    n_bs, n_live, w, per = 6, 4, 16, 8
    s = rng.random((n_bs, w - 1)).astype(np.float32)
    tok = rng.integers(0, 1000, (n_bs, w))
    pos = rng.integers(0, 4096, (n_bs, w))
    ref = rng.integers(0, 10 ** 6, (n_bs, w))
    m_cap = 16 * n_bs
    r = dvl.dvl_allocate_pack(s, n_live, per, m_cap, tok, pos, ref, fill_token=7, fill_pos=-3, fill_ref=-1)
    k, cu = r["k"], r["cu"]
    m_live = per * n_live
    assert k[n_live:].tolist() == [0] * (n_bs - n_live)
    assert cu[n_live:].tolist() == [m_live] * (n_bs - n_live + 1)
    for name, f, fill in (("tokens", tok, 7), ("positions", pos, -3), ("kv_refs", ref, -1)):
        packed = r[name]
        for i in range(n_bs):
            assert packed[cu[i]:cu[i] + k[i]].tolist() == f[i, :k[i]].tolist()
        assert packed[m_live:].tolist() == [fill] * (m_cap - m_live)


def test_retention_hand_example():
    y = [3, 10, 0, 5]
    k = [4, 8, 1, 6]
    # min(3,3) + min(10,7) + min(0,0) + min(5,5) = 15 of 18 accepted tokens
    assert dvl.retention(y, k) == pytest.approx(15 / 18)
