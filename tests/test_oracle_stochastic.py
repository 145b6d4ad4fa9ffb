"""Pins of the stochastic prefix verifier reference (oracle/stochastic.py), "DScale",
SIII-D (Prefix verifier): a hand-worked example, the temperature -> 0 limit against the
greedy verifier, the lossless property (the first output token follows the target
distribution, whatever the draft), the closed form of the acceptance law, and a
Monte-Carlo check of the sampler against the exact output law."""
import numpy as np
import pytest

import oracle
from oracle import stochastic as st


def test_hand_example():
    z = np.log(np.array([[0.5, 0.3, 0.2], [0.1, 0.1, 0.8]]))
    cu = np.array([0, 2])
    tokens = np.array([9, 0])           # anchor, draft x_1 = 0
    # u_1 = 0.6 >= P(0) = 0.5: rejected; successor from {1: 0.6, 2: 0.4} with u' = 0.5 -> 1
    acc, nxt, p = st.stochastic_accept(z, tokens, cu, 1.0, np.array([0.0, 0.6]), np.array([0.5]))
    assert acc.tolist() == [1] and nxt.tolist() == [1] and p[1] == pytest.approx(0.5)
    # u' = 0.7 -> cumulative 0.6 <= 0.7 < 1.0 -> 2
    acc, nxt, _ = st.stochastic_accept(z, tokens, cu, 1.0, np.array([0.0, 0.6]), np.array([0.7]))
    assert nxt.tolist() == [2]
    # u_1 = 0.4 < 0.5: accepted; successor from row 1 unmodified, u' = 0.15 -> 1, 0.25 -> 2
    acc, nxt, _ = st.stochastic_accept(z, tokens, cu, 1.0, np.array([0.0, 0.4]), np.array([0.15]))
    assert acc.tolist() == [2] and nxt.tolist() == [1]
    acc, nxt, _ = st.stochastic_accept(z, tokens, cu, 1.0, np.array([0.0, 0.4]), np.array([0.25]))
    assert nxt.tolist() == [2]


def test_inactive_request():
    acc, nxt, _ = st.stochastic_accept(np.zeros((2, 4)), np.zeros(2, dtype=np.int32),
                                       np.array([0, 2, 2]), 1.0, np.zeros(2), np.zeros(2))
    assert acc.tolist()[1] == 0 and nxt.tolist()[1] == -1


@pytest.mark.parametrize("seed", range(5))
def test_low_temperature_is_the_greedy_verifier(seed, orc):
    rng = np.random.default_rng(seed)
    n, V = 6, 50
    ks = rng.integers(1, 9, n)
    cu = np.concatenate([[0], np.cumsum(ks)])
    m = int(cu[-1])
    z = rng.normal(0, 1, (m, V))
    am = z.argmax(axis=1)
    tokens = rng.integers(0, V, m)
    for i in range(n):          # drafts that match the argmax for a random prefix
        cut = rng.integers(0, ks[i])
        for j in range(1, int(ks[i])):
            if j <= cut:
                tokens[cu[i] + j] = am[cu[i] + j - 1]
    u = rng.uniform(0.01, 0.99, m)
    un = rng.uniform(0.01, 0.99, n)
    acc, nxt, _ = st.stochastic_accept(z, tokens, cu, 1e-4, u, un)
    g_acc, g_nxt = oracle.greedy_accept(am.astype(np.int32), tokens.astype(np.int32), cu.astype(np.int32))
    assert acc.tolist() == g_acc.tolist()
    assert nxt.tolist() == g_nxt.tolist()


@pytest.mark.parametrize("seed", range(6))
def test_first_output_token_follows_the_target(seed):
    """Lossless: token 1 of the output is x_1 if accepted, else the successor drawn with x_1
    removed; its law is P_0 whatever x_1 is."""
    rng = np.random.default_rng(10 + seed)
    V, k, T = 7, 4, float(rng.choice([0.5, 1.0, 2.0]))
    z = rng.normal(0, 1.5, (k, V))
    drafts = rng.integers(0, V, k)
    law = st.output_distribution(z, drafts, T)
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
    first = np.zeros(V)
    for (a, y), pr in law.items():
        first[int(drafts[1]) if a >= 1 else y] += pr
    assert first == pytest.approx(st.row_probs(z[0], T), abs=1e-12)
    # acceptance closed form: P(a >= j) = prod_{l < j} P_l(x_{l+1})
    for j in range(1, k):
        tail = sum(pr for (a, y), pr in law.items() if a >= j)
        prod = np.prod([st.row_probs(z[l], T)[int(drafts[l + 1])] for l in range(j)])
        assert tail == pytest.approx(prod, abs=1e-12)


def test_sampler_matches_the_exact_law():
    rng = np.random.default_rng(42)
    V, k, T, trials = 5, 3, 1.0, 40000
    z = rng.normal(0, 1.0, (k, V))
    drafts = np.array([0, int(np.argmax(z[0])), int(np.argsort(z[1])[-2])])
    law = st.output_distribution(z, drafts, T)
    reps = trials
    Z = np.tile(z, (reps, 1))
    toks = np.tile(drafts, reps)
    cu = np.arange(0, k * reps + 1, k)
    acc, nxt, _ = st.stochastic_accept(Z, toks, cu, T, rng.random(k * reps), rng.random(reps))
    counts = {}
    for a, y in zip(acc - 1, nxt):
        counts[(int(a), int(y))] = counts.get((int(a), int(y)), 0) + 1
    chi2, dof = 0.0, 0
    for key, pr in law.items():
        e = pr * reps
        if e < 5:
            continue
        chi2 += (counts.get(key, 0) - e) ** 2 / e
        dof += 1
    assert set(counts) <= set(law)
    # 99.9 % quantile of chi-square with dof - 1 degrees of freedom is below dof + 4 sqrt(2 dof) + 10
    assert chi2 < (dof - 1) + 4 * np.sqrt(2 * (dof - 1)) + 10, (chi2, dof)
