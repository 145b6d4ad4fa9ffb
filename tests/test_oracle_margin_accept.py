"""Pins for the oracle's row top-1/top-2/margin, greedy acceptance and offsets (CPU only).

Row reduction: numpy argmax (first occurrence) and a full descending sort, on tiny rows
with planted ties and infinities (DFlash-Mini-Lab README, DFlash7-ACT top-1/top-2 margin).
Acceptance: every match pattern of a block of up to 8 slots, enumerated (DScale SIII-D,
Prefix verifier; DFlash-Mini-Lab "accept exact prefix"), and the statistical closed
form E[accept_len] = 1 + sum_j prod_{i<=j} 0.8**i (= 1 + sum_k P(prefix >= k), the
accepted-length identity on the PixelML DFlash model card) on the 0.8**i decay workload.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from speculative_decoding_verification_packed_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _np_top2(row):
    row = np.asarray(row, dtype=np.float32)
    idx = int(np.argmax(row))                      # first occurrence of the maximum
    desc = np.sort(row)[::-1]
    return idx, desc[0], desc[1], np.float32(desc[0]) - np.float32(desc[1])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_top2_matches_numpy_on_random_rows(orc, dtype):
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(64, 37, generator=g) * 3).to(dtype)
    # plant exact ties: equal maxima at two positions in some rows
    x[3, 5] = x[3, 30] = 50.0
    x[4, 0] = x[4, 36] = 50.0
    x[5, :] = 1.0
    x[6, 7] = float("inf")
    x[7, :] = float("-inf"); x[7, 9] = 0.0
    x[8, 2] = float("-inf")
    idx, t1, t2, mg = orc.row_top2(x)
    xf = x.float().numpy()
    for r in range(64):
        i_ref, a, b, m = _np_top2(xf[r])
        assert idx[r] == i_ref, r
        assert t1[r] == a and t2[r] == b
        assert (np.isnan(m) and np.isnan(mg[r])) or mg[r].view(np.int32) == np.float32(m).view(np.int32)
    assert idx[3] == 5 and t2[3] == t1[3] and mg[3] == 0.0
    assert idx[4] == 0 and idx[5] == 0 and mg[5] == 0.0
    assert t1[7] == 0.0 and t2[7] == -np.inf and idx[7] == 9


def test_top2_row_stride_and_two_wide_rows(orc):
    base = torch.tensor([[1.0, 2.0, 99.0], [3.0, 3.0, 99.0], [-5.0, 7.0, 99.0]])
    idx, t1, t2, mg = orc.row_top2(base[:, :2].contiguous())
    assert idx.tolist() == [1, 0, 1]
    assert t2.tolist() == [1.0, 3.0, -5.0]
    idx2, _, _, _ = orc.row_top2(base, row_stride=3)
    assert idx2.tolist() == [2, 2, 2]


def _enumerated_accept(pattern):
    """a = position of the first False in the match pattern (or its length)."""
    for j, ok in enumerate(pattern):
        if not ok:
            return j
    return len(pattern)


def test_accept_all_match_patterns(orc):
    rng = np.random.default_rng(0)
    for k in range(1, 9):
        pats = list(itertools.product([False, True], repeat=k - 1))
        n = len(pats)
        cu = np.arange(n + 1, dtype=np.int32) * k
        argmax = rng.integers(0, 1000, size=n * k).astype(np.int32)
        tokens = np.zeros(n * k, dtype=np.int32)
        for i, p in enumerate(pats):
            off = i * k
            tokens[off] = rng.integers(0, 1000)
            for j in range(1, k):
                tgt = argmax[off + j - 1]
                tokens[off + j] = tgt if p[j - 1] else (tgt + 1 + rng.integers(0, 5)) % 1000
        acc, nxt = orc.greedy_accept(argmax, tokens, cu)
        for i, p in enumerate(pats):
            a = _enumerated_accept(p)
            assert acc[i] == 1 + a
            assert nxt[i] == argmax[i * k + a]
            assert 1 <= acc[i] <= k
        # all drafts equal to the target argmax -> accept the whole prefix
        assert acc[-1] == k


def test_accept_inactive_and_ragged(orc):
    cu = np.array([0, 3, 3, 4, 9], dtype=np.int32)   # request 1 inactive (k=0)
    argmax = np.array([5, 6, 7, 1, 2, 3, 4, 5, 6], dtype=np.int32)
    tokens = np.array([0, 5, 6, 9, 0, 2, 9, 4, 5], dtype=np.int32)
    acc, nxt = orc.greedy_accept(argmax, tokens, cu)
    assert acc.tolist() == [3, 0, 1, 2]
    assert nxt.tolist() == [7, -1, 1, 3]


def test_expected_accept_length_under_decay_workload(orc):
    # wide_gqa_bf16 draft model: draft j matches with p = 0.8**j, k = 7 slots
    closed = 1.0 + sum(0.8 ** (j * (j + 1) / 2) for j in range(1, 7))
    assert abs(closed - 2.7259) < 1e-4
    accs = []
    for seed in range(3):
        b = wl.make_batch("wide_gqa_bf16", seed=seed, n=400, hq=1, hkv=1, d=8, vocab=64,
                          ctx_lengths=[0] * 400)
        idx, _, _, _ = orc.row_top2(b.target_logits)
        assert (idx == b.planted_argmax.numpy()).all()
        acc, nxt = orc.greedy_accept(idx, b.tokens, b.cu_slots)
        accs.append(acc.astype(np.float64))
    a = np.concatenate(accs)
    se = a.std(ddof=1) / math.sqrt(a.size)
    assert abs(a.mean() - closed) < 3 * se, (a.mean(), closed, se)


def test_draft_logits_argmax_is_draft_token(orc):
    b = wl.make_batch("wide_gqa_bf16", seed=0, n=4, hq=1, hkv=1, d=8, vocab=300,
                      ctx_lengths=[0] * 4)
    idx, _, _, mg = orc.row_top2(b.draft_logits)
    drafts = b.full["tokens"][:, 1:].reshape(-1).numpy()
    assert (idx == drafts).all()
    assert (mg > 0).all()


def test_offsets_fig6_and_relayout_fig1(orc):
    ex = json.load(open(GOLDEN))
    f6 = ex["packer_fig6"]
    cu = orc.offsets(f6["lengths"])
    assert cu[:-1].tolist() == f6["offsets"] and cu[-1] == f6["end"]
    f1 = ex["relayout_fig1"]
    a, b = orc.offsets(f1["before"]), orc.offsets(f1["after"])
    assert a[-1] == b[-1] == f1["slots"]
    assert a[1] == f1["r2_start_before"] and b[1] == f1["r2_start_after"]
    # the generator's packer agrees with the oracle's
    assert wl.prefix_offsets(f6["lengths"]).tolist() == cu.tolist()


def test_inactive_row_fraction_fig1(orc):
    ex = json.load(open(GOLDEN))
    m = ex["masked_rows_fig1"]
    cap, frac = orc.inactive_row_fraction(m["rows"], m["tile"])
    assert cap - m["rows"] == m["masked"] and frac == m["masked_fraction"]
    s = ex["short_tile_fig1"]
    cap, frac = orc.inactive_row_fraction(s["rows"], s["tile"])
    assert cap - s["rows"] == s["masked"] and frac == 0.0
    assert orc.inactive_row_fraction(17, 16) == (32, 1 - 17 / 32)


def test_budget_lengths_fill_exactly():
    g = torch.Generator().manual_seed(0)
    for n in (8, 64):
        k = wl.budget_lengths(n, 8 * n, 16, g)
        assert sum(k) == 8 * n and min(k) >= 1 and max(k) <= 16
