"""GPU parity of svp_stochastic_accept against the fp64 stochastic prefix verifier
(oracle/stochastic.py), "DScale" SIII-D.  Decisions are compared exactly except where a
uniform draw lies within rounding of its boundary (then either side is valid and the
GPU's choice is checked against the oracle's bracket); acceptance probabilities to 2e-5;
the output law of many replicated requests against the exact law (chi-square)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_packed_gb300 as svp
from oracle import stochastic as st

pytestmark = pytest.mark.gpu
TOL = 2e-5


def _batch(seed, n, V, dtype, kmax=16):
    rng = np.random.default_rng(seed)
    ks = rng.integers(0, kmax + 1, n)
    ks[rng.integers(0, n)] = kmax
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    m = int(cu[-1]) + 3
    z = torch.randn(m, V, generator=torch.Generator().manual_seed(seed)) * 2.0
    z = z.to(dtype)
    zf = z.float().numpy().astype(np.float64)
    am = zf.argmax(axis=1)
    tok = rng.integers(0, V, m).astype(np.int32)
    for i in range(n):
        for j in range(1, int(ks[i])):
            if rng.random() < 0.6:
                tok[cu[i] + j] = am[cu[i] + j - 1]
    ua = rng.random(m).astype(np.float32)
    un = rng.random(n).astype(np.float32)
    return z, zf, tok, cu, ua, un


def _borderline(zf, tok, cu, T, ua, un, i, y_gpu):
    """True when request i's outcome sits within TOL of a decision boundary."""
    off, k = int(cu[i]), int(cu[i + 1] - cu[i])
    a, excl = 0, -1
    for j in range(1, k):
        p = st.row_probs(zf[off + j - 1], T)[int(tok[off + j])]
        if abs(float(ua[off + j]) - p) < TOL:
            return True
        if ua[off + j] < p:
            a += 1
        else:
            excl = int(tok[off + j])
            break
    p = st.row_probs(zf[off + a], T)
    w = p.copy()
    if excl >= 0:
        w[excl] = 0.0
    c = np.cumsum(w) / w.sum()
    t = float(un[i])
    lo = c[y_gpu - 1] if y_gpu > 0 else 0.0
    return lo - TOL <= t <= c[y_gpu] + TOL


@pytest.mark.parametrize("case", [(0, 8, 512, torch.bfloat16, 1.0), (1, 20, 10000, torch.bfloat16, 0.7),
                                  (2, 6, 40000, torch.bfloat16, 1.5), (3, 12, 3000, torch.float32, 1.0)])
def test_matches_reference(case):
    seed, n, V, dtype, T = case
    z, zf, tok, cu, ua, un = _batch(seed, n, V, dtype)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    ws = svp.Workspace(svp.stochastic_accept_workspace_size(z.shape[0], V))
    acc, nxt, pd = svp.stochastic_accept(z.cuda(), d(tok), d(cu), d(ua), d(un), temperature=T, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    o_acc, o_nxt, o_pd = st.stochastic_accept(zf, tok, cu, T, ua.astype(np.float64), un.astype(np.float64))
    acc, nxt, pd = acc.cpu().numpy(), nxt.cpu().numpy(), pd.cpu().numpy()
    tested = ~np.isnan(o_pd) & ~np.isnan(pd)
    assert np.abs(pd[tested] - o_pd[tested]).max() <= TOL
    mism = 0
    for i in range(n):
        if acc[i] != o_acc[i] or nxt[i] != o_nxt[i]:
            mism += 1
            assert _borderline(zf, tok, cu, T, ua, un, i, int(nxt[i])), (i, acc[i], o_acc[i], nxt[i], o_nxt[i])
    assert mism <= max(1, n // 50)
    assert set(np.where(np.diff(cu) == 0)[0].tolist()) <= set(np.where(acc == 0)[0].tolist())


def test_low_temperature_equals_greedy():
    n, V = 16, 4096
    z, zf, tok, cu, ua, un = _batch(7, n, V, torch.bfloat16)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    acc, nxt, _ = svp.stochastic_accept(z.cuda(), d(tok), d(cu), d(ua), d(un), temperature=1e-4)
    idx, _, _, _ = oracle.row_top2(z)
    g_acc, g_nxt = oracle.greedy_accept(idx, tok, cu)
    assert acc.cpu().tolist() == g_acc.tolist()
    assert nxt.cpu().tolist() == g_nxt.tolist()


def test_output_law_of_replicated_requests():
    rng = np.random.default_rng(11)
    V, k, T, reps = 6, 3, 1.0, 20000
    zr = rng.normal(0, 1.0, (k, V))
    drafts = np.array([0, int(np.argmax(zr[0])), int(np.argsort(zr[1])[-2])], dtype=np.int32)
    z = torch.from_numpy(np.tile(zr, (reps, 1)).astype(np.float32))
    tok = np.tile(drafts, reps)
    cu = np.arange(0, k * reps + 1, k).astype(np.int32)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    acc, nxt, _ = svp.stochastic_accept(z.cuda(), d(tok), d(cu), d(rng.random(k * reps).astype(np.float32)),
                                        d(rng.random(reps).astype(np.float32)), temperature=T)
    law = st.output_distribution(z.numpy()[:k].astype(np.float64), drafts, T)
    counts = {}
    for a, y in zip(acc.cpu().numpy() - 1, nxt.cpu().numpy()):
        counts[(int(a), int(y))] = counts.get((int(a), int(y)), 0) + 1
    assert set(counts) <= set(law)
    chi2, dof = 0.0, 0
    for key, pr in law.items():
        e = pr * reps
        if e >= 5:
            chi2 += (counts.get(key, 0) - e) ** 2 / e
            dof += 1
    assert chi2 < (dof - 1) + 4 * np.sqrt(2 * (dof - 1)) + 10, (chi2, dof)


def test_invalid_slots_set_status_and_empty_results():
    """A decreasing cu_slots is rejected on the device: status bit, every request 0 / -1, and
    the workspace stays usable (a valid call right after agrees with the reference)."""
    n, V = 4, 3000
    z, zf, tok, cu, ua, un = _batch(21, n, V, torch.bfloat16, kmax=6)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    ws = svp.Workspace(svp.stochastic_accept_workspace_size(z.shape[0], V))
    bad = cu.copy()
    bad[1] = bad[2] + 1            # cu_slots[1] > cu_slots[2]: a decrease
    acc, nxt, _ = svp.stochastic_accept(z.cuda(), d(tok), d(bad), d(ua), d(un), temperature=1.0, ws=ws)
    assert ws.read_status() != 0
    assert acc.cpu().tolist() == [0] * n and nxt.cpu().tolist() == [-1] * n
    acc, nxt, _ = svp.stochastic_accept(z.cuda(), d(tok), d(cu), d(ua), d(un), temperature=1.0, ws=ws)
    ref_acc, ref_nxt, _ = st.stochastic_accept(zf, tok, cu, 1.0, ua.astype(np.float64), un.astype(np.float64))
    assert ws.read_status() == 0
    a, y = acc.cpu().numpy(), nxt.cpu().numpy()
    for i in range(n):
        if not _borderline(zf, tok, cu, 1.0, ua, un, i, int(y[i])):
            assert (a[i], y[i]) == (ref_acc[i], ref_nxt[i])


def test_full_size_wide_gqa_sampled_requests():
    """The launch the bench times: 224 target rows x 248,320 bf16 (32 requests of 7 slots),
    T = 1; sampled requests against the oracle run on their own rows."""
    from speculative_decoding_verification_packed_gb300 import workloads as wl
    b = wl.make_batch("wide_gqa_bf16", seed=0, device="cuda")
    V = b.target_logits.shape[1]
    rng = np.random.default_rng(21)
    ua = rng.random(b.m_cap).astype(np.float32)
    un = rng.random(b.n).astype(np.float32)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    ws = svp.Workspace(svp.stochastic_accept_workspace_size(b.m_cap, V))
    acc, nxt, pd = svp.stochastic_accept(b.target_logits, b.tokens, b.cu_slots, d(ua), d(un),
                                         temperature=1.0, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    acc, nxt, pd = acc.cpu().numpy(), nxt.cpu().numpy(), pd.cpu().numpy()
    cu = b.cu_slots.cpu().numpy()
    tok = b.tokens.cpu().numpy()
    for i in (0, 5, 13, 22, 31):
        lo, hi = int(cu[i]), int(cu[i + 1])
        zf = b.target_logits[lo:hi].float().cpu().numpy().astype(np.float64)
        cu1 = np.array([0, hi - lo], dtype=np.int32)
        o_acc, o_nxt, o_pd = st.stochastic_accept(zf, tok[lo:hi], cu1, 1.0, ua[lo:hi].astype(np.float64),
                                                  un[i:i + 1].astype(np.float64))
        tested = ~np.isnan(o_pd) & ~np.isnan(pd[lo:hi])
        assert np.abs(pd[lo:hi][tested] - o_pd[tested]).max(initial=0.0) <= TOL
        if acc[i] != o_acc[0] or nxt[i] != o_nxt[0]:
            assert _borderline(zf, tok[lo:hi], cu1, 1.0, ua[lo:hi], un[i:i + 1], 0, int(nxt[i])), \
                (i, acc[i], o_acc[0], nxt[i], o_nxt[0])


def test_requests_longer_than_a_warp():
    """Requests of up to 45 slots at a low temperature: the acceptance chain runs past the
    first 32 candidates (those are loaded before the wait on the statistics pass, the rest
    after it), with one planted late rejection."""
    n, V, T = 4, 3000, 0.02
    z, zf, tok, cu, ua, un = _batch(12, n, V, torch.bfloat16, kmax=45)
    am = zf.argmax(axis=1)
    for i in range(n):
        for j in range(1, int(cu[i + 1] - cu[i])):
            tok[cu[i] + j] = am[cu[i] + j - 1]
    big = int(np.argmax(np.diff(cu)))
    if cu[big + 1] - cu[big] > 40:
        tok[cu[big] + 40] = (am[cu[big] + 39] + 1) % V   # a late rejection (almost surely)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    ws = svp.Workspace(svp.stochastic_accept_workspace_size(z.shape[0], V))
    acc, nxt, pd = svp.stochastic_accept(z.cuda(), d(tok), d(cu), d(ua), d(un), temperature=T, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    o_acc, o_nxt, o_pd = st.stochastic_accept(zf, tok, cu, T, ua.astype(np.float64), un.astype(np.float64))
    acc, nxt, pd = acc.cpu().numpy(), nxt.cpu().numpy(), pd.cpu().numpy()
    tested = ~np.isnan(o_pd) & ~np.isnan(pd)
    assert np.abs(pd[tested] - o_pd[tested]).max() <= TOL
    assert int(o_acc.max()) > 33   # the chain did go past one warp of candidates
    for i in range(n):
        if acc[i] != o_acc[i] or nxt[i] != o_nxt[i]:
            assert _borderline(zf, tok, cu, T, ua, un, i, int(nxt[i])), (i, acc[i], o_acc[i], nxt[i], o_nxt[i])


def test_graph_replay_matches_eager():
    """The two launches captured in a CUDA graph (the acceptance pass a programmatic
    dependent of the statistics pass) over two alternating input sets reproduce the eager
    results bit for bit, replay after replay, on one shared workspace."""
    n, V = 12, 20000
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    sets = []
    for seed in (31, 32):
        z, zf, tok, cu, ua, un = _batch(seed, n, V, torch.bfloat16)
        sets.append((z.cuda(), d(tok), d(cu), d(ua), d(un)))
    m_cap = max(s[0].shape[0] for s in sets)
    ws = svp.Workspace(svp.stochastic_accept_workspace_size(m_cap, V))
    eager = []
    for s in sets:
        r = svp.stochastic_accept(*s, temperature=0.8, ws=ws)
        eager.append([x.clone() for x in r])
    torch.cuda.synchronize()
    outs = [(torch.empty(n, dtype=torch.int32, device="cuda"), torch.empty(n, dtype=torch.int32, device="cuda"),
             torch.full((s[0].shape[0],), float("nan"), device="cuda")) for s in sets]
    g = torch.cuda.CUDAGraph()
    strm = torch.cuda.Stream()
    strm.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(strm):
        with torch.cuda.graph(g, stream=strm):
            for s, o in zip(sets, outs):
                svp.stochastic_accept(*s, temperature=0.8, ws=ws, outs=o, stream=strm)
    torch.cuda.synchronize()
    for _ in range(3):
        for o in outs:
            o[0].fill_(-7)
            o[1].fill_(-7)
            o[2].fill_(float("nan"))   # entries of untested candidates stay unwritten
        g.replay()
        torch.cuda.synchronize()
        for e, o in zip(eager, outs):
            assert torch.equal(e[0], o[0]) and torch.equal(e[1], o[1])
            assert torch.equal(torch.nan_to_num(e[2], nan=-1.0), torch.nan_to_num(o[2], nan=-1.0))
    assert ws.read_status() == 0


def test_workspace_reused_across_sizes():
    """One workspace, sized for the largest call, serves calls with other m_cap and
    vocabularies: every call leaves it zeroed (tickets, row and chunk statistics), so no
    stale statistic lands in a later call's row tickets (the layout moves with m_cap)."""
    cases = [(30, 1000, torch.bfloat16), (8, 32000, torch.bfloat16), (40, 3000, torch.float32),
             (4, 151936, torch.bfloat16), (25, 500, torch.bfloat16)]
    batches = [_batch(60 + i, n, V, dtype) for i, (n, V, dtype) in enumerate(cases)]
    ws = svp.Workspace(max(svp.stochastic_accept_workspace_size(b[0].shape[0], V)
                           for b, (_, V, _) in zip(batches, cases)))
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    for (n, V, dtype), (z, zf, tok, cu, ua, un) in zip(cases, batches):
        acc, nxt, pd = svp.stochastic_accept(z.cuda(), d(tok), d(cu), d(ua), d(un), temperature=1.0, ws=ws)
        torch.cuda.synchronize()
        assert ws.read_status() == 0
        o_acc, o_nxt, o_pd = st.stochastic_accept(zf, tok, cu, 1.0, ua.astype(np.float64), un.astype(np.float64))
        acc, nxt, pd = acc.cpu().numpy(), nxt.cpu().numpy(), pd.cpu().numpy()
        tested = ~np.isnan(o_pd) & ~np.isnan(pd)
        assert np.abs(pd[tested] - o_pd[tested]).max(initial=0.0) <= TOL
        for i in range(n):
            if acc[i] != o_acc[i] or nxt[i] != o_nxt[i]:
                assert _borderline(zf, tok, cu, 1.0, ua, un, i, int(nxt[i])), (n, V, i)
        assert torch.count_nonzero(ws.buf[256:]).item() == 0   # all zero again past the header


def test_p_draft_is_optional():
    """p_draft may be NULL: accept_len and next_token equal those of a call that writes it."""
    n, V = 10, 5000
    z, zf, tok, cu, ua, un = _batch(71, n, V, torch.bfloat16)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    args = (z.cuda(), d(tok), d(cu), d(ua), d(un))
    acc1, nxt1, pd1 = svp.stochastic_accept(*args, temperature=0.9)
    outs = (torch.full((n,), -5, dtype=torch.int32, device="cuda"),
            torch.full((n,), -5, dtype=torch.int32, device="cuda"), None)
    acc2, nxt2, pd2 = svp.stochastic_accept(*args, temperature=0.9, outs=outs)
    torch.cuda.synchronize()
    assert pd2 is None
    assert torch.equal(acc1, acc2) and torch.equal(nxt1, nxt2)
