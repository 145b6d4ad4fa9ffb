"""GPU parity on seeded random configurations against the fp64 oracle: verification
attention (short tile, wide tile for blocks wider than 16, fp32 CUDA-core path), causal
prefill, fused margin + accept, the stochastic prefix verifier and the draft features.

Each case draws its shape at random (fixed seeds, so every run checks the same cases): the
number of requests, their slot counts (0 = inactive, up to 16) and context lengths (0 to
a few thousand, ending anywhere within a 128-key tile or a 16-token page), the head dim
(128 or 256), the query heads per KV head (1 to 12), contiguous or paged context, and the
tile mode.  Packed tail rows are poisoned with NaN and must stay unread and unwritten.
The logit-row cases draw the vocabulary, a padded row stride, the dtype and the value
scale, with empty requests, tie-heavy rows and rows with -inf entries.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_packed_gb300 as svp
from speculative_decoding_verification_packed_gb300 import workloads as wl
from helpers import check_margin_rows, compare_attention, gpu_verify, oracle_verify, rows_of, to_dev

pytestmark = pytest.mark.gpu

_GROUPS = {128: [(4, 4), (8, 2), (8, 1), (6, 6), (12, 1), (32, 8)],
           256: [(12, 1), (24, 2), (4, 2), (2, 2)]}
_MODES = [svp.TILE_AUTO, svp.TILE_AUTO, svp.TILE_SHORT_UNPACKED, svp.TILE_FIXED128]


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    d = int(rng.choice([128, 256]))
    hq, hkv = _GROUPS[d][int(rng.integers(len(_GROUPS[d])))]
    n = int(rng.integers(1, 7))
    lengths = [int(x) for x in rng.integers(0, 17, size=n)]
    if sum(lengths) == 0:
        lengths[0] = 1
    ctx = [int(x) if rng.random() < 0.8 else 0 for x in rng.integers(1, 3000, size=n)]
    paged = bool(rng.random() < 0.5)
    mode = _MODES[int(rng.integers(len(_MODES)))]
    if mode == svp.TILE_FIXED128 and d == 256:
        mode = svp.TILE_AUTO              # the fixed-tile contrast serves d <= 128
    return d, hq, hkv, lengths, ctx, paged, mode


@pytest.mark.parametrize("seed", range(12))
def test_random_verify_configs(seed):
    d, hq, hkv, lengths, ctx, paged, mode = _draw(seed)
    b = wl.make_batch("paged_n64_bf16" if paged else "budget8n_bf16", seed=seed, n=len(lengths),
                      lengths=lengths, ctx_lengths=ctx, hq=hq, hkv=hkv, d=d, poison=True,
                      with_logits=False)
    out, lse = gpu_verify(to_dev(b), tile_mode=mode)
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)
    assert torch.isnan(out[b.m_live:].float()).all()


@pytest.mark.parametrize("seed", range(6))
def test_random_margin_accept_configs(seed):
    rng = np.random.default_rng(2000 + seed)
    n = int(rng.integers(1, 40))
    lengths = [int(x) for x in rng.integers(0, 17, size=n)]
    if sum(lengths) == 0:
        lengths[0] = 1
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    m_cap = int(cu[-1]) + int(rng.integers(0, 5))
    vocab = int(rng.choice([7, 513, 32000, 151936]))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    g = torch.Generator().manual_seed(seed)
    logits = (torch.randn(max(m_cap, 1), vocab, generator=g) * 2).to(dtype)
    logits[int(cu[-1]):] = float("nan")                         # tail rows: never read
    live = int(cu[-1])
    amax = logits[:live].float().argmax(-1).to(torch.int32) if live else torch.zeros(0, dtype=torch.int32)
    tokens = torch.randint(0, vocab, (max(m_cap, 1),), generator=g, dtype=torch.int32)
    for i in range(n):                                           # random accepted prefixes
        off, k = int(cu[i]), lengths[i]
        stop = int(rng.integers(0, max(k, 1)))
        for j in range(1, k):
            if j <= stop:
                tokens[off + j] = amax[off + j - 1]
    outs = svp.margin_accept(logits.cuda(), tokens.cuda(), cu.cuda())
    torch.cuda.synchronize()
    r_idx = check_margin_rows(logits[:live], [o[:live] for o in outs[:4]])
    acc, nxt = oracle.greedy_accept(np.concatenate([r_idx, np.zeros(max(m_cap, 1) - live, np.int32)]),
                                    tokens, cu)
    assert np.array_equal(outs[4].cpu().numpy(), acc)
    assert np.array_equal(outs[5].cpu().numpy(), nxt)


@pytest.mark.parametrize("seed", range(6))
def test_random_stochastic_configs(seed):
    """Stochastic prefix verifier on random shapes: request count and lengths (empty ones
    included), vocabulary (2 to 151,936, odd sizes), padded row stride, dtype and
    temperature; decisions exact unless within rounding of their boundary, acceptance
    probabilities to the same bar as the fixed cases."""
    from oracle import stochastic as st
    from test_gpu_stochastic import TOL, _borderline
    rng = np.random.default_rng(3000 + seed)
    n = int(rng.integers(1, 25))
    V = [2, 17, 1000, 32000, 151936, 4099][seed]
    pad = int(rng.integers(0, 10))
    dtype = torch.float32 if seed in (1, 4) else torch.bfloat16
    T = float(rng.choice([0.3, 0.7, 1.0, 2.0]))
    ks = rng.integers(0, 21, n)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    m = max(int(cu[-1]) + int(rng.integers(0, 4)), 1)
    g = torch.Generator().manual_seed(seed)
    z = (torch.randn(m, V + pad, generator=g) * float(rng.choice([1.0, 2.0, 4.0]))).to(dtype)
    zf = z.float().numpy()[:, :V].astype(np.float64)
    am = zf.argmax(axis=1)
    tok = rng.integers(0, V, m).astype(np.int32)
    for i in range(n):
        for j in range(1, int(ks[i])):
            if rng.random() < 0.6:
                tok[cu[i] + j] = am[cu[i] + j - 1]
    ua = rng.random(m).astype(np.float32)
    un = rng.random(n).astype(np.float32)
    d = lambda a: torch.from_numpy(np.asarray(a)).cuda()
    ws = svp.Workspace(svp.stochastic_accept_workspace_size(m, V))
    acc, nxt, pd = svp.stochastic_accept(z.cuda(), d(tok), d(cu), d(ua), d(un), temperature=T, vocab=V, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    o_acc, o_nxt, o_pd = st.stochastic_accept(zf, tok, cu, T, ua.astype(np.float64), un.astype(np.float64))
    acc, nxt, pd = acc.cpu().numpy(), nxt.cpu().numpy(), pd.cpu().numpy()
    tested = ~np.isnan(o_pd) & ~np.isnan(pd)
    assert np.abs(pd[tested] - o_pd[tested]).max(initial=0.0) <= TOL
    for i in range(n):
        if acc[i] != o_acc[i] or nxt[i] != o_nxt[i]:
            assert _borderline(zf, tok, cu, T, ua, un, i, int(nxt[i])), (i, acc[i], o_acc[i], nxt[i], o_nxt[i])
    assert set(np.where(ks == 0)[0].tolist()) <= set(np.where(acc == 0)[0].tolist())


@pytest.mark.parametrize("seed", range(6))
def test_random_features_configs(seed):
    """Draft features on random shapes: rows (1 to 300), vocabulary (16 to 60,000, odd sizes),
    padded row stride, dtype, value scale, rows quantised to a coarse grid (many ties) and
    rows with up to a third of their entries -inf."""
    from oracle import features as ft
    rng = np.random.default_rng(4000 + seed)
    rows = int(rng.integers(1, 301))
    V = [16, 100, 4097, 32000, 60000, 4099][seed]
    pad = int(rng.integers(0, 10))
    dtype = torch.float32 if seed in (2, 5) else torch.bfloat16
    g = torch.Generator().manual_seed(100 + seed)
    z = torch.randn(rows, V + pad, generator=g) * float(rng.choice([0.5, 2.0, 8.0]))
    for r in range(rows):
        u = rng.random()
        if u < 0.15:
            z[r] = torch.round(z[r] * 2.0) / 2.0              # coarse grid: many equal values
        elif u < 0.3 and V >= 64:
            cut = torch.from_numpy(rng.random(V + pad) < rng.random() / 3)
            z[r][cut] = -float("inf")
    z = z.to(dtype)
    ref = ft.draft_features(z.float().numpy()[:, :V].astype(np.float64))
    out = svp.draft_features(z.cuda(), vocab=V).cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref[:, 1:16])
    assert out[:, 0].tolist() == ref[:, 0].tolist()
    assert np.array_equal(np.isfinite(out[:, 1:16]), fin)
    dd = np.abs(np.where(fin, out[:, 1:16], 0.0) - np.where(fin, ref[:, 1:16], 0.0))
    assert np.all(dd <= 6e-8 * np.maximum(np.abs(np.where(fin, ref[:, 1:16], 0.0)), np.abs(ref[:, :1])))
    assert np.abs(out[:, 16] - ref[:, 16]).max() <= 1e-4
    assert np.abs(out[:, 17] - ref[:, 17]).max() <= 1e-4 * max(1.0, np.log(V))


_WIDE_HEADS = [(4, 2), (8, 8), (6, 1), (16, 4), (2, 2), (12, 4)]


@pytest.mark.parametrize("seed", range(6))
def test_random_wide_configs(seed):
    """Candidate blocks wider than 16 (the router's 128-row wide tile): request count, block
    width 17 to 199, slot counts (0 included), context lengths, head dim 64 / 128 / 256,
    query heads per KV head, contiguous or paged context."""
    rng = np.random.default_rng(5000 + seed)
    d = [64, 128, 256][seed % 3]
    hq, hkv = _WIDE_HEADS[seed]
    n = int(rng.integers(1, 5))
    W = int(rng.integers(17, 200))
    lengths = [int(x) for x in rng.integers(0, W + 1, size=n)]
    if sum(lengths) == 0:
        lengths[0] = W
    ctx = [int(x) if rng.random() < 0.8 else 0 for x in rng.integers(1, 2500, size=n)]
    paged = bool(rng.random() < 0.5)
    b = wl.make_batch("paged_n64_bf16" if paged else "budget8n_bf16", seed=seed, n=n, W=W,
                      lengths=lengths, ctx_lengths=ctx, hq=hq, hkv=hkv, d=d, poison=True,
                      with_logits=False)
    out, lse = gpu_verify(to_dev(b), w=W)
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)
    assert torch.isnan(out[b.m_live:].float()).all()


@pytest.mark.parametrize("seed", range(4))
def test_random_fp32_configs(seed):
    """fp32 inputs (the CUDA-core path): random request count, block width up to 40, slot
    counts, context lengths, head dim 64 / 128 / 256, query heads per KV head, contiguous or
    paged context; to the fp32 bar."""
    rng = np.random.default_rng(6000 + seed)
    d = [64, 128, 256, 128][seed]
    hq, hkv = [(4, 2), (8, 1), (3, 3), (12, 4)][seed]
    n = int(rng.integers(1, 6))
    W = int(rng.integers(1, 41))
    lengths = [int(x) for x in rng.integers(0, W + 1, size=n)]
    if sum(lengths) == 0:
        lengths[0] = W
    ctx = [int(x) if rng.random() < 0.8 else 0 for x in rng.integers(1, 1200, size=n)]
    paged = bool(rng.random() < 0.5)
    b = wl.make_batch("paged_n64_bf16" if paged else "budget8n_bf16", seed=seed, n=n, W=W,
                      lengths=lengths, ctx_lengths=ctx, hq=hq, hkv=hkv, d=d, dtype="f32",
                      poison=True, with_logits=False)
    out, lse = gpu_verify(to_dev(b), w=W)
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.float32)
    assert torch.isnan(out[b.m_live:].float()).all()


_PREFILL_HEADS = [(4, 2, 128), (8, 2, 128), (8, 4, 128), (6, 2, 128), (4, 2, 64)]


@pytest.mark.parametrize("seed", range(5))
def test_random_prefill_configs(seed):
    """Causal prefill on random packed sequences: 1 to 8 sequences of 0 to 800 rows (on and off
    the 128-row tile); even query-head groups at d = 128 take the dedicated kernel, an odd
    group or d = 64 the general one."""
    import oracle
    rng = np.random.default_rng(7000 + seed)
    hq, hkv, d = _PREFILL_HEADS[seed]
    n = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.integers(0, 801, size=n)]
    lens[int(rng.integers(n))] = int(rng.choice([1, 128, 256, 513]))
    if seed == 2:
        lens.insert(1, 0)   # an empty sequence between two others
        n += 1
    parts = [wl.make_prefill(seed=100 * seed + i, s=max(L, 1), hq=hq, hkv=hkv, d=d) for i, L in enumerate(lens)]
    q = torch.cat([x[0][:L] for x, L in zip(parts, lens)])
    k = torch.cat([x[1][:L] for x, L in zip(parts, lens)])
    v = torch.cat([x[2][:L] for x, L in zip(parts, lens)])
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    ws = svp.Workspace(svp.prefill_attn_workspace_size(n, max(max(lens), 1), hq, hkv, d))
    out, lse = svp.prefill_attn(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max_s=max(max(lens), 1), ws=ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    ref_o, ref_l = oracle.attention(q, k, v, torch.zeros(n, dtype=torch.int32), cu, hkv=hkv,
                                    scale=d ** -0.5, k_ctx=k[:0], v_ctx=v[:0],
                                    cu_ctx=torch.zeros(n + 1, dtype=torch.int64), threads=16)
    compare_attention(out, lse, ref_o, ref_l, np.arange(int(cu[-1])), torch.bfloat16)
