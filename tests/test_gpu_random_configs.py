"""GPU parity on seeded random configurations: verification attention and fused margin +
accept against the fp64 oracle.

Each case draws its shape at random (fixed seeds, so every run checks the same cases): the
number of requests, their slot counts (0 = inactive, up to 16) and context lengths (0 to
a few thousand, ending anywhere within a 128-key tile or a 16-token page), the head dim
(128 or 256), the query heads per KV head (1 to 12), contiguous or paged context, and the
tile mode.  Packed tail rows are poisoned with NaN and must stay unread and unwritten.
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
