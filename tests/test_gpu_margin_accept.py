"""GPU parity: row top-1/top-2/margin and greedy acceptance vs the oracle (bit-exact).

Accept lengths, next tokens and argmax indices must match exactly; top-1/top-2 values
and the fp32 margin are compared bit for bit (same input values, same fp32 subtraction).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_packed_gb300 as svp
from speculative_decoding_verification_packed_gb300 import workloads as wl
from helpers import check_margin_rows

pytestmark = pytest.mark.gpu


_check_rows = check_margin_rows


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("vocab", [2, 7, 512, 40000, 248320])
def test_draft_margin_random_rows(dtype, vocab):
    g = torch.Generator().manual_seed(vocab)
    x = (torch.randn(37, vocab, generator=g) * 2).to(dtype)
    x[1, :] = 3.0                                  # all equal: idx 0, margin 0
    x[2, vocab - 1] = 100.0                        # max at the last index
    x[3, 0] = 100.0; x[3, vocab - 1] = 100.0      # tie at both ends
    x[4, :] = float("-inf"); x[4, vocab // 2] = -5.0
    x[5, :] = float("-inf")                        # all -inf: margin NaN
    outs = svp.draft_margin(x.cuda())
    torch.cuda.synchronize()
    _check_rows(x, outs)


def test_draft_margin_strided_and_unaligned_rows():
    import ctypes
    g = torch.Generator().manual_seed(1)
    base = torch.randn(20, 1003, generator=g).to(torch.bfloat16)
    dev = base.cuda()
    n_rows, vocab = 20, 1000
    outs = [torch.empty(n_rows, dtype=torch.int32, device="cuda")] + \
           [torch.empty(n_rows, dtype=torch.float32, device="cuda") for _ in range(3)]
    ws = svp.Workspace(svp.draft_margin_workspace_size(n_rows, vocab))
    # rows start 2 bytes past a 16-byte boundary, row stride 1003 > vocab
    st = svp.lib().svp_draft_margin(ctypes.c_void_p(dev.data_ptr() + 2), 1003, n_rows, vocab,
                                    svp.SVP_BF16, outs[0].data_ptr(), outs[1].data_ptr(),
                                    outs[2].data_ptr(), outs[3].data_ptr(), ws.ptr, ws.nbytes,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == svp.SVP_OK
    torch.cuda.synchronize()
    _check_rows(base[:, 1:1001].contiguous(), outs)
    # aligned rows with padding beyond the vocabulary
    padded = torch.zeros(20, 1008, dtype=torch.bfloat16)
    padded[:, :1000] = base[:, :1000]
    padded[:, 1000:] = 1000.0                      # must be ignored
    outs = svp.draft_margin(padded.cuda(), vocab=1000)
    torch.cuda.synchronize()
    _check_rows(base[:, :1000].contiguous(), outs)


def test_margin_accept_tiny_fp32():
    b = wl.make_batch("tiny_fp32", seed=0, poison=True)
    outs = svp.margin_accept(b.target_logits.cuda(), b.tokens.cuda(), b.cu_slots.cuda())
    torch.cuda.synchronize()
    rows = np.arange(b.m_live)
    r_idx = _check_rows(b.target_logits[:b.m_live], [o[:b.m_live] for o in outs[:4]])
    acc, nxt = oracle.greedy_accept(np.concatenate([r_idx, np.zeros(b.m_cap - b.m_live, np.int32)]),
                                    b.tokens, b.cu_slots)
    assert np.array_equal(outs[4].cpu().numpy(), acc)
    assert np.array_equal(outs[5].cpu().numpy(), nxt)


def test_margin_accept_wide_vocab_workload():
    b = wl.make_batch("wide_gqa_bf16", seed=0, hq=2, hkv=1, d=64, ctx_lengths=[0] * 32)
    outs = svp.margin_accept(b.target_logits.cuda(), b.tokens.cuda(), b.cu_slots.cuda())
    torch.cuda.synchronize()
    r_idx = _check_rows(b.target_logits, outs)
    acc, nxt = oracle.greedy_accept(r_idx, b.tokens, b.cu_slots)
    assert np.array_equal(outs[4].cpu().numpy(), acc)
    assert np.array_equal(outs[5].cpu().numpy(), nxt)
    assert (outs[4].cpu().numpy() <= 7).all() and (outs[4].cpu().numpy() >= 1).all()
    # draft-side margins over the draft logits
    d = svp.draft_margin(b.draft_logits.cuda())
    torch.cuda.synchronize()
    _check_rows(b.draft_logits, d)


def test_full_vocab_planted_ties_across_chunks():
    # The launch the bench times (224 rows x 248,320 bf16): each row is cut into chunks
    # scanned by different warps and CTAs, and the row's maximum is planted twice or three
    # times in different chunks (or both ends of the row), so the lowest-index rule must
    # survive the cross-warp, cross-CTA merge of the chunk partials.
    V, rows = 248320, 224
    g = torch.Generator().manual_seed(17)
    x = (torch.randn(rows, V, generator=g) * 2).clamp(-12.0, 12.0).to(torch.bfloat16)
    pos = torch.randint(0, V, (rows, 3), generator=g)
    planted = []
    for r in range(rows):
        ks = 2 if r % 3 else 3
        ids = sorted(set(int(v) for v in pos[r, :ks]))
        if r % 7 == 0:
            ids = [0, V - 1]                                  # both ends of the row
        x[r, ids] = 16.0
        planted.append(min(ids))
    outs = svp.draft_margin(x.cuda())
    torch.cuda.synchronize()
    r_idx = _check_rows(x, outs)
    assert r_idx.tolist() == planted
    assert (outs[3].cpu() == 0).all()                         # tied maximum: margin 0
    # the fused kernel on the same rows: 32 requests of 7 slots, tokens = planted argmaxes
    cu = torch.arange(0, rows + 1, 7, dtype=torch.int32)
    tokens = torch.full((rows,), -1, dtype=torch.int32)
    for i in range(32):
        for j in range(1, 7):
            tokens[7 * i + j] = planted[7 * i + j - 1] if j <= (i % 7) else (planted[7 * i + j - 1] + 1) % V
    fo = svp.margin_accept(x.cuda(), tokens.cuda(), cu.cuda())
    torch.cuda.synchronize()
    _check_rows(x, fo)
    acc, nxt = oracle.greedy_accept(r_idx, tokens, cu)
    assert np.array_equal(fo[4].cpu().numpy(), acc)
    assert np.array_equal(fo[5].cpu().numpy(), nxt)
    assert fo[4].cpu().tolist() == [1 + min(i % 7, 6) for i in range(32)]


def test_margin_accept_budget_rows_up_to_sixteen():
    # bf16 rows of requests with up to 16 slots (budget 8N lengths: the finishing warp merges
    # a request's rows eight at a time), drafts planted to match the row argmax up to a
    # chosen point: full acceptance of 16, a first-draft miss, and everything in between
    V, n = 32000, 8
    g = torch.Generator().manual_seed(21)
    lengths = [16, 1, 9, 16, 8, 2, 5, 7]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    m_cap = int(cu[-1]) + 3
    logits = (torch.randn(m_cap, V, generator=g) * 2).to(torch.bfloat16)
    amax = logits.float().argmax(-1).to(torch.int32)
    tokens = torch.randint(0, V, (m_cap,), generator=g, dtype=torch.int32)
    stop = [16, 0, 4, 11, 8, 1, 0, 3]          # drafts that match before the first miss
    for i in range(n):
        off, k = int(cu[i]), lengths[i]
        for j in range(1, k):
            tokens[off + j] = amax[off + j - 1] if j <= stop[i] else (amax[off + j - 1] + 1) % V
    outs = svp.margin_accept(logits.cuda(), tokens.cuda(), cu.cuda())
    torch.cuda.synchronize()
    live = int(cu[-1])
    r_idx = _check_rows(logits[:live], [o[:live] for o in outs[:4]])
    acc, nxt = oracle.greedy_accept(np.concatenate([r_idx, np.zeros(m_cap - live, np.int32)]),
                                    tokens, cu)
    assert np.array_equal(outs[4].cpu().numpy(), acc)
    assert np.array_equal(outs[5].cpu().numpy(), nxt)
    assert acc.tolist() == [1 + min(stop[i], lengths[i] - 1) for i in range(n)]


def test_margin_accept_inactive_and_tail_not_read():
    V = 1000
    g = torch.Generator().manual_seed(3)
    cu = torch.tensor([0, 3, 3, 8, 8], dtype=torch.int32)      # requests 1 and 3 inactive
    m_cap = 12
    logits = torch.randn(m_cap, V, generator=g)
    logits[8:] = float("nan")                                   # tail: must not be read
    argmax = logits[:8].argmax(-1).to(torch.int32)
    tokens = torch.randint(0, V, (m_cap,), generator=g, dtype=torch.int32)
    tokens[1] = argmax[0]; tokens[2] = argmax[1]               # request 0: full accept
    tokens[4] = argmax[3]                                       # request 2: accept 1 draft
    outs = svp.margin_accept(logits.cuda(), tokens.cuda(), cu.cuda())
    torch.cuda.synchronize()
    r_idx = _check_rows(logits[:8], [o[:8] for o in outs[:4]])
    acc, nxt = oracle.greedy_accept(np.concatenate([r_idx, np.zeros(4, np.int32)]), tokens, cu)
    assert outs[4].cpu().tolist() == acc.tolist() == [3, 0, 2, 0]
    assert outs[5].cpu().tolist() == nxt.tolist()
    assert outs[5].cpu().tolist()[1] == -1
    assert (outs[0][8:].cpu() == -1).all()                      # tail rows untouched


def test_greedy_accept_all_patterns():
    rng = np.random.default_rng(0)
    k = 8
    import itertools
    pats = list(itertools.product([False, True], repeat=k - 1))
    n = len(pats)
    cu = (np.arange(n + 1) * k).astype(np.int32)
    argmax = rng.integers(0, 1000, size=n * k).astype(np.int32)
    tokens = rng.integers(0, 1000, size=n * k).astype(np.int32)
    for i, p in enumerate(pats):
        for j in range(1, k):
            tgt = argmax[i * k + j - 1]
            tokens[i * k + j] = tgt if p[j - 1] else (tgt + 1) % 1000
    acc, nxt = svp.greedy_accept(torch.from_numpy(argmax).cuda(), torch.from_numpy(tokens).cuda(),
                                 torch.from_numpy(cu).cuda())
    r_acc, r_nxt = oracle.greedy_accept(argmax, tokens, cu)
    assert np.array_equal(acc.cpu().numpy(), r_acc)
    assert np.array_equal(nxt.cpu().numpy(), r_nxt)


def test_repeated_margin_calls_reuse_workspace():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(50, 30000, generator=g).to(torch.bfloat16).cuda()
    a = svp.draft_margin(x)
    b = svp.draft_margin(x)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_margin_workspace_returns_to_zero_and_serves_any_size():
    ws = svp.Workspace(svp.margin_accept_workspace_size(40, 300, 5000))
    g = torch.Generator().manual_seed(9)
    for m_cap, n in ((300, 40), (20, 3), (300, 40)):
        lengths = torch.randint(0, 8, (n,), generator=g)
        cu = torch.zeros(n + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lengths, 0)
        cu = cu.clamp(max=m_cap)
        logits = torch.randn(m_cap, 5000, generator=g)
        tokens = torch.randint(0, 5000, (m_cap,), generator=g, dtype=torch.int32)
        outs = svp.margin_accept(logits.cuda(), tokens.cuda(), cu.cuda(), ws=ws)
        torch.cuda.synchronize()
        live = int(cu[-1])
        r_idx = _check_rows(logits[:live], [o[:live] for o in outs[:4]])
        acc, nxt = oracle.greedy_accept(np.concatenate([r_idx, np.zeros(m_cap - live, np.int32)]),
                                        tokens, cu)
        assert np.array_equal(outs[4].cpu().numpy(), acc)
        assert np.array_equal(outs[5].cpu().numpy(), nxt)
        assert ws.read_status() == 0
        assert int(ws.buf[256:].to(torch.int32).sum()) == 0


def test_null_outputs_through_the_abi():
    """Any output pointer of svp_draft_margin / svp_margin_accept may be NULL (called
    through the C ABI directly; the binding always passes all of them): the outputs that are
    given equal those of a call that writes everything, and the NULL ones are skipped."""
    import ctypes
    L = svp.lib()
    g = torch.Generator().manual_seed(17)
    rows, V = 40, 32000
    z = (torch.randn(rows, V, generator=g) * 2).to(torch.bfloat16).cuda()
    full = svp.draft_margin(z)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream().cuda_stream
    ws = svp.Workspace(svp.draft_margin_workspace_size(rows, V))
    for keep in range(4):
        outs = [torch.full((rows,), -5, dtype=torch.int32 if i == 0 else torch.float32, device="cuda")
                for i in range(4)]
        ptrs = [outs[i].data_ptr() if i == keep else None for i in range(4)]
        rc = L.svp_draft_margin(z.data_ptr(), V, rows, V, svp.SVP_BF16, *ptrs, ws.ptr, ws.nbytes, st)
        assert rc == svp.SVP_OK
        torch.cuda.synchronize()
        assert torch.equal(outs[keep], full[keep])
    # fused: only the per-request results
    n = 5
    cu = torch.tensor([0, 8, 8, 15, 31, 40], dtype=torch.int32).cuda()
    tok = torch.randint(0, V, (rows,), generator=g, dtype=torch.int32).cuda()
    ref = svp.margin_accept(z, tok, cu)
    torch.cuda.synchronize()
    acc = torch.full((n,), -5, dtype=torch.int32, device="cuda")
    nxt = torch.full((n,), -5, dtype=torch.int32, device="cuda")
    wsa = svp.Workspace(svp.margin_accept_workspace_size(n, rows, V))
    rc = L.svp_margin_accept(z.data_ptr(), V, rows, V, svp.SVP_BF16, tok.data_ptr(), cu.data_ptr(), n,
                             None, None, None, None, acc.data_ptr(), nxt.data_ptr(), wsa.ptr, wsa.nbytes, st)
    assert rc == svp.SVP_OK
    torch.cuda.synchronize()
    assert torch.equal(acc, ref[4]) and torch.equal(nxt, ref[5])
