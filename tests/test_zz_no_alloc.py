"""The allocation-free margin + accept entry point (svp_margin_accept_noalloc).

Some callers cannot allocate device memory (a host framework that owns every device
allocation, or a path where cudaMalloc is not allowed); this entry point keeps its scratch
in a fixed array inside the library.  The tests call it through the C ABI: twice in a row,
checking every output against svp_margin_accept (with its own workspace) and against the
oracle, bit for bit as in the other margin/accept tests; and on a non-blocking stream,
which may be the process's first call (the one that clears the array).  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_packed_gb300 as svp
from speculative_decoding_verification_packed_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    L = svp.lib()
    fn = L.svp_margin_accept_noalloc
    vp = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int, vp, vp,
                   ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp]
    return fn


def _outs(m_cap, n):
    return (torch.full((m_cap,), -7, dtype=torch.int32, device="cuda"),
            torch.full((m_cap,), float("nan"), device="cuda"),
            torch.full((m_cap,), float("nan"), device="cuda"),
            torch.full((m_cap,), float("nan"), device="cuda"),
            torch.full((n,), -7, dtype=torch.int32, device="cuda"),
            torch.full((n,), -7, dtype=torch.int32, device="cuda"))


def _call_noalloc(fn, logits, tokens, cu, outs, stream=None):
    m_cap, vocab = logits.shape
    n = cu.shape[0] - 1
    code = svp.SVP_BF16 if logits.dtype == torch.bfloat16 else svp.SVP_F32
    s = torch.cuda.current_stream() if stream is None else stream
    return fn(logits.data_ptr(), vocab, m_cap, vocab, code, tokens.data_ptr(), cu.data_ptr(), n,
              outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), outs[3].data_ptr(),
              outs[4].data_ptr(), outs[5].data_ptr(), s.cuda_stream)


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.int32)


def _check_oracle(b, outs):
    """Live rows bit-exact against the oracle's row scan; accept / next token exact."""
    live = int(b.cu_slots[-1])
    logits = b.target_logits[:live]
    r_idx, r_t1, r_t2, r_mg = oracle.row_top2(logits)
    idx, t1, t2, mg = (o[:live].cpu().numpy() for o in outs[:4])
    assert np.array_equal(idx, r_idx)
    assert np.array_equal(_bits(t1), _bits(r_t1))
    assert np.array_equal(_bits(t2), _bits(r_t2))
    assert (((_bits(mg) == _bits(r_mg)) | (np.isnan(mg) & np.isnan(r_mg)))).all()
    am = np.concatenate([r_idx, np.zeros(b.m_cap - live, np.int32)])
    acc, nxt = oracle.greedy_accept(am, b.tokens, b.cu_slots)
    assert np.array_equal(outs[4].cpu().numpy(), acc)
    assert np.array_equal(outs[5].cpu().numpy(), nxt)


def _case(case):
    if case == "tiny_fp32":
        return wl.make_batch("tiny_fp32", seed=3, poison=True)
    return wl.make_batch("wide_gqa_bf16", seed=5, n=12, hq=1, hkv=1, d=64,
                         ctx_lengths=[0] * 12, lengths=[7, 1, 3, 7, 7, 2, 7, 0, 5, 7, 7, 4],
                         m_cap=64)


def test_noalloc_on_a_side_stream_matches_oracle():
    # Callers with their own streams: when this is the process's first call, the clear of
    # the fixed scratch must be complete before the kernel runs on this non-blocking stream.
    b = _case("wide_vocab_bf16")
    fn = _noalloc_fn()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        logits = b.target_logits.cuda()
        tokens = b.tokens.cuda()
        cu = b.cu_slots.cuda()
        m_cap, n = logits.shape[0], cu.shape[0] - 1
        outs = _outs(m_cap, n)
        assert _call_noalloc(fn, logits, tokens, cu, outs, stream=side) == svp.SVP_OK
    side.synchronize()
    _check_oracle(b, outs)


def _same(a, b):
    for x, y in zip(a, b):
        x, y = x.cpu(), y.cpu()
        if x.dtype == torch.float32:
            xb, yb = x.view(torch.int32), y.view(torch.int32)
            both_nan = torch.isnan(x) & torch.isnan(y)
            assert bool(((xb == yb) | both_nan).all())
        else:
            assert torch.equal(x, y)


@pytest.mark.parametrize("case", ["tiny_fp32", "wide_vocab_bf16"])
def test_noalloc_matches_workspace_entry_point_twice(case):
    b = _case(case)
    logits = b.target_logits.cuda()
    tokens = b.tokens.cuda()
    cu = b.cu_slots.cuda()
    m_cap, n = logits.shape[0], cu.shape[0] - 1
    ref = svp.margin_accept(logits, tokens, cu, outs=_outs(m_cap, n))
    fn = _noalloc_fn()
    for _ in range(2):                      # two calls in a row share the fixed scratch
        outs = _outs(m_cap, n)
        assert _call_noalloc(fn, logits, tokens, cu, outs) == svp.SVP_OK
        torch.cuda.synchronize()
        _same(outs, ref)
        _check_oracle(b, outs)
    live = int(b.cu_slots[-1])
    assert (outs[0][live:].cpu() == -7).all()          # rows past cu_slots[n] untouched


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _noalloc_fn()
    rows, vocab, n = 65536, 262144, 64
    # the sizes must need more than the fixed 2 MiB of scratch, checked through the
    # workspace query first, so the call below is refused on the host and never enqueues
    # anything; the buffers are real but far too small for these sizes
    need = svp.margin_accept_workspace_size(n, rows, vocab)
    assert need > (2 << 20) * 4
    small_i = torch.zeros(64, dtype=torch.int32, device="cuda")
    small_f = torch.zeros(64, dtype=torch.float32, device="cuda")
    logits = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()
    rc = fn(p(logits), vocab, rows, vocab, svp.SVP_BF16, p(small_i), p(small_i), n, p(small_i),
            p(small_f), p(small_f), p(small_f), p(small_i), p(small_i), None)
    assert rc == svp.SVP_EWORKSPACE
