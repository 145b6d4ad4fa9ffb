"""GPU parity: verification attention (C ABI via the binding) vs the fp64 oracle.

Same seeded inputs on both sides; element-wise comparison on every packed row (small
and medium cases) or on sampled requests (full-size paged and wide-head workloads).
Bars: bf16 max-abs 2e-2 and mean-abs 2e-3, fp32 max-abs 1e-4; lse within 4e-3 (bf16:
twice the bf16 rounding bound of the row sum) or 1e-4 (fp32).
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_packed_gb300 as svp
from speculative_decoding_verification_packed_gb300 import workloads as wl
from helpers import compare_attention, gpu_verify, oracle_verify, rows_of, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lengths", [[4, 12, 8], [10, 8, 6]])
def test_tiny_fp32_packed_and_relayout(lengths):
    b = wl.make_batch("tiny_fp32", seed=0, lengths=lengths, poison=True)
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.float32)


@pytest.mark.parametrize("seed", [0, 1])
def test_small_bf16_ragged_several_tiles(seed):
    # contexts that end mid-tile, an empty context, a single-slot request, k up to 16
    b = wl.make_batch("budget8n_bf16", seed=seed, n=5, lengths=[16, 1, 7, 3, 9],
                      ctx_lengths=[0, 65, 200, 1000, 63], hq=8, hkv=2, d=128, poison=True)
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)
    # packed tail rows are never written
    assert torch.isnan(out[b.m_live:].float()).all()


@pytest.mark.parametrize("d,hq,hkv", [(64, 4, 1), (128, 32, 8), (256, 24, 2)])
def test_head_dims_and_group_sizes(d, hq, hkv):
    b = wl.make_batch("budget8n_bf16", seed=3, n=3, lengths=[7, 16, 2],
                      ctx_lengths=[300, 129, 64], hq=hq, hkv=hkv, d=d, poison=True)
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_full_width_workload():
    b = wl.make_batch("full_width_bf16", seed=0)
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_budget8n_workload():
    b = wl.make_batch("budget8n_bf16", seed=0)
    assert b.m_live == 64
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_peaky_queries_force_rescaling():
    # queries scaled x4: large score spread moves the running maximum many times
    b = wl.make_batch("budget8n_bf16", seed=2, n=3, lengths=[16, 5, 9],
                      ctx_lengths=[2000, 333, 70], hq=8, hkv=2, d=128)
    b.q = (b.q.float() * 4).to(torch.bfloat16)
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_paged_full_size_sampled_requests():
    b = wl.make_batch("paged_n64_bf16", seed=0, device="cuda")
    out, lse = gpu_verify(b)
    bc = to_dev(b, "cpu")
    sample = [0, 17, 40, 63]
    ref_o, ref_l = oracle_verify(bc, requests=sample)
    compare_attention(out, lse, ref_o, ref_l, rows_of(bc, sample), torch.bfloat16)


def test_wide_head_workload_sampled_requests():
    b = wl.make_batch("wide_gqa_bf16", seed=0, with_logits=False)
    out, lse = gpu_verify(to_dev(b))
    sample = [0, 5, 31]
    ref_o, ref_l = oracle_verify(b, requests=sample)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b, sample), torch.bfloat16)


def test_paged_equals_contiguous_on_gpu():
    b = wl.make_batch("paged_n64_bf16", seed=1, n=4, lengths=[16, 3, 1, 9],
                      ctx_lengths=[1000, 17, 0, 4096], poison=True)
    bd = to_dev(b)
    out_p, lse_p = gpu_verify(bd)
    ks, vs, cuc = [], [], [0]
    bt = b.block_table
    for i, L in enumerate(b.ctx_len.tolist()):
        t = torch.arange(L)
        pages = bt[i, t // 16].long()
        ks.append(b.k_cache[pages, :, t % 16])
        vs.append(b.v_cache[pages, :, t % 16])
        cuc.append(cuc[-1] + L)
    bd.paged = False
    bd.k_ctx = torch.cat(ks).cuda()
    bd.v_ctx = torch.cat(vs).cuda()
    bd.cu_ctx = torch.tensor(cuc, dtype=torch.int64, device="cuda")
    out_c, lse_c = gpu_verify(bd)
    rows = rows_of(b)
    assert torch.equal(out_p[rows], out_c[rows])
    assert torch.equal(lse_p[rows], lse_c[rows])


def test_packed_equals_alone_and_relayout_on_gpu():
    b1 = wl.make_batch("full_width_bf16", seed=4, n=3, lengths=[4, 12, 8], ctx_lengths=[700, 64, 2000])
    b2 = wl.make_batch("full_width_bf16", seed=4, n=3, lengths=[10, 8, 6], ctx_lengths=[700, 64, 2000])
    o1, l1 = gpu_verify(to_dev(b1))
    o2, l2 = gpu_verify(to_dev(b2))
    c1, c2 = b1.cu_slots.tolist(), b2.cu_slots.tolist()
    for i, (ka, kb) in enumerate(zip([4, 12, 8], [10, 8, 6])):
        m = min(ka, kb)
        d = (o1[c1[i]:c1[i] + m].float() - o2[c2[i]:c2[i] + m].float()).abs().max().item()
        assert d <= 1e-2, (i, d)
    # request 0 alone at full width, truncated
    b0 = wl.make_batch("full_width_bf16", seed=4, n=3, lengths=[16, 16, 16], ctx_lengths=[700, 64, 2000])
    o0, _ = gpu_verify(to_dev(b0))
    d = (o0[0:4].float() - o1[0:4].float()).abs().max().item()
    assert d <= 1e-2


@pytest.mark.parametrize("mode", [svp.TILE_FIXED128, svp.TILE_SHORT, svp.TILE_WIDE,
                                  svp.TILE_SHORT_UNPACKED])
def test_tile_modes_match_oracle(mode):
    b = wl.make_batch("budget8n_bf16", seed=5, n=4, lengths=[16, 2, 11, 5],
                      ctx_lengths=[513, 64, 1500, 0], hq=8, hkv=2, d=128, poison=True)
    out, lse = gpu_verify(to_dev(b), tile_mode=mode)
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_unpacked_short_tile_at_head_dim_256():
    # the GQA-unpacked contrast at d = 256 (one query head per 32-row tile, 12 heads per KV
    # head), with split pairs and contexts ending mid-tile
    b = wl.make_batch("wide_gqa_bf16", seed=8, n=3, lengths=[7, 3, 7], ctx_lengths=[700, 130, 0],
                      hq=12, hkv=1, d=256, poison=True, with_logits=False)
    out, lse = gpu_verify(to_dev(b), tile_mode=svp.TILE_SHORT_UNPACKED)
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_wide_router_for_long_candidate_blocks():
    # w > 16 routes to the 128-row wide tile (causal over the candidates)
    b = wl.make_batch("budget8n_bf16", seed=6, n=3, W=160, lengths=[150, 17, 40],
                      ctx_lengths=[300, 0, 1111], hq=4, hkv=2, d=128, poison=True)
    out, lse = gpu_verify(to_dev(b), w=160)
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_prefill_small():
    q, k, v = wl.make_prefill(seed=0, s=700, hq=4, hkv=2, d=128)
    cu = torch.tensor([0, 700], dtype=torch.int32)
    out, lse = svp.prefill_attn(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max_s=700)
    torch.cuda.synchronize()
    import oracle
    ref_o, ref_l = oracle.attention(q, k, v, torch.zeros(1, dtype=torch.int32), cu, hkv=2,
                                    scale=128 ** -0.5, k_ctx=k[:0], v_ctx=v[:0],
                                    cu_ctx=torch.zeros(2, dtype=torch.int64), threads=16)
    compare_attention(out, lse, ref_o, ref_l, np.arange(700), torch.bfloat16)


def test_prefill_4096_sampled_heads():
    q, k, v = wl.make_prefill(seed=0)
    cu = torch.tensor([0, 4096], dtype=torch.int32)
    out, lse = svp.prefill_attn(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max_s=4096)
    torch.cuda.synchronize()
    import oracle
    for h in (0, 13, 31):
        g = h // 4
        ref_o, ref_l = oracle.attention(q[:, h:h + 1].contiguous(), k[:, g:g + 1].contiguous(),
                                        v[:, g:g + 1].contiguous(), torch.zeros(1, dtype=torch.int32),
                                        cu, hkv=1, scale=128 ** -0.5, k_ctx=k[:0, :1], v_ctx=v[:0, :1],
                                        cu_ctx=torch.zeros(2, dtype=torch.int64), threads=16)
        compare_attention(out[:, h:h + 1], lse[:, h:h + 1], ref_o, ref_l, np.arange(4096),
                          torch.bfloat16)


def test_prefill_scores_jumping_between_tiles():
    # Every query leans on the all-ones direction and the keys are shifted along it by 0, 3
    # and 6 every two 128-key tiles, so rows that see tile 2 or tile 4 meet scores about 50
    # (in log2 units) above everything before: the exponent reference must move in the middle
    # of the row, with O and the row sum rescaled.  Exact softmax in the oracle.
    s = 700
    q, k, v = wl.make_prefill(seed=4, s=s, hq=4, hkv=2, d=128)
    shift = torch.tensor([0.0, 0.0, 3.0, 3.0, 6.0, 6.0]).repeat_interleave(128)[:s]
    q = (q.float() + 1.0).to(torch.bfloat16)
    k = (k.float() + shift[:, None, None]).to(torch.bfloat16)
    cu = torch.tensor([0, s], dtype=torch.int32)
    out, lse = svp.prefill_attn(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max_s=s)
    torch.cuda.synchronize()
    import oracle
    ref_o, ref_l = oracle.attention(q, k, v, torch.zeros(1, dtype=torch.int32), cu, hkv=2,
                                    scale=128 ** -0.5, k_ctx=k[:0], v_ctx=v[:0],
                                    cu_ctx=torch.zeros(2, dtype=torch.int64), threads=16)
    compare_attention(out, lse, ref_o, ref_l, np.arange(s), torch.bfloat16)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 2)])
def test_prefill_varlen_sequences(hq, hkv):
    # several packed sequences, lengths off the 128-row tile (one shorter than a tile, one
    # exactly a tile); G = 4 takes the dedicated kernel, G = 3 (odd) the general one
    lens = [300, 128, 77, 1000]
    parts = [wl.make_prefill(seed=20 + i, s=L, hq=hq, hkv=hkv, d=128) for i, L in enumerate(lens)]
    q = torch.cat([x[0] for x in parts])
    k = torch.cat([x[1] for x in parts])
    v = torch.cat([x[2] for x in parts])
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    out, lse = svp.prefill_attn(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max_s=max(lens))
    torch.cuda.synchronize()
    import oracle
    n = len(lens)
    ref_o, ref_l = oracle.attention(q, k, v, torch.zeros(n, dtype=torch.int32), cu, hkv=hkv,
                                    scale=128 ** -0.5, k_ctx=k[:0], v_ctx=v[:0],
                                    cu_ctx=torch.zeros(n + 1, dtype=torch.int64), threads=16)
    compare_attention(out, lse, ref_o, ref_l, np.arange(int(cu[-1])), torch.bfloat16)


def test_inactive_requests_and_empty_batch():
    b = wl.make_batch("budget8n_bf16", seed=7, n=4, lengths=[3, 0, 5, 0],
                      ctx_lengths=[100, 50, 0, 10], hq=8, hkv=2, d=128, poison=True)
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_bad_metadata_sets_status_and_gpu_stays_healthy():
    b = wl.make_batch("budget8n_bf16", seed=8, n=3, lengths=[4, 4, 4],
                      ctx_lengths=[100, 100, 100], hq=8, hkv=2, d=128)
    bd = to_dev(b)
    bd.cu_slots = torch.tensor([0, 4, 2, 12], dtype=torch.int32, device="cuda")  # decreasing
    n = 3
    ws = svp.Workspace(svp.verify_attn_workspace_size(n, b.m_cap, 16, 8, 2, 128))
    svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots, w=16, ws=ws,
                           k_ctx=bd.k_ctx, v_ctx=bd.v_ctx, cu_ctx=bd.cu_ctx)
    st = ws.read_status()
    assert st & svp.DEV_BAD_SLOTS
    bd.cu_slots = b.cu_slots.cuda()
    bd.ctx_len = torch.tensor([100, 100, 10 ** 6], dtype=torch.int32, device="cuda")  # too long
    svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots, w=16, ws=ws,
                           k_ctx=bd.k_ctx, v_ctx=bd.v_ctx, cu_ctx=bd.cu_ctx)
    assert ws.read_status() & svp.DEV_BAD_CONTEXT
    # still healthy: a valid call afterwards matches the oracle
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)
    assert ws.read_status() == 0


@pytest.mark.parametrize("ctx", [[5000, 3000, 8000, 700], [10, 70, 0, 3]])
def test_repeated_calls_are_deterministic_and_leave_tickets_zero(ctx):
    # the second case has fewer KV tiles than SMs, so some CTAs get no work
    b = wl.make_batch("full_width_bf16", seed=9, n=4, ctx_lengths=ctx)
    bd = to_dev(b)
    ws = svp.Workspace(svp.verify_attn_workspace_size(4, b.m_cap, 16, 32, 8, 128))
    kw = dict(k_ctx=bd.k_ctx, v_ctx=bd.v_ctx, cu_ctx=bd.cu_ctx, w=16, ws=ws)
    o1, l1 = svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots, **kw)
    o2, l2 = svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    pairs = 4 * 8   # requests x KV heads (one row block): tickets are the last words
    tickets = ws.buf[-1024:].view(torch.int32)
    assert int(tickets.abs().sum()) == 0
    assert ws.read_status() == 0
    ref_o, ref_l = oracle_verify(b)
    compare_attention(o1, l1, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_workspace_reuse_across_sizes_and_mismatch_flag():
    # one workspace serves calls with different n; a different head_dim is refused
    big = wl.make_batch("budget8n_bf16", seed=11, n=6, lengths=[16, 3, 9, 1, 12, 7],
                        ctx_lengths=[900, 20, 3000, 5, 130, 64], hq=8, hkv=2, d=128)
    small = wl.make_batch("budget8n_bf16", seed=12, n=2, lengths=[5, 16],
                          ctx_lengths=[70, 400], hq=8, hkv=2, d=128)
    ws = svp.Workspace(max(svp.verify_attn_workspace_size(6, big.m_cap, 16, 8, 2, 128),
                           svp.verify_attn_workspace_size(6, big.m_cap, 16, 8, 2, 256)))
    for b in (small, big, small):
        bd = to_dev(b)
        o, l = svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots, w=16,
                                      ws=ws, k_ctx=bd.k_ctx, v_ctx=bd.v_ctx, cu_ctx=bd.cu_ctx)
        torch.cuda.synchronize()
        assert ws.read_status() == 0
        ref_o, ref_l = oracle_verify(b)
        compare_attention(o, l, ref_o, ref_l, rows_of(b), torch.bfloat16)
    other = wl.make_batch("budget8n_bf16", seed=13, n=2, lengths=[5, 16],
                          ctx_lengths=[70, 400], hq=8, hkv=2, d=256)
    bd = to_dev(other)
    svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots, w=16, ws=ws,
                           k_ctx=bd.k_ctx, v_ctx=bd.v_ctx, cu_ctx=bd.cu_ctx)
    assert ws.read_status() & svp.DEV_WORKSPACE


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("d,hq,k", [(128, 4, 9), (256, 12, 7)])
def test_one_long_pair_split_over_many_ctas(paged, d, hq, k):
    # a single (request, KV head) pair of ~40 KV tiles is cut into ~40 pieces, so the
    # last-arrival merge runs several passes (eight pieces each at d = 128; at d = 256 three
    # slabs of one 128-column block fit the staging ring, so each block takes many passes)
    b = wl.make_batch("paged_n64_bf16" if paged else "budget8n_bf16", seed=14, n=1,
                      lengths=[k], ctx_lengths=[5000], hq=hq, hkv=1, d=d, poison=True)
    out, lse = gpu_verify(to_dev(b))
    ref_o, ref_l = oracle_verify(b)
    compare_attention(out, lse, ref_o, ref_l, rows_of(b), torch.bfloat16)


def test_lse_is_optional():
    """lse may be NULL: the outputs are bit-identical to a run that writes it, for the
    verification kernel with pairs split over several CTAs (the merge reads the pieces'
    statistics from the workspace, not from lse) and for the dedicated prefill kernel."""
    b = wl.make_batch("budget8n_bf16", seed=21, n=4, lengths=[16, 3, 9, 1],
                      ctx_lengths=[3000, 700, 0, 5000], hq=8, hkv=2, d=128, poison=True)
    bd = to_dev(b)
    out1, lse1 = gpu_verify(bd)
    ws = svp.Workspace(svp.verify_attn_workspace_size(bd.n, bd.m_cap, bd.W, bd.hq, bd.hkv, bd.d,
                                                      bd.q.dtype, svp.TILE_AUTO))
    out2, lse2 = svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots, w=bd.W,
                                        k_ctx=bd.k_ctx, v_ctx=bd.v_ctx, cu_ctx=bd.cu_ctx,
                                        want_lse=False, ws=ws)
    torch.cuda.synchronize()
    assert lse2 is None and ws.read_status() == 0
    assert torch.equal(out1[:b.m_live], out2[:b.m_live])
    q, k, v = wl.make_prefill(seed=3, s=500, hq=4, hkv=2, d=128)
    cu = torch.tensor([0, 500], dtype=torch.int32).cuda()
    p1, l1 = svp.prefill_attn(q.cuda(), k.cuda(), v.cuda(), cu, max_s=500)
    p2, l2 = svp.prefill_attn(q.cuda(), k.cuda(), v.cuda(), cu, max_s=500, want_lse=False)
    torch.cuda.synchronize()
    assert l2 is None and torch.equal(p1, p2)
