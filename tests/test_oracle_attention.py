"""Pins for the oracle's packed verification attention (CPU only).

The oracle (oracle/svp_oracle.c) is checked against things other than itself:
library routines on special cases (torch SDPA / logsumexp in float64), closed forms,
and the layout invariants the pages state (DScale, SII-C Fig. 1 relayout; SIII-C
Flat-buffer packer; SIII-D request-local causal masking).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from speculative_decoding_verification_packed_gb300 import workloads as wl


def _rand(shape, gen, scale=1.0):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * scale


def _tiny(seed=0, n=3, hq=4, hkv=2, d=8, lengths=(2, 3, 1), ctx=(3, 0, 5), qscale=1.0):
    g = torch.Generator().manual_seed(seed)
    lengths = list(lengths)
    cu = wl.prefix_offsets(lengths)
    m = int(cu[-1])
    q = _rand((m, hq, d), g, qscale)
    kn = _rand((m, hkv, d), g)
    vn = _rand((m, hkv, d), g)
    cu_ctx = [0]
    for L in ctx:
        cu_ctx.append(cu_ctx[-1] + L)
    kc = _rand((cu_ctx[-1], hkv, d), g)
    vc = _rand((cu_ctx[-1], hkv, d), g)
    return dict(q=q, k_new=kn, v_new=vn, k_ctx=kc, v_ctx=vc,
                cu_ctx=torch.tensor(cu_ctx, dtype=torch.int64),
                ctx_len=torch.tensor(list(ctx), dtype=torch.int32),
                cu_slots=cu, hkv=hkv, scale=1.0 / math.sqrt(d))


def _run(orc, t, **kw):
    return orc.attention(t["q"], t["k_new"], t["v_new"], t["ctx_len"], t["cu_slots"],
                         hkv=t["hkv"], scale=kw.pop("scale", t["scale"]), k_ctx=t["k_ctx"],
                         v_ctx=t["v_ctx"], cu_ctx=t["cu_ctx"], **kw)


def _sdpa_reference(t):
    """Per request: float64 SDPA with an explicit boolean mask (library routine)."""
    q, kn, vn = t["q"].double(), t["k_new"].double(), t["v_new"].double()
    kc, vc = t["k_ctx"].double(), t["v_ctx"].double()
    cu, cuc, L = t["cu_slots"].tolist(), t["cu_ctx"].tolist(), t["ctx_len"].tolist()
    hq, hkv = q.shape[1], kn.shape[1]
    G = hq // hkv
    out = torch.full(q.shape, float("nan"), dtype=torch.float64)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float64)
    for i in range(len(L)):
        k = cu[i + 1] - cu[i]
        if k == 0:
            continue
        keys = torch.cat([kc[cuc[i]:cuc[i + 1]], kn[cu[i]:cu[i + 1]]], 0)  # [L+k, hkv, d]
        vals = torch.cat([vc[cuc[i]:cuc[i + 1]], vn[cu[i]:cu[i + 1]]], 0)
        keys = keys.repeat_interleave(G, dim=1).transpose(0, 1)  # [hq, L+k, d]
        vals = vals.repeat_interleave(G, dim=1).transpose(0, 1)
        qq = q[cu[i]:cu[i + 1]].transpose(0, 1)                   # [hq, k, d]
        nk = L[i] + k
        mask = torch.zeros(k, nk, dtype=torch.bool)
        mask[:, :L[i]] = True
        mask[:, L[i]:] = torch.tril(torch.ones(k, k, dtype=torch.bool))
        o = F.scaled_dot_product_attention(qq, keys, vals, attn_mask=mask, scale=t["scale"])
        s = (qq @ keys.transpose(-1, -2)) * t["scale"]
        s = s.masked_fill(~mask, float("-inf"))
        out[cu[i]:cu[i + 1]] = o.transpose(0, 1)
        lse[cu[i]:cu[i + 1]] = torch.logsumexp(s, -1).transpose(0, 1)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_library_sdpa_with_mask(orc, seed):
    t = _tiny(seed=seed, lengths=(2, 3, 1, 4), ctx=(3, 0, 5, 2), n=4)
    out, lse = _run(orc, t)
    ref_o, ref_l = _sdpa_reference(t)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_visible_values(orc):
    t = _tiny(seed=3)
    t["q"] = torch.zeros_like(t["q"])
    out, lse = _run(orc, t)
    cu, cuc, L = t["cu_slots"].tolist(), t["cu_ctx"].tolist(), t["ctx_len"].tolist()
    G = t["q"].shape[1] // t["hkv"]
    for i in range(len(L)):
        for j in range(cu[i + 1] - cu[i]):
            for h in range(t["q"].shape[1]):
                vis = torch.cat([t["v_ctx"][cuc[i]:cuc[i + 1], h // G],
                                 t["v_new"][cu[i]:cu[i] + j + 1, h // G]], 0).double()
                np.testing.assert_allclose(out[cu[i] + j, h], vis.mean(0).numpy(), atol=1e-13)
                assert abs(lse[cu[i] + j, h] - math.log(L[i] + j + 1)) < 1e-13


def test_constant_values_per_kv_head_pin_gqa_grouping(orc):
    # every value row of KV head g equals c_g -> each query head h returns c_{h // G}
    t = _tiny(seed=4, hq=6, hkv=3)
    c = torch.arange(3 * 8, dtype=torch.float32).reshape(3, 8) * 0.25 - 1.0
    t["v_ctx"] = c.expand_as(t["v_ctx"]).contiguous()
    t["v_new"] = c.expand_as(t["v_new"]).contiguous()
    out, _ = _run(orc, t)
    for h in range(6):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(c[h // 2].double().numpy(),
                                                              out[:, h].shape), rtol=0, atol=1e-14)


def test_single_dominant_key(orc):
    # score margin >= 50 -> the output is that key's value row (to fp64 rounding)
    t = _tiny(seed=5, lengths=(3,), ctx=(6,), n=1, hq=2, hkv=1)
    d = 8
    t["k_ctx"] = torch.zeros_like(t["k_ctx"])
    t["k_new"] = torch.zeros_like(t["k_new"])
    t["k_ctx"][4, 0, 0] = 1.0
    t["q"] = torch.zeros_like(t["q"])
    t["q"][:, :, 0] = 200.0 * math.sqrt(d)   # score of context key 4 = 200, others 0
    out, _ = _run(orc, t)
    for j in range(3):
        for h in range(2):
            np.testing.assert_allclose(out[j, h], t["v_ctx"][4, 0].double().numpy(), atol=1e-60)


def test_two_keys_logistic_closed_form(orc):
    # L=1, k=1: keys {context 0, candidate 0}; o = sigmoid(s0-s1) v0 + sigmoid(s1-s0) v1
    t = _tiny(seed=6, lengths=(1,), ctx=(1,), n=1, hq=1, hkv=1, d=4)
    out, lse = _run(orc, t)
    q = t["q"][0, 0].double()
    s0 = float(t["scale"] * (q @ t["k_ctx"][0, 0].double()))
    s1 = float(t["scale"] * (q @ t["k_new"][0, 0].double()))
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    ref = w0 * t["v_ctx"][0, 0].double() + w1 * t["v_new"][0, 0].double()
    np.testing.assert_allclose(out[0, 0], ref.numpy(), atol=1e-14)
    lse_ref = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
    assert abs(lse[0, 0] - lse_ref) < 1e-14


def test_one_slot_empty_context_returns_own_value(orc):
    t = _tiny(seed=7, lengths=(1, 1), ctx=(0, 0), n=2)
    out, lse = _run(orc, t)
    G = 2
    for r in range(2):
        for h in range(4):
            np.testing.assert_array_equal(out[r, h], t["v_new"][r, h // G].double().numpy())
            s = t["scale"] * float(t["q"][r, h].double() @ t["k_new"][r, h // G].double())
            assert abs(lse[r, h] - s) < 1e-14


def test_empty_context_is_textbook_causal_attention(orc):
    t = _tiny(seed=8, lengths=(5,), ctx=(0,), n=1, hq=2, hkv=2, d=8)
    out, _ = _run(orc, t)
    q = t["q"].double().transpose(0, 1)
    k = t["k_new"].double().transpose(0, 1)
    v = t["v_new"].double().transpose(0, 1)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=t["scale"])
    np.testing.assert_allclose(out, ref.transpose(0, 1).numpy(), atol=1e-13)


def test_single_slot_is_decode_attention(orc):
    t = _tiny(seed=9, lengths=(1,), ctx=(7,), n=1, hq=2, hkv=1, d=8)
    out, _ = _run(orc, t)
    keys = torch.cat([t["k_ctx"], t["k_new"]], 0).double().repeat_interleave(2, 1).transpose(0, 1)
    vals = torch.cat([t["v_ctx"], t["v_new"]], 0).double().repeat_interleave(2, 1).transpose(0, 1)
    q = t["q"].double().transpose(0, 1)
    ref = F.scaled_dot_product_attention(q, keys, vals, scale=t["scale"])
    np.testing.assert_allclose(out, ref.transpose(0, 1).numpy(), atol=1e-13)


def _wl_run(orc, b, **kw):
    if b.paged:
        return orc.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv,
                             scale=b.scale, k_cache=b.k_cache, v_cache=b.v_cache,
                             block_table=b.block_table, cache_strides=b.cache_strides, **kw)
    return orc.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv,
                         scale=b.scale, k_ctx=b.k_ctx, v_ctx=b.v_ctx, cu_ctx=b.cu_ctx, **kw)


def test_packed_equals_alone_at_full_width_truncated(orc):
    # tiny_fp32 batch: each request run alone with all W rows, truncated to k_i rows
    b = wl.make_batch("tiny_fp32", seed=0)
    out, lse = _wl_run(orc, b, threads=4)
    cu = b.cu_slots.tolist()
    cuc = b.cu_ctx.tolist()
    for i in range(b.n):
        alone = dict(q=b.full["q"][i], k_new=b.full["k_new"][i], v_new=b.full["v_new"][i],
                     k_ctx=b.k_ctx[cuc[i]:cuc[i + 1]], v_ctx=b.v_ctx[cuc[i]:cuc[i + 1]],
                     cu_ctx=torch.tensor([0, cuc[i + 1] - cuc[i]], dtype=torch.int64),
                     ctx_len=b.ctx_len[i:i + 1], cu_slots=torch.tensor([0, b.W], dtype=torch.int32),
                     hkv=b.hkv, scale=b.scale)
        o1, l1 = _run(orc, alone)
        k = cu[i + 1] - cu[i]
        np.testing.assert_array_equal(out[cu[i]:cu[i + 1]], o1[:k])
        np.testing.assert_array_equal(lse[cu[i]:cu[i + 1]], l1[:k])


def test_relayout_moves_offsets_without_changing_rows(orc):
    # Fig. 1 (Challenge 3): [4,12,8] -> [10,8,6]; common rows of every request unchanged
    b1 = wl.make_batch("tiny_fp32", seed=0)
    b2 = wl.make_batch("tiny_fp32", seed=0, lengths=[10, 8, 6])
    assert b1.cu_slots.tolist()[1] == 4 and b2.cu_slots.tolist()[1] == 10
    o1, l1 = _wl_run(orc, b1)
    o2, l2 = _wl_run(orc, b2)
    c1, c2 = b1.cu_slots.tolist(), b2.cu_slots.tolist()
    for i, (ka, kb) in enumerate(zip([4, 12, 8], [10, 8, 6])):
        m = min(ka, kb)
        np.testing.assert_array_equal(o1[c1[i]:c1[i] + m], o2[c2[i]:c2[i] + m])
        np.testing.assert_array_equal(l1[c1[i]:c1[i] + m], l2[c2[i]:c2[i] + m])


def test_paged_equals_contiguous(orc):
    b = wl.make_batch("paged_n64_bf16", seed=1, n=3, lengths=[5, 16, 1],
                      ctx_lengths=[33, 16, 70], hq=4, hkv=2, d=16, poison=True)
    out_p, lse_p = _wl_run(orc, b)
    # gather the same tokens into a contiguous context
    ks, vs, cuc = [], [], [0]
    bt = b.block_table.tolist()
    for i, L in enumerate(b.ctx_len.tolist()):
        pages = [bt[i][t // 16] for t in range(L)]
        ks.append(torch.stack([b.k_cache[p, :, t % 16] for t, p in enumerate(pages)]))
        vs.append(torch.stack([b.v_cache[p, :, t % 16] for t, p in enumerate(pages)]))
        cuc.append(cuc[-1] + L)
    out_c, lse_c = orc.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv,
                                 scale=b.scale, k_ctx=torch.cat(ks), v_ctx=torch.cat(vs),
                                 cu_ctx=torch.tensor(cuc, dtype=torch.int64))
    np.testing.assert_array_equal(out_p, out_c)
    np.testing.assert_array_equal(lse_p, lse_c)
    assert np.isfinite(out_p[:b.m_live]).all()


def test_request_permutation_permutes_outputs(orc):
    t = _tiny(seed=10, lengths=(2, 3, 1), ctx=(3, 1, 5))
    out, _ = _run(orc, t)
    perm = [2, 0, 1]
    cu, cuc = t["cu_slots"].tolist(), t["cu_ctx"].tolist()
    lens = [cu[i + 1] - cu[i] for i in range(3)]
    rows = torch.cat([torch.arange(cu[i], cu[i + 1]) for i in perm])
    ctx_rows = torch.cat([torch.arange(cuc[i], cuc[i + 1]) for i in perm])
    tp = dict(q=t["q"][rows], k_new=t["k_new"][rows], v_new=t["v_new"][rows],
              k_ctx=t["k_ctx"][ctx_rows], v_ctx=t["v_ctx"][ctx_rows],
              cu_ctx=wl.prefix_offsets([cuc[i + 1] - cuc[i] for i in perm]).to(torch.int64),
              ctx_len=t["ctx_len"][perm], cu_slots=wl.prefix_offsets([lens[i] for i in perm]),
              hkv=t["hkv"], scale=t["scale"])
    out_p, _ = _run(orc, tp)
    np.testing.assert_array_equal(out_p, out[rows.numpy()])


def test_rows_outside_requests_untouched_and_inactive_requests(orc):
    t = _tiny(seed=11, lengths=(2, 0, 3), ctx=(3, 4, 0))
    m = int(t["cu_slots"][-1])
    pad = 4
    for key in ("q", "k_new", "v_new"):
        t[key] = torch.cat([t[key], torch.full((pad,) + tuple(t[key].shape[1:]), float("nan"))])
    out, lse = _run(orc, t)
    assert np.isnan(out[m:]).all() and np.isnan(lse[m:]).all()
    assert np.isfinite(out[:m]).all()


def test_threads_do_not_change_results(orc):
    b = wl.make_batch("tiny_fp32", seed=2)
    o1, l1 = _wl_run(orc, b, threads=1)
    o8, l8 = _wl_run(orc, b, threads=8)
    np.testing.assert_array_equal(o1, o8)
    np.testing.assert_array_equal(l1, l8)
