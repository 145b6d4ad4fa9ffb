"""Graph-captured fixed-address step ("DScale", SIII-D, Algorithm 2): allocate and pack,
verify, accept, captured once and replayed while the lengths change.  Every replay is
checked against the references: allocator / packer (oracle/dvl.py) bit-exact, attention
of the packed rows (fp64 oracle) within the bf16 bars, margins and acceptance bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from oracle import dvl
from speculative_decoding_verification_packed_gb300.pipeline import VerifyPipeline
from tests.helpers import compare_attention

pytestmark = pytest.mark.gpu


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def test_replayed_step_matches_references():
    torch.manual_seed(0)
    rng = np.random.default_rng(0)
    n_bs, w, per, hq, hkv, d, vocab = 6, 16, 8, 8, 2, 128, 512
    ctx = rng.integers(0, 300, n_bs).astype(np.int32)
    cu_ctx = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int64)
    k_ctx = torch.randn(int(cu_ctx[-1]), hkv, d).to(torch.bfloat16)
    v_ctx = torch.randn(int(cu_ctx[-1]), hkv, d).to(torch.bfloat16)
    dev = lambda t: t.cuda()
    pipe = VerifyPipeline(n_bs, hq=hq, hkv=hkv, d=d, vocab=vocab, w=w, budget_per_req=per,
                          ctx_len=dev(torch.from_numpy(ctx)),
                          kv_tensors=dict(k_ctx=dev(k_ctx), v_ctx=dev(v_ctx),
                                          cu_ctx=dev(torch.from_numpy(cu_ctx))))
    captured = False
    for step, n_live in enumerate([6, 4, 5]):
        scores = rng.random((n_bs, w - 1)).astype(np.float32)
        tokens = rng.integers(0, vocab, (n_bs, w)).astype(np.int32)
        positions = rng.integers(0, 4096, (n_bs, w)).astype(np.int32)
        q_full = torch.randn(n_bs * w, hq, d).to(torch.bfloat16)
        k_full = torch.randn(n_bs * w, hkv, d).to(torch.bfloat16)
        v_full = torch.randn(n_bs * w, hkv, d).to(torch.bfloat16)
        logits_full = (torch.randn(n_bs * w, vocab) * 2).to(torch.bfloat16)
        # drafts that often match the target argmax of the previous slot, so that
        # acceptance lengths vary
        am = logits_full.float().argmax(dim=1).view(n_bs, w).numpy()
        for i in range(n_bs):
            for j in range(1, w):
                if rng.random() < 0.7:
                    tokens[i, j] = am[i, j - 1]
        # write the step's inputs in place (fixed addresses), then replay
        pipe.scores.copy_(torch.from_numpy(scores))
        pipe.n_live.fill_(n_live)
        pipe.tokens.copy_(torch.from_numpy(tokens))
        pipe.positions.copy_(torch.from_numpy(positions))
        pipe.q_full.copy_(q_full)
        pipe.k_full.copy_(k_full)
        pipe.v_full.copy_(v_full)
        pipe.logits_full.copy_(logits_full)
        if not captured:
            pipe.capture()
            captured = True
        pipe.step()
        torch.cuda.synchronize()
        a = pipe.alloc
        ref = dvl.dvl_allocate_pack(scores, n_live, per, pipe.m_cap, tokens, positions,
                                    np.arange(n_bs * w).reshape(n_bs, w), 0, 0, -1)
        assert a["k"].cpu().tolist() == ref["k"].tolist()
        cu = a["cu_slots"].cpu()
        assert cu.tolist() == ref["cu"].tolist()
        assert a["tokens"].cpu().tolist() == ref["tokens"].tolist()
        assert a["positions"].cpu().tolist() == ref["positions"].tolist()
        refs = ref["kv_refs"]
        live = refs >= 0
        take = lambda full: torch.where(torch.from_numpy(live).view(-1, *([1] * (full.dim() - 1))),
                                        full[torch.from_numpy(np.where(live, refs, 0))],
                                        torch.zeros((), dtype=full.dtype))
        qp, kp, vp, lp = take(q_full), take(k_full), take(v_full), take(logits_full)
        ro, rl = oracle.attention(qp, kp, vp, torch.from_numpy(ctx), cu, hkv=hkv, scale=d ** -0.5,
                                  k_ctx=k_ctx, v_ctx=v_ctx, cu_ctx=torch.from_numpy(cu_ctx), threads=8)
        rows = np.arange(int(cu[-1]))
        compare_attention(pipe.out, pipe.lse, ro, rl, rows, torch.bfloat16)
        idx, t1, t2, mg = oracle.row_top2(lp[rows])
        g_idx, g_t1, g_t2, g_mg = (x.cpu().numpy()[rows] for x in pipe.margin_outs[:4])
        assert g_idx.tolist() == idx.tolist()
        assert g_mg.tolist() == mg.tolist()
        am_p = np.full(pipe.m_cap, -1, dtype=np.int32)
        am_p[rows] = idx
        acc, nxt = oracle.greedy_accept(am_p, ref["tokens"].astype(np.int32), cu)
        assert pipe.accept_len.cpu().tolist() == acc.tolist(), step
        assert pipe.next_token.cpu().tolist() == nxt.tolist(), step
        assert pipe.ws_attn.read_status() == 0 and pipe.ws_dvl.read_status() == 0
